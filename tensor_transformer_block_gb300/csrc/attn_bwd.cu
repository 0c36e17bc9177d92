// Attention backward cores on tcgen05.  The pages give no attention backward;
// these kernels differentiate the forward's definition (see include/tpblock.h):
//   Dsum = rowsum(dO * O)                       (k_attn_dsum)
//   P = exp(S/sqrt(d) - LSE), dS = P * (dP - Dsum), dP = dO V^T
//   dV = P^T dO, dK = dS^T Q / sqrt(d)          (k_attn_dkdv: one CTA per key block of
//                                                a key/value head, summing over the
//                                                query heads of its group)
//   dQ = dS K / sqrt(d)                         (k_attn_dq:   one CTA per query block)
// Each CTA owns its output rows and loops over the blocks it needs, so results
// are deterministic (no atomics).  P is recomputed from the saved LSE.
// Warp roles as in the forward: warp 4 TMA, warp 5 MMA, warps 0-3 one row each.
#include <cmath>

#include "attn.cuh"
#include "host_util.cuh"
#include "ptx.cuh"

namespace tpb {
namespace {

constexpr int BLK = 128;
constexpr int NTHREADS = 192;
constexpr float kLog2e = 1.4426950408889634f;

// -------------------------------------------------------------------- Dsum
template <int D>
__global__ void k_attn_dsum(const uint4* __restrict__ o, const uint4* __restrict__ dout, float* __restrict__ dsum,
                            const AttnDims a) {
  const long long T = static_cast<long long>(a.B) * a.S;
  const long long total = static_cast<long long>(a.N) * T * a.hN;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long base = idx * (D / 8);  // uint4 = 8 bf16
    float s = 0.0f;
#pragma unroll 4
    for (int v = 0; v < D / 8; ++v) {
      const uint4 x = o[base + v], y = dout[base + v];
      s += bf16lo_to_f32(x.x) * bf16lo_to_f32(y.x) + bf16hi_to_f32(x.x) * bf16hi_to_f32(y.x);
      s += bf16lo_to_f32(x.y) * bf16lo_to_f32(y.y) + bf16hi_to_f32(x.y) * bf16hi_to_f32(y.y);
      s += bf16lo_to_f32(x.z) * bf16lo_to_f32(y.z) + bf16hi_to_f32(x.z) * bf16hi_to_f32(y.z);
      s += bf16lo_to_f32(x.w) * bf16lo_to_f32(y.w) + bf16hi_to_f32(x.w) * bf16hi_to_f32(y.w);
    }
    const long long shard = idx / (T * a.hN);
    const long long rem = idx - shard * T * a.hN;
    const long long t = rem / a.hN;
    const int jj = static_cast<int>(rem - t * a.hN);
    const long long bb = t / a.S, ss = t - bb * a.S;
    const long long j = shard * a.hN + jj;
    dsum[(bb * a.H + j) * a.S + ss] = s;
  }
}

struct BwdCommon {
  uint32_t sb;
  uint32_t bar0;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * static_cast<uint32_t>(i); }
};

// Writes a warp's 32 accumulator rows x D columns (fp32 in TMEM, times ``mul``)
// as bf16 into a staging area laid out as D/64 boxes of 32 x 64 (swizzled).
template <int D>
__device__ __forceinline__ void stage_rows_from_tmem(uint32_t taddr, uint32_t stage, int lane, float mul) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + 32 * c, v);
    tmem_ld_wait(v);
    const uint32_t cb = static_cast<uint32_t>(c >> 1), g0 = static_cast<uint32_t>((c & 1) * 4);
#pragma unroll
    for (int g = 0; g < 4; ++g)
      st_shared_v4(stage + cb * 4096 + lane * 128 + (((g0 + g) ^ static_cast<uint32_t>(lane & 7)) << 4),
                   pack_bf16x2(__uint_as_float(v[8 * g + 0]) * mul, __uint_as_float(v[8 * g + 1]) * mul),
                   pack_bf16x2(__uint_as_float(v[8 * g + 2]) * mul, __uint_as_float(v[8 * g + 3]) * mul),
                   pack_bf16x2(__uint_as_float(v[8 * g + 4]) * mul, __uint_as_float(v[8 * g + 5]) * mul),
                   pack_bf16x2(__uint_as_float(v[8 * g + 6]) * mul, __uint_as_float(v[8 * g + 7]) * mul));
  }
}

// K-major operand product over K = D: D (+)= A B^T, A and B tiles of ``rows_b``
// rows stored as 64-column swizzled chunks of ``chunk_b`` bytes (A chunks 16 KB).
template <int D>
__device__ __forceinline__ void mma_kmajor(uint32_t d_tmem, uint32_t sa, uint32_t sb, uint32_t chunk_b, uint32_t idesc,
                                           bool acc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t in = static_cast<uint32_t>((kk & 3) * 32);
    const uint32_t kc = static_cast<uint32_t>(kk >> 2);
    tc_mma_bf16(d_tmem, sdesc_sw128(sa + kc * 16384 + in, 16, 1024), sdesc_sw128(sb + kc * chunk_b + in, 16, 1024),
                idesc, (acc || kk > 0) ? 1u : 0u);
  }
}

// ------------------------------------------------------------------ dK / dV
// One CTA per (128-key block, key/value head, batch); loops over the query heads
// of the head's group and, for each, over the 64-query blocks whose
// Qh, Ql, dO tiles and LSE / Dsum rows are double-buffered, as are the S^T and
// dP^T tiles in TMEM, so block i+1's products run while the key-row threads turn
// block i's scores into P^T and dS^T.
constexpr int QB = 64;
enum : int {
  K_KVF = 0, K_QF = 1 /* 2 */, K_QE = 3 /* 2 */, K_STF = 5 /* 2 */, K_STE = 7 /* 2 */,
  K_PSF = 9, K_PSE = 10, K_ACC = 11, K_DR = 12, K_NB = 13
};

template <int D>
struct DkdvCfg {
  static constexpr int CH = D / 64;
  static constexpr int KTILE = CH * 16384;  // 128 key rows x D
  static constexpr int QTILE = CH * 8192;   // 64 query rows x D
  static constexpr int OFF_KH = 0, OFF_KL = KTILE, OFF_V = 2 * KTILE;
  static constexpr int OFF_Q = 3 * KTILE;   // [stage][Qh, Ql, dO]
  static constexpr int OFF_P = OFF_Q + 6 * QTILE;  // [128 keys][64 queries] bf16, 16 KB
  static constexpr int OFF_DS = OFF_P + 16384;
  static constexpr int OFF_LSE = OFF_DS + 16384;   // [2][64] fp32
  static constexpr int OFF_DD = OFF_LSE + 512;     // [2][64] fp32
  static constexpr int OFF_BAR = OFF_DD + 512;
  static constexpr int OFF_MISC = OFF_BAR + K_NB * 8;
  static constexpr int USED = OFF_MISC + 16;
  static constexpr int SMEM = (USED + 1024 > 122880) ? USED + 1024 : 122880;
  static_assert(USED + 1024 <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_attn_dkdv(const __grid_constant__ CUtensorMap tmQKV128, const __grid_constant__ CUtensorMap tmQKV64,
                const __grid_constant__ CUtensorMap tmDO64, const __grid_constant__ CUtensorMap tmDQKV,
                const float* __restrict__ lse, const float* __restrict__ dsum, const AttnDims a,
                const float scale_log2, const float scale, unsigned* err, const unsigned long long timeout_ns) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const BwdCommon cm{raw + pad, raw + pad + C::OFF_BAR};
  const uint32_t sKh = cm.sb + C::OFF_KH, sKl = cm.sb + C::OFF_KL, sV = cm.sb + C::OFF_V;
  auto sQh = [&](int st) { return cm.sb + C::OFF_Q + static_cast<uint32_t>((3 * st + 0) * C::QTILE); };
  auto sQl = [&](int st) { return cm.sb + C::OFF_Q + static_cast<uint32_t>((3 * st + 1) * C::QTILE); };
  auto sDO = [&](int st) { return cm.sb + C::OFF_Q + static_cast<uint32_t>((3 * st + 2) * C::QTILE); };
  const uint32_t sP = cm.sb + C::OFF_P, sDS = cm.sb + C::OFF_DS;
  float* lse_s = reinterpret_cast<float*>(smem + C::OFF_LSE);
  float* dd_s = reinterpret_cast<float*>(smem + C::OFF_DD);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* never_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (a.S + QB - 1) / QB;
  const int kb = static_cast<int>(blockIdx.x);  // low key blocks have the most causal work: first
  const int jkv = blockIdx.y, b = blockIdx.z;   // global key/value head
  const int shard = jkv / a.hkvN, kvh = jkv % a.hkvN;
  const int g = a.group();
  const int k0 = kb * BLK;
  const int q_start = a.causal ? (k0 / QB) : 0;
  const int nq = nqb - q_start;
  const int nit = nq * g;  // (query head of the group, query block) pairs
  const int cKh = a.col_k(kvh), cV = a.col_v(kvh), cKl = a.col_kl(kvh);
  const int dcK = a.hN * D + kvh * D, dcV = (a.hN + a.hkvN + kvh) * D;  // in dQKV

  if (threadIdx.x == 0) {
    for (int i = 0; i < K_NB; ++i) {
      const bool by_warps = i == K_PSF || i == K_STE || i == K_STE + 1;
      mbar_init(cm.bar(i), by_warps ? 4 : 1);
    }
    *abort_flag = 0;
    *never_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{err, abort_flag, timeout_ns};
  const WaitCtx wdrain{err, never_flag, timeout_ns};
  // TMEM: S^T [s*64, +64), dP^T [128 + s*64, +64), dV [256, +D), dK [256+D, +D)
  const uint32_t tDV = tmem + 256, tDK = tmem + 256 + D;
  // iteration it: local query head jq(it) of the group, query block q0(it)
  auto jq_of = [&](int it) { return kvh * g + it / nq; };
  auto q0_of = [&](int it) { return (q_start + it % nq) * QB; };

  if (warp == 4) {
    // producer warp: lane 0 issues the TMA copies; all lanes stage each block's
    // LSE and Dsum rows (plain loads: any S), published by the same barrier
    if (lane == 0) {
      mbar_arrive_expect_tx(cm.bar(K_KVF), 3 * C::KTILE);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_load_4d(sKh + c * 16384, &tmQKV128, cm.bar(K_KVF), cKh + 64 * c, k0, b, shard);
        tma_load_4d(sKl + c * 16384, &tmQKV128, cm.bar(K_KVF), cKl + 64 * c, k0, b, shard);
        tma_load_4d(sV + c * 16384, &tmQKV128, cm.bar(K_KVF), cV + 64 * c, k0, b, shard);
      }
    }
    int issued = 0;
    for (int it = 0; it < nit; ++it) {
      const int st = it & 1;
      const uint32_t ph = static_cast<uint32_t>((it >> 1) & 1);
      const int q0 = q0_of(it), jq = jq_of(it);
      const size_t row_base = (static_cast<size_t>(b) * a.H + shard * a.hN + jq) * a.S;
      if (!__all_sync(0xffffffffu, mbar_wait(cm.bar(K_QE + st), ph ^ 1u, wc))) break;
      for (int t = lane; t < QB; t += 32) {
        const int q = q0 + t;
        lse_s[st * QB + t] = q < a.S ? lse[row_base + q] : 0.0f;
        dd_s[st * QB + t] = q < a.S ? dsum[row_base + q] : 0.0f;
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) {
        const uint32_t fb = cm.bar(K_QF + st);
        mbar_arrive_expect_tx(fb, 3 * C::QTILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_4d(sQh(st) + c * 8192, &tmQKV64, fb, a.col_q(jq) + 64 * c, q0, b, shard);
          tma_load_4d(sQl(st) + c * 8192, &tmQKV64, fb, a.col_ql(jq) + 64 * c, q0, b, shard);
          tma_load_4d(sDO(st) + c * 8192, &tmDO64, fb, jq * D + 64 * c, q0, b, shard);
        }
      }
      issued = it + 1;
    }
    if (lane == 0) {
      mbar_wait(cm.bar(K_KVF), 0, wdrain);
      for (int it = issued - 2 < 0 ? 0 : issued - 2; it < issued; ++it)
        mbar_wait(cm.bar(K_QF + (it & 1)), (it >> 1) & 1, wdrain);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, QB, false, false);
      constexpr uint32_t ID_G = idesc_bf16(128, D, false, true);
      bool ok = mbar_wait(cm.bar(K_KVF), 0, wc), any = false;
      auto issue_sd = [&](int it) -> bool {
        const int st = it & 1;
        const uint32_t ph = static_cast<uint32_t>((it >> 1) & 1);
        if (!mbar_wait(cm.bar(K_QF + st), ph, wc) || !mbar_wait(cm.bar(K_STE + st), ph ^ 1u, wc)) return false;
        tc_fence_after();
        const uint32_t tS = tmem + static_cast<uint32_t>(st * 64), tP = tmem + 128 + static_cast<uint32_t>(st * 64);
        mma_kmajor<D>(tS, sKh, sQh(st), 8192, ID_S, false);
        mma_kmajor<D>(tS, sKl, sQh(st), 8192, ID_S, true);
        mma_kmajor<D>(tS, sKh, sQl(st), 8192, ID_S, true);
        mma_kmajor<D>(tP, sV, sDO(st), 8192, ID_S, false);
        any = true;
        tc_commit(cm.bar(K_STF + st));
        return true;
      };
      if (ok && nit > 0) ok = issue_sd(0);
      for (int it = 0; it < nit && ok; ++it) {
        const int st = it & 1;
        if (it + 1 < nit && !issue_sd(it + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(cm.bar(K_PSF), it & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < QB / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          // A: P^T / dS^T [128 keys][64 queries] K-major; B: dO / Qh tiles read MN-major (N = d)
          tc_mma_bf16(tDV, sdesc_sw128(sP + kk * 32, 16, 1024), sdesc_sw128(sDO(st) + kk * 2048, 8192, 1024), ID_G,
                      acc);
          tc_mma_bf16(tDK, sdesc_sw128(sDS + kk * 32, 16, 1024), sdesc_sw128(sQh(st) + kk * 2048, 8192, 1024), ID_G,
                      acc);
        }
        tc_commit(cm.bar(K_QE + st));
        tc_commit(cm.bar(K_PSE));
      }
      if (ok) tc_commit(cm.bar(K_ACC));
      if (any) {
        tc_commit(cm.bar(K_DR));
        mbar_wait(cm.bar(K_DR), 0, wdrain);
      }
    }
  } else {
    const int r = warp * 32 + lane;
    const int key = k0 + r;
    const uint32_t trow = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t rsw = static_cast<uint32_t>(r & 7);
    bool ok = true;
    for (int it = 0; it < nit; ++it) {
      const int st = it & 1;
      const uint32_t ph = static_cast<uint32_t>((it >> 1) & 1);
      const int q0 = q0_of(it);
      ok = __all_sync(0xffffffffu, mbar_wait(cm.bar(K_STF + st), ph, wc) && mbar_wait(cm.bar(K_QF + st), ph, wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t vs0[32], vs1[32], vp0[32], vp1[32];
      tmem_ld32(tmem + trow + st * 64, vs0);
      tmem_ld32(tmem + trow + st * 64 + 32, vs1);
      tmem_ld32(tmem + trow + 128 + st * 64, vp0);
      tmem_ld32(tmem + trow + 128 + st * 64 + 32, vp1);
      tmem_ld_wait(vs0);
      tmem_ld_wait(vs1);
      tmem_ld_wait(vp0);
      tmem_ld_wait(vp1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cm.bar(K_STE + st));  // the S^T / dP^T buffers may be refilled
      const bool need_mask = (a.causal && q0 < k0 + BLK) || (q0 + QB > a.S) || (k0 + BLK > a.S);
      const float* ls = lse_s + st * QB;
      const float* ds = dd_s + st * QB;
      uint32_t pk[32], dk[32];
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        float p2[2], d2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int qc = e + u;
          const int q = q0 + qc;
          const float sv = __uint_as_float(qc < 32 ? vs0[qc] : vs1[qc - 32]);
          const float dpv = __uint_as_float(qc < 32 ? vp0[qc] : vp1[qc - 32]);
          float p = exp2f(sv * scale_log2 - ls[qc] * kLog2e);
          if (need_mask && (q >= a.S || key >= a.S || (a.causal && key > q))) p = 0.0f;
          p2[u] = p;
          d2[u] = p * (dpv - ds[qc]);
        }
        pk[e >> 1] = pack_bf16x2(p2[0], p2[1]);
        dk[e >> 1] = pack_bf16x2(d2[0], d2[1]);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(cm.bar(K_PSE), (it & 1) ^ 1, wc));
      if (!ok) break;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint32_t ad = static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(g) ^ rsw) << 4);
        st_shared_v4(sP + ad, pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        st_shared_v4(sDS + ad, dk[4 * g], dk[4 * g + 1], dk[4 * g + 2], dk[4 * g + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(cm.bar(K_PSF));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(cm.bar(K_ACC), 0, wc));
    if (ok) {
      tc_fence_after();
      // all MMAs are complete: the Q/dO stages are free for staging (2 x 4 warps x CH x 4 KB)
      const uint32_t stV = cm.sb + C::OFF_Q + static_cast<uint32_t>(warp * C::CH * 4096);
      const uint32_t stK = cm.sb + C::OFF_Q + static_cast<uint32_t>((4 + warp) * C::CH * 4096);
      stage_rows_from_tmem<D>(tDV + trow, stV, lane, 1.0f);
      stage_rows_from_tmem<D>(tDK + trow, stK, lane, scale);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && k0 + warp * 32 < a.S) {
#pragma unroll
        for (int cb = 0; cb < C::CH; ++cb) {
          tma_store_4d(&tmDQKV, stV + cb * 4096, dcV + 64 * cb, k0 + warp * 32, b, shard);
          tma_store_4d(&tmDQKV, stK + cb * 4096, dcK + 64 * cb, k0 + warp * 32, b, shard);
        }
        bulk_commit();
      }
    }
    __syncwarp();
    if (lane == 0) bulk_wait0();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------- dQ
// One CTA per (128-query block, head, batch); loops over 64-key blocks whose
// Kh, Kl, V tiles are double-buffered, as are the S and dP tiles in TMEM.
constexpr int KBQ = 64;
enum : int {
  Q_QF = 0, Q_KF = 1 /* 2 */, Q_KE = 3 /* 2 */, Q_SF = 5 /* 2 */, Q_SE = 7 /* 2 */,
  Q_DSF = 9, Q_DSE = 10, Q_ACC = 11, Q_DR = 12, Q_NB = 13
};

template <int D>
struct DqCfg {
  static constexpr int CH = D / 64;
  static constexpr int QTILE = CH * 16384;  // 128 query rows x D
  static constexpr int KTILE = CH * 8192;   // 64 key rows x D
  static constexpr int OFF_QH = 0, OFF_QL = QTILE, OFF_DO = 2 * QTILE;
  static constexpr int OFF_K = 3 * QTILE;   // [stage][Kh, Kl, V]
  static constexpr int OFF_DS = OFF_K + 6 * KTILE;  // [128 queries][64 keys] bf16, 16 KB
  static constexpr int OFF_BAR = OFF_DS + 16384;
  static constexpr int OFF_MISC = OFF_BAR + Q_NB * 8;
  static constexpr int USED = OFF_MISC + 16;
  static constexpr int SMEM = (USED + 1024 > 122880) ? USED + 1024 : 122880;
  static_assert(USED + 1024 <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_attn_dq(const __grid_constant__ CUtensorMap tmQKV128, const __grid_constant__ CUtensorMap tmQKV64,
              const __grid_constant__ CUtensorMap tmDO128, const __grid_constant__ CUtensorMap tmDQKV,
              const float* __restrict__ lse, const float* __restrict__ dsum, const AttnDims a, const float scale_log2,
              const float scale, unsigned* err, const unsigned long long timeout_ns) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const BwdCommon cm{raw + pad, raw + pad + C::OFF_BAR};
  const uint32_t sQh = cm.sb + C::OFF_QH, sQl = cm.sb + C::OFF_QL, sDO = cm.sb + C::OFF_DO;
  auto sKh = [&](int st) { return cm.sb + C::OFF_K + static_cast<uint32_t>((3 * st + 0) * C::KTILE); };
  auto sKl = [&](int st) { return cm.sb + C::OFF_K + static_cast<uint32_t>((3 * st + 1) * C::KTILE); };
  auto sV = [&](int st) { return cm.sb + C::OFF_K + static_cast<uint32_t>((3 * st + 2) * C::KTILE); };
  const uint32_t sDS = cm.sb + C::OFF_DS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* never_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = (a.S + BLK - 1) / BLK;
  const int qb = nb - 1 - static_cast<int>(blockIdx.x);
  const int j = blockIdx.y, b = blockIdx.z;
  const int shard = j / a.hN, jj = j % a.hN, kvh = jj / a.group();
  const int q0 = qb * BLK;
  const int nkb = (a.S + KBQ - 1) / KBQ;
  const int nkv = a.causal ? min((min(q0 + BLK, a.S) - 1) / KBQ + 1, nkb) : nkb;
  const int cQh = a.col_q(jj), cKh = a.col_k(kvh), cV = a.col_v(kvh);
  const int cQl = a.col_ql(jj), cKl = a.col_kl(kvh);

  if (threadIdx.x == 0) {
    for (int i = 0; i < Q_NB; ++i) {
      const bool by_warps = i == Q_DSF || i == Q_SE || i == Q_SE + 1;
      mbar_init(cm.bar(i), by_warps ? 4 : 1);
    }
    *abort_flag = 0;
    *never_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{err, abort_flag, timeout_ns};
  const WaitCtx wdrain{err, never_flag, timeout_ns};
  // TMEM: S [s*64, +64), dP [128 + s*64, +64), dQ [256, +D)

  if (warp == 4) {
    if (lane == 0) {
      mbar_arrive_expect_tx(cm.bar(Q_QF), 3 * C::QTILE);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_load_4d(sQh + c * 16384, &tmQKV128, cm.bar(Q_QF), cQh + 64 * c, q0, b, shard);
        tma_load_4d(sQl + c * 16384, &tmQKV128, cm.bar(Q_QF), cQl + 64 * c, q0, b, shard);
        tma_load_4d(sDO + c * 16384, &tmDO128, cm.bar(Q_QF), jj * D + 64 * c, q0, b, shard);
      }
      int issued = 0;
      for (int it = 0; it < nkv; ++it) {
        const int st = it & 1;
        const uint32_t ph = static_cast<uint32_t>((it >> 1) & 1);
        if (!mbar_wait(cm.bar(Q_KE + st), ph ^ 1u, wc)) break;
        const uint32_t fb = cm.bar(Q_KF + st);
        mbar_arrive_expect_tx(fb, 3 * C::KTILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_4d(sKh(st) + c * 8192, &tmQKV64, fb, cKh + 64 * c, it * KBQ, b, shard);
          tma_load_4d(sKl(st) + c * 8192, &tmQKV64, fb, cKl + 64 * c, it * KBQ, b, shard);
          tma_load_4d(sV(st) + c * 8192, &tmQKV64, fb, cV + 64 * c, it * KBQ, b, shard);
        }
        issued = it + 1;
      }
      mbar_wait(cm.bar(Q_QF), 0, wdrain);
      for (int it = issued - 2 < 0 ? 0 : issued - 2; it < issued; ++it)
        mbar_wait(cm.bar(Q_KF + (it & 1)), (it >> 1) & 1, wdrain);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, KBQ, false, false);
      constexpr uint32_t ID_G = idesc_bf16(128, D, false, true);
      bool ok = mbar_wait(cm.bar(Q_QF), 0, wc), any = false;
      auto issue_sp = [&](int it) -> bool {
        const int st = it & 1;
        const uint32_t ph = static_cast<uint32_t>((it >> 1) & 1);
        if (!mbar_wait(cm.bar(Q_KF + st), ph, wc) || !mbar_wait(cm.bar(Q_SE + st), ph ^ 1u, wc)) return false;
        tc_fence_after();
        const uint32_t tS = tmem + static_cast<uint32_t>(st * 64), tP = tmem + 128 + static_cast<uint32_t>(st * 64);
        mma_kmajor<D>(tS, sQh, sKh(st), 8192, ID_S, false);
        mma_kmajor<D>(tS, sQh, sKl(st), 8192, ID_S, true);
        mma_kmajor<D>(tS, sQl, sKh(st), 8192, ID_S, true);
        mma_kmajor<D>(tP, sDO, sV(st), 8192, ID_S, false);
        any = true;
        tc_commit(cm.bar(Q_SF + st));
        return true;
      };
      if (ok && nkv > 0) ok = issue_sp(0);
      for (int it = 0; it < nkv && ok; ++it) {
        const int st = it & 1;
        if (it + 1 < nkv && !issue_sp(it + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(cm.bar(Q_DSF), it & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < KBQ / 16; ++kk)
          tc_mma_bf16(tmem + 256, sdesc_sw128(sDS + kk * 32, 16, 1024), sdesc_sw128(sKh(st) + kk * 2048, 8192, 1024),
                      ID_G, (it > 0 || kk > 0) ? 1u : 0u);
        tc_commit(cm.bar(Q_KE + st));
        tc_commit(cm.bar(Q_DSE));
      }
      if (ok) tc_commit(cm.bar(Q_ACC));
      if (any) {
        tc_commit(cm.bar(Q_DR));
        mbar_wait(cm.bar(Q_DR), 0, wdrain);
      }
    }
  } else {
    const int r = warp * 32 + lane;
    const int q = q0 + r;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t rsw = static_cast<uint32_t>(r & 7);
    const bool qvalid = q < a.S;
    const size_t ridx = (static_cast<size_t>(b) * a.H + j) * a.S + q;
    const float lse2 = qvalid ? lse[ridx] * kLog2e : 0.0f;
    const float dd = qvalid ? dsum[ridx] : 0.0f;
    bool ok = true;
    for (int it = 0; it < nkv; ++it) {
      const int st = it & 1;
      const uint32_t ph = static_cast<uint32_t>((it >> 1) & 1);
      const int kbase = it * KBQ;
      ok = __all_sync(0xffffffffu, mbar_wait(cm.bar(Q_SF + st), ph, wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t vs0[32], vs1[32], vp0[32], vp1[32];
      tmem_ld32(trow + st * 64, vs0);
      tmem_ld32(trow + st * 64 + 32, vs1);
      tmem_ld32(trow + 128 + st * 64, vp0);
      tmem_ld32(trow + 128 + st * 64 + 32, vp1);
      tmem_ld_wait(vs0);
      tmem_ld_wait(vs1);
      tmem_ld_wait(vp0);
      tmem_ld_wait(vp1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cm.bar(Q_SE + st));
      const bool need_mask = (a.causal && kbase + KBQ > q0) || (kbase + KBQ > a.S) || !qvalid;
      uint32_t dk[32];
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        float d2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int kc = e + u;
          const int key = kbase + kc;
          const float sv = __uint_as_float(kc < 32 ? vs0[kc] : vs1[kc - 32]);
          const float dpv = __uint_as_float(kc < 32 ? vp0[kc] : vp1[kc - 32]);
          float p = exp2f(sv * scale_log2 - lse2);
          if (need_mask && (!qvalid || key >= a.S || (a.causal && key > q))) p = 0.0f;
          d2[u] = p * (dpv - dd);
        }
        dk[e >> 1] = pack_bf16x2(d2[0], d2[1]);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(cm.bar(Q_DSE), (it & 1) ^ 1, wc));
      if (!ok) break;
#pragma unroll
      for (int g = 0; g < 8; ++g)
        st_shared_v4(sDS + static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(g) ^ rsw) << 4), dk[4 * g],
                     dk[4 * g + 1], dk[4 * g + 2], dk[4 * g + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(cm.bar(Q_DSF));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(cm.bar(Q_ACC), 0, wc));
    if (ok) {
      tc_fence_after();
      // all MMAs are complete: the Qh tile is free for staging
      const uint32_t stQ = sQh + static_cast<uint32_t>(warp * C::CH * 4096);
      stage_rows_from_tmem<D>(trow + 256, stQ, lane, scale);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && q0 + warp * 32 < a.S) {
#pragma unroll
        for (int cb = 0; cb < C::CH; ++cb) tma_store_4d(&tmDQKV, stQ + cb * 4096, jj * D + 64 * cb, q0 + warp * 32, b, shard);
        bulk_commit();
      }
    }
    __syncwarp();
    if (lane == 0) bulk_wait0();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
int launch_bwd_d(const AttnDims& a, const void* qkv, const void* o, const void* dout, const float* lse, float* dsum,
                 void* dqkv, unsigned* err, unsigned long long timeout_ns, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(k_attn_dkdv<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, DkdvCfg<D>::SMEM) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_attn_dq<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::SMEM) != cudaSuccess)
      return 2;
    configured = true;
  }
  const uint64_t S = static_cast<uint64_t>(a.S), Bb = static_cast<uint64_t>(a.B), Nn = static_cast<uint64_t>(a.N);
  CUtensorMap tq128, tq64, tdo128, tdo64, tdq;
  const uint64_t qd[4] = {static_cast<uint64_t>(a.qkv_width()), S, Bb, Nn};
  const uint64_t gd[4] = {static_cast<uint64_t>(a.dqkv_width()), S, Bb, Nn};
  const uint64_t od[4] = {static_cast<uint64_t>(a.hN) * D, S, Bb, Nn};
  const uint32_t box128[4] = {64, 128, 1, 1};
  const uint32_t box64[4] = {64, 64, 1, 1};
  const uint32_t box32[4] = {64, 32, 1, 1};
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!encode_tmap(&tq128, bf, 4, qkv, qd, box128, sw) || !encode_tmap(&tq64, bf, 4, qkv, qd, box64, sw) ||
      !encode_tmap(&tdo128, bf, 4, dout, od, box128, sw) || !encode_tmap(&tdo64, bf, 4, dout, od, box64, sw) ||
      !encode_tmap(&tdq, bf, 4, dqkv, gd, box32, sw))
    return 2;

  const long long rows = static_cast<long long>(a.N) * a.B * a.S * a.hN;
  const int sms = device_sm_count();
  long long blocks = (rows + 255) / 256;
  if (blocks > static_cast<long long>(sms) * 8) blocks = static_cast<long long>(sms) * 8;
  int slot = timing_begin(kKAttnDsum, st);
  k_attn_dsum<D><<<static_cast<int>(blocks), 256, 0, st>>>(static_cast<const uint4*>(o),
                                                           static_cast<const uint4*>(dout), dsum, a);
  bool ok = cudaGetLastError() == cudaSuccess;
  timing_end(slot, st);
  if (!ok) return 2;
  const int nb = (a.S + BLK - 1) / BLK;
  const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  const float scale_log2 = scale * kLog2e;
  const dim3 grid(nb, a.H, a.B), grid_kv(nb, a.Hkv, a.B);
  slot = timing_begin(kKAttnDkdv, st);
  k_attn_dkdv<D><<<grid_kv, NTHREADS, DkdvCfg<D>::SMEM, st>>>(tq128, tq64, tdo64, tdq, lse, dsum, a, scale_log2,
                                                          scale, err, timeout_ns);
  ok = cudaGetLastError() == cudaSuccess;
  timing_end(slot, st);
  if (!ok) return 2;
  slot = timing_begin(kKAttnDq, st);
  k_attn_dq<D><<<grid, NTHREADS, DqCfg<D>::SMEM, st>>>(tq128, tq64, tdo128, tdq, lse, dsum, a, scale_log2, scale,
                                                      err, timeout_ns);
  ok = cudaGetLastError() == cudaSuccess;
  timing_end(slot, st);
  return ok ? 0 : 2;
}

}  // namespace

int launch_attn_bwd(const AttnDims& a, const void* qkv, const void* o, const void* dout, const float* lse,
                    float* dsum, void* dqkv, unsigned* err, unsigned long long timeout_ns, cudaStream_t st) {
  if (a.B < 1 || a.S < 1 || a.H < 1 || a.N < 1 || a.hN * a.N != a.H) return 1;
  if (a.Hkv < 1 || a.hkvN * a.N != a.Hkv || a.H % a.Hkv || a.hN % a.hkvN) return 1;
  if (a.H > 65535 || a.B > 65535) return 1;
  if (a.d == 128) return launch_bwd_d<128>(a, qkv, o, dout, lse, dsum, dqkv, err, timeout_ns, st);
  if (a.d == 64) return launch_bwd_d<64>(a, qkv, o, dout, lse, dsum, dqkv, err, timeout_ns, st);
  return 1;
}

}  // namespace tpb
