// Attention backward cores on tcgen05.  The pages give no attention backward;
// these kernels differentiate the forward's definition (see include/tpblock.h):
//   Dsum = rowsum(dO * O)                       (k_attn_dsum)
//   P = exp(S/sqrt(d) - LSE), dS = P * (dP - Dsum), dP = dO V^T
//   dV = P^T dO, dK = dS^T Q / sqrt(d)          (k_attn_dkdv: one CTA per key block of
//                                                a key/value head, summing over the
//                                                query heads of its group)
//   dQ = dS K / sqrt(d)                         (k_attn_dq:   one CTA per query block)
// Each CTA owns its output rows and loops over the blocks it needs, so results
// are deterministic (no atomics).  P is recomputed from the saved LSE.  Blocks are
// 128 x 128 (M=128, N=128 tensor-core products); Q, K, V, P, dO and dS are fp16,
// so every product is an fp16 MMA.  P and dS never leave TMEM: they are
// written over the first halves of the score columns they come from and feed the
// next products as the TMEM A operand.
// Warp roles: warp 8 TMA, warp 9 MMA, warps 0-7 elementwise (warp w owns TMEM lanes
// 32 (w % 4).. and the column half w / 4 of every 128-column block).
#include <cuda_fp16.h>

#include <cmath>

#include "attn.cuh"
#include "host_util.cuh"
#include "ptx.cuh"

namespace tpb {
namespace {

constexpr int BLK = 128;
constexpr int NTHREADS = 320;
constexpr float kLog2e = 1.4426950408889634f;

// -------------------------------------------------------------------- Dsum
// One row (a token's d values of one head) per group of D/8 lanes: each lane loads
// one 16-byte vector of O and of dO, so a warp's loads are contiguous, and the
// group adds its partial dot products with shuffles.  The loop runs whole warps
// (a group past the last row adds zeros and stores nothing), so every shuffle
// has all 32 lanes.  dO is fp16; O is fp16 or bf16 (a.o_f16).
__device__ __forceinline__ float2 f16x2_to_f32(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
__device__ __forceinline__ float dot8(const uint4& x, const uint4& y, bool x_f16) {
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 yy = f16x2_to_f32(ys[i]);
    const float2 xx = x_f16 ? f16x2_to_f32(xs[i]) : make_float2(bf16lo_to_f32(xs[i]), bf16hi_to_f32(xs[i]));
    s = fmaf(xx.x, yy.x, s);
    s = fmaf(xx.y, yy.y, s);
  }
  return s;
}
template <int D>
__global__ void k_attn_dsum(const uint4* __restrict__ o, const uint4* __restrict__ dout, float* __restrict__ dsum,
                            const AttnDims a, unsigned* err) {
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();
  constexpr int LPR = D / 8;  // lanes (16-byte vectors) per row
  static_assert(32 % LPR == 0, "a row's lanes lie in one warp");
  const long long T = static_cast<long long>(a.B) * a.S;
  const long long total = static_cast<long long>(a.N) * T * a.hN;
  const int lane = threadIdx.x & 31, sub = lane % LPR;
  const long long warp0 = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) / 32;
  const long long nwarps = static_cast<long long>(gridDim.x) * blockDim.x / 32;
  for (long long w = warp0; w * (32 / LPR) < total; w += nwarps) {
    const long long idx = w * (32 / LPR) + lane / LPR;  // this lane's row
    const bool valid = idx < total;
    float s = 0.0f;
    if (valid) s = dot8(o[idx * LPR + sub], dout[idx * LPR + sub], a.o_f16 != 0);
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (valid && sub == 0) {
      // row idx = (shard T + t) hN + jj -> Dsum[b][head][s]; 32-bit (the launcher
      // keeps B S H below 2^31), three divisions per row instead of 64-bit ones
      const uint32_t ui = static_cast<uint32_t>(idx), hN = static_cast<uint32_t>(a.hN);
      const uint32_t q = ui / hN, jj = ui - q * hN;
      const uint32_t T32 = static_cast<uint32_t>(T), shard = q / T32, t = q - shard * T32;
      const uint32_t S32 = static_cast<uint32_t>(a.S), bb = t / S32, ss = t - bb * S32;
      const uint32_t di = (bb * static_cast<uint32_t>(a.H) + shard * hN + jj) * S32 + ss;
      if (TP_DCHECK(di < static_cast<uint32_t>(a.B * a.H * a.S), err)) dsum[di] = s;
    }
  }
}

struct BwdCommon {
  uint32_t sb;
  uint32_t bar0;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * static_cast<uint32_t>(i); }
};

// Writes a warp's 32 accumulator rows x D columns (fp32 in TMEM, times ``mul``)
// as bf16 (or f16: fp16) into a staging area laid out as D/64 boxes of 32 x 64
// (swizzled).
template <int D>
__device__ __forceinline__ void stage_rows_from_tmem(uint32_t taddr, uint32_t stage, int lane, float mul, bool f16) {
  auto pk2 = [f16](float x, float y) { return f16 ? pack_f16x2(x, y) : pack_bf16x2(x, y); };
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + 32 * c, v);
    tmem_ld_wait(v);
    const uint32_t cb = static_cast<uint32_t>(c >> 1), g0 = static_cast<uint32_t>((c & 1) * 4);
#pragma unroll
    for (int g = 0; g < 4; ++g)
      st_shared_v4(stage + cb * 4096 + lane * 128 + (((g0 + g) ^ static_cast<uint32_t>(lane & 7)) << 4),
                   pk2(__uint_as_float(v[8 * g + 0]) * mul, __uint_as_float(v[8 * g + 1]) * mul),
                   pk2(__uint_as_float(v[8 * g + 2]) * mul, __uint_as_float(v[8 * g + 3]) * mul),
                   pk2(__uint_as_float(v[8 * g + 4]) * mul, __uint_as_float(v[8 * g + 5]) * mul),
                   pk2(__uint_as_float(v[8 * g + 6]) * mul, __uint_as_float(v[8 * g + 7]) * mul));
  }
}

// Zeros for a warp's 32 rows x D columns (an output block no query or key reaches).
template <int D>
__device__ __forceinline__ void stage_zero_rows(uint32_t stage, int lane) {
#pragma unroll
  for (int cb = 0; cb < D / 64; ++cb)
#pragma unroll
    for (int g = 0; g < 8; ++g) st_shared_v4(stage + cb * 4096 + lane * 128 + g * 16, 0u, 0u, 0u, 0u);
}

// TMEM column offset of the A operand of K-step kk (16 columns of a 128-wide block
// whose two 64-column halves each keep their 16-bit values in their first 32 columns).
__device__ __forceinline__ uint32_t half_packed_col(int kk) {
  return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8);
}

// ------------------------------------------------------------------ dK / dV
// One CTA per (128-key block, key/value head, batch); loops over the query heads
// of the head's group and, for each, over the 128-query blocks whose Q, dO tiles
// and LSE / Dsum rows are double-buffered.  Per block: S^T = K Q^T and
// dP^T = V dO^T into TMEM; the elementwise warps turn them into P^T (fp16) and
// dS^T = P^T (dP^T - Dsum) (fp16) in place; dV += P^T dO and dK += dS^T Q with
// A from TMEM.  Each product has its own barrier so that the elementwise phases
// overlap the tensor core: P^T is computed while dP^T is, dS^T while dV is, and the
// next block's S^T (dP^T) starts as soon as this block's dV (dK) has read P^T (dS^T).
enum : int {
  K_KVF = 0, K_QF = 1 /* 2 */, K_QE = 3 /* 2 */, K_SF = 5, K_DPF = 6, K_PF = 7, K_DSF = 8, K_DVD = 9, K_ACC = 10,
  K_DR = 11, K_NB = 12
};

template <int D>
struct DkdvCfg {
  static constexpr int CH = D / 64;
  static constexpr int TILE = CH * 16384;  // 128 rows x D 16-bit values
  static constexpr int OFF_K = 0, OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;           // [stage][Q, dO]
  static constexpr int OFF_LSE = OFF_Q + 4 * TILE; // [2][128] fp32
  static constexpr int OFF_DD = OFF_LSE + 1024;    // [2][128] fp32
  static constexpr int OFF_STG = OFF_DD + 1024;    // [8 warps] 32 keys x 32 queries fp16: dS^T staging
  static constexpr int OFF_BAR = OFF_STG + 8 * 2048;
  static constexpr int OFF_MISC = OFF_BAR + K_NB * 8;
  static constexpr int USED = OFF_MISC + 16;
  static constexpr int SMEM = (USED + 1024 > 122880) ? USED + 1024 : 122880;
  static_assert(USED + 1024 <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_attn_dkdv(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmDO,
                const __grid_constant__ CUtensorMap tmDQKV, const __grid_constant__ CUtensorMap tmDS,
                const float* __restrict__ lse, const float* __restrict__ dsum, const AttnDims a, const float scale_log2,
                const float scale, const WorkOrder ord, unsigned* err, const unsigned long long timeout_ns) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const BwdCommon cm{raw + pad, raw + pad + C::OFF_BAR};
  const uint32_t sK = cm.sb + C::OFF_K, sV = cm.sb + C::OFF_V;
  auto sQ = [&](int st) { return cm.sb + C::OFF_Q + static_cast<uint32_t>((2 * st) * C::TILE); };
  auto sDO = [&](int st) { return cm.sb + C::OFF_Q + static_cast<uint32_t>((2 * st + 1) * C::TILE); };
  float* lse_s = reinterpret_cast<float*>(smem + C::OFF_LSE);
  float* dd_s = reinterpret_cast<float*>(smem + C::OFF_DD);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* never_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (a.S + BLK - 1) / BLK;
  int unit, rank;
  ord.decode(static_cast<int>(blockIdx.x), unit, rank);
  const int kb = rank;                             // low key blocks have the most causal work
  const int jkv = unit % a.Hkv, b = unit / a.Hkv;  // global key/value head
  const int shard = jkv / a.hkvN, kvh = jkv % a.hkvN;
  const int g = a.group();
  const int k0 = kb * BLK;
  const int q_start = a.causal ? kb : 0;  // 128-query blocks: the diagonal block first
  const int nq = nqb - q_start;
  const int nit = nq * g;  // (query head of the group, query block) pairs
  const int cK = a.col_k(kvh), cV = a.col_v(kvh);
  const int dcK = a.hN * D + kvh * D, dcV = (a.hN + a.hkvN + kvh) * D;  // in dQKV
  auto jq_of = [&](int it) { return kvh * g + it / nq; };
  auto q0_of = [&](int it) { return (q_start + it % nq) * BLK; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < K_NB; ++i) mbar_init(cm.bar(i), (i == K_PF || i == K_DSF) ? 8 : 1);
    *abort_flag = 0;
    *never_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();
  const WaitCtx wc{err, abort_flag, timeout_ns};
  const WaitCtx wdrain{err, never_flag, timeout_ns};
  // TMEM: S^T / P^T [0, 128), dP^T / dS^T [128, 256), dV [256, +D), dK [256 + D, +D)
  const uint32_t tDV = tmem + 256, tDK = tmem + 256 + D;

  if (warp == 8) {
    // producer warp: lane 0 issues the TMA copies; all lanes stage each block's
    // LSE and Dsum rows (plain loads: any S), published by the same barrier
    if (lane == 0) {
      mbar_arrive_expect_tx(cm.bar(K_KVF), 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_load_4d(sK + c * 16384, &tmQKV, cm.bar(K_KVF), cK + 64 * c, k0, b, shard);
        tma_load_4d(sV + c * 16384, &tmQKV, cm.bar(K_KVF), cV + 64 * c, k0, b, shard);
      }
    }
    int issued = 0;
    for (int it = 0; it < nit; ++it) {
      const int st = it & 1;
      const uint32_t ph = static_cast<uint32_t>((it >> 1) & 1);
      const int q0 = q0_of(it), jq = jq_of(it);
      const size_t row_base = (static_cast<size_t>(b) * a.H + shard * a.hN + jq) * a.S;
      if (!__all_sync(0xffffffffu, mbar_wait(cm.bar(K_QE + st), ph ^ 1u, wc))) break;
      for (int t = lane; t < BLK; t += 32) {
        const int q = q0 + t;
        const bool in = q < a.S && TP_DCHECK(row_base + q < static_cast<size_t>(a.B) * a.H * a.S, err);
        // negated, so that the elementwise phases add them with paired fp32 instructions
        lse_s[st * BLK + t] = in ? -(lse[row_base + q] * kLog2e) : 0.0f;
        dd_s[st * BLK + t] = in ? -dsum[row_base + q] : 0.0f;
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) {
        const uint32_t fb = cm.bar(K_QF + st);
        mbar_arrive_expect_tx(fb, 2 * C::TILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_4d(sQ(st) + c * 16384, &tmQKV, fb, a.col_q(jq) + 64 * c, q0, b, shard);
          tma_load_4d(sDO(st) + c * 16384, &tmDO, fb, jq * D + 64 * c, q0, b, shard);
        }
      }
      issued = it + 1;
    }
    if (lane == 0) {
      mbar_wait(cm.bar(K_KVF), 0, wdrain);
      for (int it = issued - 2 < 0 ? 0 : issued - 2; it < issued; ++it)
        mbar_wait(cm.bar(K_QF + (it & 1)), (it >> 1) & 1, wdrain);
    }
  } else if (warp == 9) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_f16(128, BLK, false, false);   // K Q^T
      constexpr uint32_t ID_P = idesc_f16(128, BLK, false, false);   // V dO^T
      constexpr uint32_t ID_DV = idesc_f16(128, D, false, true);     // P^T dO
      constexpr uint32_t ID_DK = idesc_f16(128, D, false, true);     // dS^T Q
      auto s_mmas = [&](int st) {  // S^T = K Q^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>((kk >> 2) * 16384 + (kk & 3) * 32);
          tc_mma_bf16(tmem, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ(st) + off, 16, 1024), ID_S,
                      kk > 0 ? 1u : 0u);
        }
      };
      auto dp_mmas = [&](int st) {  // dP^T = V dO^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>((kk >> 2) * 16384 + (kk & 3) * 32);
          tc_mma_bf16(tmem + 128, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO(st) + off, 16, 1024), ID_P,
                      kk > 0 ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(cm.bar(K_KVF), 0, wc) && (nit == 0 || mbar_wait(cm.bar(K_QF), 0, wc)), any = false;
      if (ok && nit > 0) {
        tc_fence_after();
        s_mmas(0);
        tc_commit(cm.bar(K_SF));
        dp_mmas(0);
        tc_commit(cm.bar(K_DPF));
        any = true;
      }
      for (int it = 0; it < nit && ok; ++it) {
        const int st = it & 1, st1 = (it + 1) & 1;
        const bool more = it + 1 < nit;
        if (!mbar_wait(cm.bar(K_PF), static_cast<uint32_t>(it & 1), wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BLK / 16; ++kk)
          tc_mma_bf16_ts(tDV, tmem + half_packed_col(kk), sdesc_sw128(sDO(st) + kk * 2048, 16384, 1024), ID_DV,
                         (it > 0 || kk > 0) ? 1u : 0u);
        tc_commit(cm.bar(K_DVD));
        if (!mbar_wait(cm.bar(K_DSF), static_cast<uint32_t>(it & 1), wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BLK / 16; ++kk)
          tc_mma_bf16_ts(tDK, tmem + 128 + half_packed_col(kk), sdesc_sw128(sQ(st) + kk * 2048, 16384, 1024), ID_DK,
                         (it > 0 || kk > 0) ? 1u : 0u);
        tc_commit(cm.bar(K_QE + st));
        tc_commit(cm.bar(K_ACC));
        if (more) {
          // the next block's S^T once this block's dV has read P^T (dK keeps the tensor
          // core busy meanwhile), its dP^T once dK has read dS^T
          if (!mbar_wait(cm.bar(K_QF + st1), static_cast<uint32_t>(((it + 1) >> 1) & 1), wc) ||
              !mbar_wait(cm.bar(K_DVD), static_cast<uint32_t>(it & 1), wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          s_mmas(st1);
          tc_commit(cm.bar(K_SF));
          if (!mbar_wait(cm.bar(K_ACC), static_cast<uint32_t>(it & 1), wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          dp_mmas(st1);
          tc_commit(cm.bar(K_DPF));
        }
      }
      if (any) {
        tc_commit(cm.bar(K_DR));
        mbar_wait(cm.bar(K_DR), 0, wdrain);
      }
    }
  } else {
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;
    const int key = k0 + r;
    const uint32_t trow = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t cS = static_cast<uint32_t>(64 * half);  // this warp's columns within a block
    bool ok = true;
    for (int it = 0; it < nit; ++it) {
      const int st = it & 1;
      const uint32_t ph = static_cast<uint32_t>((it >> 1) & 1);
      const int q0 = q0_of(it) + 64 * half;
      ok = __all_sync(0xffffffffu, mbar_wait(cm.bar(K_SF), static_cast<uint32_t>(it & 1), wc) &&
                                       mbar_wait(cm.bar(K_QF + st), ph, wc));
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = (a.causal && q0 < k0 + BLK) || (q0 + 64 > a.S) || (k0 + BLK > a.S);
      const float4* ls4 = reinterpret_cast<const float4*>(lse_s + st * BLK + 64 * half);  // -LSE * log2(e)
      const float4* ds4 = reinterpret_cast<const float4*>(dd_s + st * BLK + 64 * half);  // -Dsum
      float p[64];
      // P^T = exp(S^T / sqrt(d) - LSE), fp16, over the first half of these columns
      {
        uint32_t v[2][32];
        tmem_ld32(tmem + trow + cS, v[0]);
        tmem_ld32(tmem + trow + cS + 32, v[1]);
        tmem_ld_wait(v[0]);
        tmem_ld_wait(v[1]);
        // the exponent arguments s * scale - LSE two at a time (paired fp32 FMA; each
        // half rounded as the scalar FMA rounds it)
        const uint64_t sc2 = f32x2(scale_log2, scale_log2);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l4 = ls4[c4];
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            const int qc = 4 * c4 + u;
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(v[qc >> 5][qc & 31]), __uint_as_float(v[qc >> 5][(qc + 1) & 31])),
                                  sc2, u == 0 ? f32x2(l4.x, l4.y) : f32x2(l4.z, l4.w)),
                        x0, x1);
            p[qc] = ex2_approx(x0);
            p[qc + 1] = ex2_approx(x1);
          }
        }
      }
      if (need_mask) {  // warp-uniform: only diagonal and ragged blocks
#pragma unroll
        for (int qc = 0; qc < 64; ++qc)
          if (q0 + qc >= a.S || key >= a.S || (a.causal && key > q0 + qc)) p[qc] = 0.0f;
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = pack_f16x2(p[2 * e], p[2 * e + 1]);
        tmem_st32(tmem + trow + cS, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cm.bar(K_PF));
      // dS^T = P^T (dP^T - Dsum), fp16, over the first half of the dP^T columns
      ok = __all_sync(0xffffffffu, mbar_wait(cm.bar(K_DPF), static_cast<uint32_t>(it & 1), wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t dk[32];
      {
        uint32_t v[2][32];
        tmem_ld32(tmem + trow + 128 + cS, v[0]);
        tmem_ld32(tmem + trow + 128 + cS + 32, v[1]);
        tmem_ld_wait(v[0]);
        tmem_ld_wait(v[1]);
        // P * (dP - Dsum) two at a time (paired fp32 add and multiply)
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 d4 = ds4[c4];
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            const int qc = 4 * c4 + u;
            const uint64_t t = add_f32x2(f32x2(__uint_as_float(v[qc >> 5][qc & 31]),
                                               __uint_as_float(v[qc >> 5][(qc + 1) & 31])),
                                         u == 0 ? f32x2(d4.x, d4.y) : f32x2(d4.z, d4.w));
            float y0, y1;
            f32x2_split(mul_f32x2(f32x2(p[qc], p[qc + 1]), t), y0, y1);
            dk[2 * c4 + u / 2] = pack_f16x2(y0, y1);
          }
        }
      }
      tmem_st32(tmem + trow + 128 + cS, dk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cm.bar(K_DSF));
      {
        // the same dS^T values (the warp's 32 keys x the half's 64 queries) to the dS
        // tile of (query head, query block, key block), from which k_attn_dq forms dQ:
        // two 32 x 32 boxes staged in the warp's 2 KB (64-byte rows, 64-byte swizzle)
        // and written by TMA, after dS^T has been handed to the dK product, so that
        // the copies overlap it
        const long long tile = ds_tile_index(a, b, shard * a.hN + jq_of(it), q_start + it % nq, kb);
        const uint32_t stg = cm.sb + C::OFF_STG + static_cast<uint32_t>(warp * 2048);
        const bool tile_ok = TP_DCHECK(tile >= 0 && tile < ds_tiles(a), err);
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          if (lane == 0) bulk_wait_read0();  // the previous box has left the staging area
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_shared_v4(stg + lane * 64 + ((static_cast<uint32_t>(c) ^ ((lane >> 1) & 3)) << 4), dk[16 * rr + 4 * c],
                         dk[16 * rr + 4 * c + 1], dk[16 * rr + 4 * c + 2], dk[16 * rr + 4 * c + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && tile_ok) {
            tma_store_2d(&tmDS, stg, 64 * half + 32 * rr, static_cast<int>(tile * BLK) + quad * 32);
            bulk_commit();
          }
        }
      }
    }
    if (ok && nit > 0) ok = __all_sync(0xffffffffu, mbar_wait(cm.bar(K_ACC), static_cast<uint32_t>((nit - 1) & 1), wc));
    if (ok) {
      tc_fence_after();
      // all MMAs are complete: the Q/dO stages are free for staging (8 warps x CH x 4 KB)
      const uint32_t stage = cm.sb + C::OFF_Q + static_cast<uint32_t>((half * 4 + quad) * C::CH * 4096);
      if (nit > 0)
        stage_rows_from_tmem<D>((half == 0 ? tDV : tDK) + trow, stage, lane, half == 0 ? 1.0f : scale,
                                a.dqkv_f16 != 0);
      else
        stage_zero_rows<D>(stage, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && k0 + quad * 32 < a.S) {
        const int col = half == 0 ? dcV : dcK;
#pragma unroll
        for (int cb = 0; cb < C::CH; ++cb) tma_store_4d(&tmDQKV, stage + cb * 4096, col + 64 * cb, k0 + quad * 32, b, shard);
        bulk_commit();
      }
    }
    __syncwarp();
    if (lane == 0) bulk_wait0();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------- dQ
// dQ = sum over key blocks of dS K / sqrt(d), from the dS tiles the dK/dV kernel
// wrote: no score, probability or dP recomputation, one product per block.  One
// CTA per (128-query block, query head, batch), heaviest causal blocks first.
// Each stage holds one key block's dS^T tile (the MMA's A operand, MN-major: two
// 64-query chunks of 128 key rows) and its K tile (B, MN-major, D/64 chunks); the
// fp32 accumulator (128 x D) stays in TMEM.
//   warp 4: TMA producer; warp 5: MMA issuer (one elected thread);
//   warps 0-3: epilogue (TMEM lane quadrant w), dQ scaled and stored once at the end.
constexpr int kDqStages = 3;
constexpr int DQ_THREADS = 192;
enum : int { Q_F = 0 /* [stage] */, Q_E = kDqStages /* [stage] */, Q_ACC = 2 * kDqStages, Q_DR, Q_NB };

template <int D>
struct DqCfg {
  static constexpr int CH = D / 64;
  static constexpr int DS_BYTES = 2 * 16384;       // 128 keys x 128 queries, fp16
  static constexpr int K_BYTES = CH * 16384;       // 128 keys x D, fp16
  static constexpr int STAGE = DS_BYTES + K_BYTES;
  static constexpr int OFF_BAR = kDqStages * STAGE;
  static constexpr int OFF_MISC = OFF_BAR + Q_NB * 8;
  static constexpr int USED = OFF_MISC + 16;
  static constexpr int SMEM = USED + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(DQ_THREADS, 1)
    k_attn_dq(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmDS,
              const __grid_constant__ CUtensorMap tmDQKV, const AttnDims a, const float scale, const WorkOrder ord,
              unsigned* err, const unsigned long long timeout_ns) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const BwdCommon cm{raw + pad, raw + pad + C::OFF_BAR};
  auto sDS = [&](int st) { return cm.sb + static_cast<uint32_t>(st * C::STAGE); };
  auto sK = [&](int st) { return cm.sb + static_cast<uint32_t>(st * C::STAGE + C::DS_BYTES); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* never_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = (a.S + BLK - 1) / BLK;
  int unit, rank;
  ord.decode(static_cast<int>(blockIdx.x), unit, rank);
  const int qb = nb - 1 - rank;  // the last query blocks have the most causal work
  const int j = unit % a.H, b = unit / a.H;
  const int shard = j / a.hN, jj = j % a.hN, kvh = jj / a.group();
  const int q0 = qb * BLK;
  const int nkv = a.causal ? qb + 1 : nb;
  const int cK = a.col_k(kvh);
  const long long tile0 = ds_tile_index(a, b, j, qb, 0);  // the key blocks' tiles are consecutive

  if (threadIdx.x == 0) {
    for (int i = 0; i < Q_NB; ++i) mbar_init(cm.bar(i), 1);
    *abort_flag = 0;
    *never_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();
  const WaitCtx wc{err, abort_flag, timeout_ns};
  const WaitCtx wdrain{err, never_flag, timeout_ns};

  if (warp == 4) {
    if (lane == 0) {
      const bool coords_ok = TP_DCHECK(cK % 8 == 0 && tile0 >= 0 && tile0 + nkv <= ds_tiles(a), err);
      int issued = 0;
      for (int kb = 0; kb < nkv && coords_ok; ++kb) {
        const int st = kb % kDqStages;
        if (!mbar_wait(cm.bar(Q_E + st), static_cast<uint32_t>(((kb / kDqStages) & 1) ^ 1), wc)) break;
        mbar_arrive_expect_tx(cm.bar(Q_F + st), C::STAGE);
        const int row = static_cast<int>((tile0 + kb) * BLK);
        tma_load_2d(sDS(st), &tmDS, cm.bar(Q_F + st), 0, row);
        tma_load_2d(sDS(st) + 16384, &tmDS, cm.bar(Q_F + st), 64, row);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          tma_load_4d(sK(st) + c * 16384, &tmQKV, cm.bar(Q_F + st), cK + 64 * c, kb * BLK, b, shard);
        issued = kb + 1;
      }
      // every issued copy lands before the CTA may exit
      for (int k = (issued > kDqStages ? issued - kDqStages : 0); k < issued; ++k)
        mbar_wait(cm.bar(Q_F + k % kDqStages), static_cast<uint32_t>((k / kDqStages) & 1), wdrain);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // D (queries x d) += A (dS: queries x keys, MN-major) B (K: keys x d, MN-major)
      constexpr uint32_t ID_DQ = idesc_f16(128, D, true, true);
      bool ok = true, any = false;
      for (int kb = 0; kb < nkv && ok; ++kb) {
        const int st = kb % kDqStages;
        if (!mbar_wait(cm.bar(Q_F + st), static_cast<uint32_t>((kb / kDqStages) & 1), wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BLK / 16; ++kk)
          tc_mma_bf16(tmem, sdesc_sw128(sDS(st) + kk * 2048, 16384, 1024), sdesc_sw128(sK(st) + kk * 2048, 16384, 1024),
                      ID_DQ, (kb > 0 || kk > 0) ? 1u : 0u);
        tc_commit(cm.bar(Q_E + st));
        any = true;
      }
      if (ok && any) tc_commit(cm.bar(Q_ACC));
      if (any) {
        tc_commit(cm.bar(Q_DR));
        mbar_wait(cm.bar(Q_DR), 0, wdrain);
      }
    }
  } else {
    const int quad = warp;
    bool ok = nkv == 0 || __all_sync(0xffffffffu, mbar_wait(cm.bar(Q_ACC), 0, wc));
    if (ok) {
      tc_fence_after();
      // every MMA is complete: stage 0's dS buffer is free for staging
      const uint32_t stage = sDS(0) + static_cast<uint32_t>(quad * C::CH * 4096);
      if (nkv > 0)
        stage_rows_from_tmem<D>(tmem + (static_cast<uint32_t>(quad * 32) << 16), stage, lane, scale, a.dqkv_f16 != 0);
      else
        stage_zero_rows<D>(stage, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && q0 + quad * 32 < a.S) {
#pragma unroll
        for (int cb = 0; cb < C::CH; ++cb)
          tma_store_4d(&tmDQKV, stage + cb * 4096, jj * D + 64 * cb, q0 + quad * 32, b, shard);
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
    tmem_dealloc(tmem, 128);
  }
}

template <int D>
int launch_bwd_d(const AttnDims& a, const void* qkv, const void* o, const void* dout, const float* lse, float* dsum,
                 void* dsbuf, void* dqkv, unsigned* err, unsigned long long timeout_ns, cudaStream_t st) {
  static std::atomic<bool> configured_kv[kMaxDevices], configured_q[kMaxDevices];
  if (!set_smem_limit_once(reinterpret_cast<const void*>(k_attn_dkdv<D>), DkdvCfg<D>::SMEM, configured_kv) ||
      !set_smem_limit_once(reinterpret_cast<const void*>(k_attn_dq<D>), DqCfg<D>::SMEM, configured_q))
    return 2;
  // the dS tiles: [tiles * 128 key rows][128 query columns] fp16; written in 32 x 32
  // boxes (64-byte swizzle) by dK/dV, read in 64 x 128 boxes (128-byte swizzle) by dQ
  CUtensorMap tds, tds_st;
  {
    const uint64_t dd[2] = {128u, static_cast<uint64_t>(ds_tiles(a)) * 128u};
    const uint32_t dbox[2] = {64, 128}, sbox[2] = {32, 32};
    if (!encode_tmap(&tds, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, dsbuf, dd, dbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap(&tds_st, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, dsbuf, dd, sbox, CU_TENSOR_MAP_SWIZZLE_64B))
      return 2;
  }
  const uint64_t S = static_cast<uint64_t>(a.S), Bb = static_cast<uint64_t>(a.B), Nn = static_cast<uint64_t>(a.N);
  CUtensorMap tq, tdo, tdq;
  const uint64_t qd[4] = {static_cast<uint64_t>(a.qkv_width()), S, Bb, Nn};
  const uint64_t gd[4] = {static_cast<uint64_t>(a.dqkv_width()), S, Bb, Nn};
  const uint64_t od[4] = {static_cast<uint64_t>(a.hN) * D, S, Bb, Nn};
  const uint32_t box128[4] = {64, 128, 1, 1};
  const uint32_t box32[4] = {64, 32, 1, 1};
  // 16-bit elements (fp16 Q, K, V, dO; O fp16 or bf16; bf16 dQKV): the copies do not interpret them
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!encode_tmap(&tq, bf, 4, qkv, qd, box128, sw) || !encode_tmap(&tdo, bf, 4, dout, od, box128, sw) ||
      !encode_tmap(&tdq, bf, 4, dqkv, gd, box32, sw))
    return 2;

  const long long rows = static_cast<long long>(a.N) * a.B * a.S * a.hN;
  const int sms = device_sm_count();
  if (rows >= (1ll << 31)) return 1;                // Dsum's 32-bit row indices
  long long blocks = (rows * (D / 8) + 255) / 256;  // D/8 lanes per row
  if (blocks > static_cast<long long>(sms) * 8) blocks = static_cast<long long>(sms) * 8;
  int slot = timing_begin(kKAttnDsum, st);
  bool ok = launch_k(k_attn_dsum<D>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1,
                     static_cast<const uint4*>(o), static_cast<const uint4*>(dout), dsum, a, err) == cudaSuccess;
  timing_end(slot, st);
  if (!ok) return 2;
  const int nb = (a.S + BLK - 1) / BLK;
  const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  const float scale_log2 = scale * kLog2e;
  const WorkOrder ord_q = make_work_order(a.B * a.H, nb, sms), ord_kv = make_work_order(a.B * a.Hkv, nb, sms);
  slot = timing_begin(kKAttnDkdv, st);
  ok = launch_k(k_attn_dkdv<D>, dim3(ord_kv.ctas()), dim3(NTHREADS), DkdvCfg<D>::SMEM, st, 1, tq, tdo, tdq, tds_st,
                lse, dsum, a, scale_log2, scale, ord_kv, err, timeout_ns) == cudaSuccess;
  timing_end(slot, st);
  if (!ok) return 2;
  slot = timing_begin(kKAttnDq, st);
  ok = launch_k(k_attn_dq<D>, dim3(ord_q.ctas()), dim3(DQ_THREADS), DqCfg<D>::SMEM, st, 1, tq, tds, tdq, a, scale,
                ord_q, err, timeout_ns) == cudaSuccess;
  timing_end(slot, st);
  return ok ? 0 : 2;
}

}  // namespace

int launch_attn_bwd(const AttnDims& a, const void* qkv, const void* o, const void* dout, const float* lse,
                    float* dsum, void* dsbuf, void* dqkv, unsigned* err, unsigned long long timeout_ns,
                    cudaStream_t st) {
  if (!dsbuf || (reinterpret_cast<uintptr_t>(dsbuf) & 15u)) return 1;
  if (a.B < 1 || a.S < 1 || a.H < 1 || a.N < 1 || a.hN * a.N != a.H) return 1;
  if (a.Hkv < 1 || a.hkvN * a.N != a.Hkv || a.H % a.Hkv || a.hN % a.hkvN) return 1;
  if (a.H > 65535 || a.B > 65535) return 1;
  if (a.d == 128) return launch_bwd_d<128>(a, qkv, o, dout, lse, dsum, dsbuf, dqkv, err, timeout_ns, st);
  if (a.d == 64) return launch_bwd_d<64>(a, qkv, o, dout, lse, dsum, dsbuf, dqkv, err, timeout_ns, st);
  return 1;
}

}  // namespace tpb
