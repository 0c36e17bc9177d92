// Fused per-head attention forward on tcgen05:
//   O_j = softmax(mask(Q_j K_j^T / sqrt(d))) V_j,  LSE = log sum exp(scaled scores)
// (damodev 3D并行 §1.2.2 per-head attention; the blockwise online-softmax
// recurrence is the one sunjinbo 并行方式 §CP uses to combine per-block results).
//
// One CTA per (128-query block, head, batch), heaviest causal blocks first.
//   warp 4: TMA producer (Qh, Ql once; Kh, Kl and V per block of 128 keys)
//   warp 5: MMA issuer: S = Qh Kh^T + Qh Kl^T + Ql Kh^T into one of two TMEM score
//           buffers, then O_blk = P V into a TMEM output buffer (P from shared memory)
//   warps 0-3: one query row per thread: row max, exp2, P (bf16) to shared memory,
//           running (m, l) and the fp32 output row in registers, rescaled per block
// S for block j+1 is computed while the softmax threads work on block j.
#include <cmath>

#include "attn.cuh"
#include "host_util.cuh"
#include "ptx.cuh"

namespace tpb {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int NTHREADS = 192;

enum : int {
  B_QF = 0, B_KF, B_KE, B_VF, B_VE, B_SF0, B_SF1, B_SE0, B_SE1, B_PF, B_PE, B_OF, B_OE, B_DR, NBARS
};

template <int D>
struct FwdCfg {
  static constexpr int CH = D / 64;
  static constexpr int TILE = CH * 16384;  // 128 rows x D bf16 as 64-column swizzled chunks
  static constexpr int OFF_QH = 0, OFF_QL = TILE, OFF_KH = 2 * TILE, OFF_KL = 3 * TILE, OFF_V = 4 * TILE;
  static constexpr int OFF_P = 5 * TILE;
  static constexpr int OFF_BAR = OFF_P + 32768;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int USED = OFF_MISC + 16;
  // at least 120 KB so that one CTA (and its 512 TMEM columns) holds an SM
  static constexpr int SMEM = (USED + 1024 > 122880) ? USED + 1024 : 122880;
};

// S (+)= A B^T over K = D for K-major 128-row tiles in 64-column swizzled chunks.
template <int D>
__device__ __forceinline__ void mma_rows_kmajor(uint32_t d_tmem, uint32_t sa, uint32_t sb, uint32_t idesc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>((kk >> 2) * 16384 + (kk & 3) * 32);
    tc_mma_bf16(d_tmem, sdesc_sw128(sa + off, 16, 1024), sdesc_sw128(sb + off, 16, 1024), idesc,
                (acc || kk > 0) ? 1u : 0u);
  }
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_attn_fwd(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmO, const AttnDims a,
               float* __restrict__ lse, const float scale_log2, unsigned* err, const unsigned long long timeout_ns) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t bar0 = sb + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* never_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  const uint32_t sQh = sb + C::OFF_QH, sQl = sb + C::OFF_QL, sKh = sb + C::OFF_KH, sKl = sb + C::OFF_KL;
  const uint32_t sV = sb + C::OFF_V, sP = sb + C::OFF_P;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (a.S + BQ - 1) / BQ;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.x);
  const int j = blockIdx.y, b = blockIdx.z;
  const int shard = j / a.hN, jj = j % a.hN;
  const int q0 = qb * BQ;
  const int nkb = (a.S + BKV - 1) / BKV;
  const int nkv = a.causal ? min(qb + 1, nkb) : nkb;
  const int cQh = jj * D, cKh = (a.hN + jj) * D, cV = (2 * a.hN + jj) * D;
  const int cQl = (3 * a.hN + jj) * D, cKl = (4 * a.hN + jj) * D;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBARS; ++i) {
      const bool by_warps = (i == B_SE0 || i == B_SE1 || i == B_PF || i == B_OE);
      mbar_init(bar(i), by_warps ? 4 : 1);
    }
    *abort_flag = 0;
    *never_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&tmQKV);
    prefetch_tmap(&tmO);
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

  if (warp == 4) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int kiss = 0, viss = 0;
      mbar_arrive_expect_tx(bar(B_QF), 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_load_4d(sQh + c * 16384, &tmQKV, bar(B_QF), cQh + 64 * c, q0, b, shard);
        tma_load_4d(sQl + c * 16384, &tmQKV, bar(B_QF), cQl + 64 * c, q0, b, shard);
      }
      for (int kv = 0; kv < nkv; ++kv) {
        const uint32_t ph = static_cast<uint32_t>(kv & 1);
        if (!mbar_wait(bar(B_KE), ph ^ 1u, wc)) break;
        mbar_arrive_expect_tx(bar(B_KF), 2 * C::TILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_4d(sKh + c * 16384, &tmQKV, bar(B_KF), cKh + 64 * c, kv * BKV, b, shard);
          tma_load_4d(sKl + c * 16384, &tmQKV, bar(B_KF), cKl + 64 * c, kv * BKV, b, shard);
        }
        kiss = kv + 1;
        if (!mbar_wait(bar(B_VE), ph ^ 1u, wc)) break;
        mbar_arrive_expect_tx(bar(B_VF), C::TILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          tma_load_4d(sV + c * 16384, &tmQKV, bar(B_VF), cV + 64 * c, kv * BKV, b, shard);
        viss = kv + 1;
      }
      mbar_wait(bar(B_QF), 0, wdrain);
      if (kiss) mbar_wait(bar(B_KF), (kiss - 1) & 1, wdrain);
      if (viss) mbar_wait(bar(B_VF), (viss - 1) & 1, wdrain);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_PV = idesc_bf16(128, D, false, true);
      bool ok = mbar_wait(bar(B_QF), 0, wc), any = false;
      auto issue_s = [&](int kv) -> bool {
        const int st = kv & 1;
        const uint32_t ph = static_cast<uint32_t>((kv >> 1) & 1);
        if (!mbar_wait(bar(B_KF), kv & 1, wc)) return false;
        if (!mbar_wait(bar(B_SE0 + st), ph ^ 1u, wc)) return false;
        tc_fence_after();
        const uint32_t dt = tmem + static_cast<uint32_t>(st * 128);
        mma_rows_kmajor<D>(dt, sQh, sKh, ID_S, false);
        mma_rows_kmajor<D>(dt, sQh, sKl, ID_S, true);
        mma_rows_kmajor<D>(dt, sQl, sKh, ID_S, true);
        any = true;
        tc_commit(bar(B_KE));
        tc_commit(bar(B_SF0 + st));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int kv = 0; kv < nkv && ok; ++kv) {
        if (kv + 1 < nkv && !issue_s(kv + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(bar(B_PF), kv & 1, wc) || !mbar_wait(bar(B_VF), kv & 1, wc) ||
            !mbar_wait(bar(B_OE), (kv & 1) ^ 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(sP + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sV + kk * 2048, 16384, 1024);
          tc_mma_bf16(tmem + 256, ad, bd, ID_PV, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(B_VE));
        tc_commit(bar(B_PE));
        tc_commit(bar(B_OF));
      }
      if (any) {
        tc_commit(bar(B_DR));
        mbar_wait(bar(B_DR), 0, wdrain);
      }
    }
  } else {
    // -------------------------------------------------------------- softmax / output
    const int r = warp * 32 + lane;
    const int q = q0 + r;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t rsw = static_cast<uint32_t>(r & 7);
    float o[D];
#pragma unroll
    for (int e = 0; e < D; ++e) o[e] = 0.0f;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int kv = 0; kv < nkv; ++kv) {
      const int st = kv & 1;
      const uint32_t ph = static_cast<uint32_t>((kv >> 1) & 1);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B_SF0 + st), ph, wc));
      if (!ok) break;
      tc_fence_after();
      const bool masked = (a.causal && kv == qb) || ((kv + 1) * BKV > a.S);
      const int kbase = kv * BKV;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(trow + st * 128 + 32 * c, v);
        tmem_ld_wait(v);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float s = __uint_as_float(v[e]) * scale_log2;
          if (masked) {
            const int key = kbase + 32 * c + e;
            if (key >= a.S || (a.causal && key > q)) s = -INFINITY;
          }
          mx = fmaxf(mx, s);
        }
      }
      const float m_new = fmaxf(m, mx);
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
      const float alpha = exp2f(m - m_use);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B_PE), (kv & 1) ^ 1, wc));
      if (!ok) break;
      float ls = 0.0f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(trow + st * 128 + 32 * c, v);
        tmem_ld_wait(v);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float s0 = __uint_as_float(v[e]) * scale_log2, s1 = __uint_as_float(v[e + 1]) * scale_log2;
          if (masked) {
            const int key = kbase + 32 * c + e;
            if (key >= a.S || (a.causal && key > q)) s0 = -INFINITY;
            if (key + 1 >= a.S || (a.causal && key + 1 > q)) s1 = -INFINITY;
          }
          const uint32_t pp = pack_bf16x2(exp2f(s0 - m_use), exp2f(s1 - m_use));
          ls += bf16lo_to_f32(pp) + bf16hi_to_f32(pp);
          pk[e >> 1] = pp;
        }
        const uint32_t kc = static_cast<uint32_t>(c >> 1), g0 = static_cast<uint32_t>((c & 1) * 4);
#pragma unroll
        for (int g = 0; g < 4; ++g)
          st_shared_v4(sP + kc * 16384 + r * 128 + (((g0 + g) ^ rsw) << 4), pk[4 * g], pk[4 * g + 1], pk[4 * g + 2],
                       pk[4 * g + 3]);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_SE0 + st));
        mbar_arrive(bar(B_PF));
      }
      l = l * alpha + ls;
      m = m_new;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B_OF), kv & 1, wc));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(trow + 256 + 32 * c, v);
        tmem_ld_wait(v);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[32 * c + e] = fmaf(o[32 * c + e], alpha, __uint_as_float(v[e]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OE));
    }
    if (ok) {
      // every P.V product is complete, so the P buffer is free: stage O there
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      const uint32_t stage = sP + static_cast<uint32_t>(warp * C::CH * 4096);
#pragma unroll
      for (int cb = 0; cb < C::CH; ++cb)
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float* x = &o[64 * cb + 8 * g];
          st_shared_v4(stage + cb * 4096 + lane * 128 + ((static_cast<uint32_t>(g) ^ static_cast<uint32_t>(lane & 7)) << 4),
                       pack_bf16x2(x[0] * inv, x[1] * inv), pack_bf16x2(x[2] * inv, x[3] * inv),
                       pack_bf16x2(x[4] * inv, x[5] * inv), pack_bf16x2(x[6] * inv, x[7] * inv));
        }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && q0 + warp * 32 < a.S) {
#pragma unroll
        for (int cb = 0; cb < C::CH; ++cb) tma_store_4d(&tmO, stage + cb * 4096, jj * D + 64 * cb, q0 + warp * 32, b, shard);
        bulk_commit();
      }
      if (q < a.S) lse[(static_cast<size_t>(b) * a.H + j) * a.S + q] = (m + log2f(l)) * 0.6931471805599453f;
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
int launch_fwd_d(const AttnDims& a, const void* qkv, void* o, float* lse, unsigned* err, unsigned long long timeout_ns,
                 cudaStream_t st) {
  using C = FwdCfg<D>;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(k_attn_fwd<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return 2;
    configured = true;
  }
  CUtensorMap tq, to;
  const uint64_t qd[4] = {static_cast<uint64_t>(kQkvPlanes) * a.hN * D, static_cast<uint64_t>(a.S),
                          static_cast<uint64_t>(a.B), static_cast<uint64_t>(a.N)};
  const uint32_t qbox[4] = {64, 128, 1, 1};
  const uint64_t od[4] = {static_cast<uint64_t>(a.hN) * D, static_cast<uint64_t>(a.S), static_cast<uint64_t>(a.B),
                          static_cast<uint64_t>(a.N)};
  const uint32_t obox[4] = {64, 32, 1, 1};
  if (!encode_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, qkv, qd, qbox, CU_TENSOR_MAP_SWIZZLE_128B)) return 2;
  if (!encode_tmap(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, o, od, obox, CU_TENSOR_MAP_SWIZZLE_128B)) return 2;
  const int nqb = (a.S + BQ - 1) / BQ;
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  dim3 grid(nqb, a.H, a.B);
  const int slot = timing_begin(kKAttnCore, st);
  k_attn_fwd<D><<<grid, NTHREADS, C::SMEM, st>>>(tq, to, a, lse, scale_log2, err, timeout_ns);
  const bool ok = cudaGetLastError() == cudaSuccess;
  timing_end(slot, st);
  return ok ? 0 : 2;
}

}  // namespace

int launch_attn_fwd(const AttnDims& a, const void* qkv, void* o, float* lse, unsigned* err,
                    unsigned long long timeout_ns, cudaStream_t st) {
  if (a.B < 1 || a.S < 1 || a.H < 1 || a.N < 1 || a.hN * a.N != a.H) return 1;
  if (a.H > 65535 || a.B > 65535) return 1;
  if (a.d == 128) return launch_fwd_d<128>(a, qkv, o, lse, err, timeout_ns, st);
  if (a.d == 64) return launch_fwd_d<64>(a, qkv, o, lse, err, timeout_ns, st);
  return 1;
}

}  // namespace tpb
