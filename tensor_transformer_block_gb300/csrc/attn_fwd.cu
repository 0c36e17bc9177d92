// Fused per-head attention forward on tcgen05:
//   O_j = softmax(mask(Q_j K_j^T / sqrt(d))) V_j,  LSE = log sum exp(scaled scores)
// (damodev 3D并行 §1.2.2 per-head attention; the blockwise online-softmax
// recurrence is the one sunjinbo 并行方式 §CP uses to combine per-block results).
//
// One CTA per (256 queries = two 128-query tiles, query head, batch), heaviest
// causal blocks first; the key/value tiles are those of the head's group.  Keys are processed in blocks of 64; K and V each have two
// shared-memory stages, so the copies of block kv+1 overlap the work on block kv.
//   warp 8: TMA producer: both tiles' Qh, Ql once; Kh, Kl and V per key block
//   warp 9: MMA issuer: per key block, S = Qh Kh^T + Qh Kl^T + Ql Kh^T (split-bf16
//           scores) for each tile into one of the tile's two TMEM score buffers,
//           then O_tile += P V with P read from TMEM and V from shared memory
//   warps 0-3 / 4-7: the softmax warpgroup of tile 0 / tile 1, one query row per
//           thread: one TMEM read of the score block, masked row max, exp2, and P
//           (bf16) written over the first half of the same score buffer.  The
//           running max is only moved (and the row of O in TMEM rescaled) when a
//           block's max exceeds it by more than 8 (log2 units); otherwise the stale
//           max stays, P <= 2^8, and the final O / l is unchanged because the max
//           cancels.  Only a rescale waits for the previous block's P V, so the
//           softmax of block kv+1 overlaps the P V of block kv, and while one
//           warpgroup works on its softmax the tensor core works on the other tile.
// TMEM (512 columns): tile t's score buffers at 128 t and 128 t + 64 (64 columns;
// P, 64 bf16 per row, in their first 32), its O at 256 + 128 t.  A score buffer
// is refilled (block kv+2) only once the P V that read its P (block kv) is done.
// P ready / P V done for even and odd blocks go to separate barriers, and every
// waiter observes block kv-2 before it waits for block kv, so a parity wait never
// meets a barrier two phases away from it (the softmax of block kv+1 may finish
// before the MMA warp has taken block kv's P).
#include <cmath>

#include "attn.cuh"
#include "host_util.cuh"
#include "ptx.cuh"

namespace tpb {
namespace {

constexpr int BQ = 128;    // queries per tile
constexpr int QT = 2;      // tiles per CTA
constexpr int BKV = 64;    // keys per block
constexpr int NTHREADS = 320;
constexpr int WARP_PRODUCER = 8;
constexpr int WARP_MMA = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256

enum : int {
  B_QF = 0,
  B_KF = 1,   // [stage]: 1, 2
  B_KE = 3,   // [stage]: 3, 4
  B_VF = 5,   // [stage]: 5, 6
  B_VE = 7,   // [stage]: 7, 8
  B_SF = 9,   // [tile][buffer]: scores ready (9..12)
  B_PF = 13,  // [tile][block parity]: P written to TMEM, 4 arrivals (13..16)
  B_PE = 17,  // [tile][block parity]: P.V complete (17..20)
  B_DR = 21, NBARS = 22
};

template <int D>
struct FwdCfg {
  static constexpr int CH = D / 64;
  static constexpr int QTILE = CH * 16384;   // 128 rows x D bf16 in 64-column swizzled chunks
  static constexpr int KTILE = CH * 8192;    // 64 rows x D
  static constexpr int OFF_Q = 0;            // [tile][hi, lo]
  static constexpr int OFF_K = 4 * QTILE;    // [stage][hi, lo]
  static constexpr int OFF_V = OFF_K + 4 * KTILE;  // [stage]
  static constexpr int OFF_BAR = OFF_V + 2 * KTILE;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int USED = OFF_MISC + 16;
  // at least 120 KB so that a second CTA (which would wait for the TMEM this one
  // holds) never shares the SM
  static constexpr int SMEM = (USED + 1024 > 122880) ? USED + 1024 : 122880;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(D <= 128, "head dim");
};

// S (+)= A B^T over K = D: A a 128-row tile (16 KB chunks), B a 64-row tile (8 KB chunks).
template <int D>
__device__ __forceinline__ void mma_scores(uint32_t d_tmem, uint32_t sa, uint32_t sb, uint32_t idesc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t in = static_cast<uint32_t>((kk & 3) * 32), kc = static_cast<uint32_t>(kk >> 2);
    tc_mma_bf16(d_tmem, sdesc_sw128(sa + kc * 16384 + in, 16, 1024), sdesc_sw128(sb + kc * 8192 + in, 16, 1024), idesc,
                (acc || kk > 0) ? 1u : 0u);
  }
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_attn_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
               const __grid_constant__ CUtensorMap tmO, const AttnDims a, float* __restrict__ lse,
               const float scale_log2, unsigned* err, const unsigned long long timeout_ns) {
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
  auto sQ = [&](int t, int lo) { return sb + C::OFF_Q + static_cast<uint32_t>((2 * t + lo) * C::QTILE); };
  auto sKh = [&](int st) { return sb + C::OFF_K + static_cast<uint32_t>(2 * st * C::KTILE); };
  auto sKl = [&](int st) { return sb + C::OFF_K + static_cast<uint32_t>((2 * st + 1) * C::KTILE); };
  auto sV = [&](int st) { return sb + C::OFF_V + static_cast<uint32_t>(st * C::KTILE); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (a.S + QT * BQ - 1) / (QT * BQ);
  const int qb = nqb - 1 - static_cast<int>(blockIdx.x);
  const int j = blockIdx.y, b = blockIdx.z;
  const int shard = j / a.hN, jj = j % a.hN, kvh = jj / a.group();
  const int q0 = qb * QT * BQ;
  const int nkb = (a.S + BKV - 1) / BKV;
  // key blocks each tile needs (causal: up to its last query)
  int nkv_t[QT];
#pragma unroll
  for (int t = 0; t < QT; ++t) {
    const int qlast = min(q0 + (t + 1) * BQ, a.S) - 1;
    nkv_t[t] = (q0 + t * BQ >= a.S) ? 0 : (a.causal ? min(qlast / BKV + 1, nkb) : nkb);
  }
  const int nkv = max(nkv_t[0], nkv_t[1]);
  const int cQh = a.col_q(jj), cKh = a.col_k(kvh), cV = a.col_v(kvh);
  const int cQl = a.col_ql(jj), cKl = a.col_kl(kvh);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBARS; ++i) {
      const bool by_warps = i >= B_PF && i < B_PF + 2 * QT;
      mbar_init(bar(i), by_warps ? 4 : 1);
    }
    *abort_flag = 0;
    *never_flag = 0;
    fence_mbar_init();
  }
  if (warp == WARP_PRODUCER && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmKV);
    prefetch_tmap(&tmO);
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{err, abort_flag, timeout_ns};
  const WaitCtx wdrain{err, never_flag, timeout_ns};

  if (warp == WARP_PRODUCER) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int kiss = 0, viss = 0;  // key blocks whose K / V copies were issued
      mbar_arrive_expect_tx(bar(B_QF), 4 * C::QTILE);
#pragma unroll
      for (int t = 0; t < QT; ++t)
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_4d(sQ(t, 0) + c * 16384, &tmQ, bar(B_QF), cQh + 64 * c, q0 + t * BQ, b, shard);
          tma_load_4d(sQ(t, 1) + c * 16384, &tmQ, bar(B_QF), cQl + 64 * c, q0 + t * BQ, b, shard);
        }
      for (int kv = 0; kv < nkv; ++kv) {
        const int st = kv & 1;
        const uint32_t ph = static_cast<uint32_t>((kv >> 1) & 1);
        if (!mbar_wait(bar(B_KE + st), ph ^ 1u, wc)) break;
        mbar_arrive_expect_tx(bar(B_KF + st), 2 * C::KTILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_4d(sKh(st) + c * 8192, &tmKV, bar(B_KF + st), cKh + 64 * c, kv * BKV, b, shard);
          tma_load_4d(sKl(st) + c * 8192, &tmKV, bar(B_KF + st), cKl + 64 * c, kv * BKV, b, shard);
        }
        kiss = kv + 1;
        if (!mbar_wait(bar(B_VE + st), ph ^ 1u, wc)) break;
        mbar_arrive_expect_tx(bar(B_VF + st), C::KTILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          tma_load_4d(sV(st) + c * 8192, &tmKV, bar(B_VF + st), cV + 64 * c, kv * BKV, b, shard);
        viss = kv + 1;
      }
      // every issued copy lands before the CTA may exit
      mbar_wait(bar(B_QF), 0, wdrain);
      for (int k = (kiss > 2 ? kiss - 2 : 0); k < kiss; ++k)
        mbar_wait(bar(B_KF + (k & 1)), static_cast<uint32_t>((k >> 1) & 1), wdrain);
      for (int k = (viss > 2 ? viss - 2 : 0); k < viss; ++k)
        mbar_wait(bar(B_VF + (k & 1)), static_cast<uint32_t>((k >> 1) & 1), wdrain);
    }
  } else if (warp == WARP_MMA) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t ID_S = idesc_bf16(128, BKV, false, false);
      constexpr uint32_t ID_PV = idesc_bf16(128, D, false, true);
      bool ok = mbar_wait(bar(B_QF), 0, wc), any = false;
      // scores of key block kv for every tile that needs it, then release the K stage
      auto issue_s = [&](int kv) -> bool {
        const int st = kv & 1;
        if (!mbar_wait(bar(B_KF + st), static_cast<uint32_t>((kv >> 1) & 1), wc)) return false;
#pragma unroll
        for (int t = 0; t < QT; ++t) {
          if (kv >= nkv_t[t]) continue;
          // the P V of block kv-2 has read the P this buffer held
          if (kv >= 2 && !mbar_wait(bar(B_PE + 2 * t + st), static_cast<uint32_t>(((kv - 2) >> 1) & 1), wc))
            return false;
          tc_fence_after();
          const uint32_t dt = tmem + static_cast<uint32_t>(t * 128 + st * BKV);
          mma_scores<D>(dt, sQ(t, 0), sKh(st), ID_S, false);
          mma_scores<D>(dt, sQ(t, 0), sKl(st), ID_S, true);
          mma_scores<D>(dt, sQ(t, 1), sKh(st), ID_S, true);
          tc_commit(bar(B_SF + 2 * t + st));
        }
        any = true;
        tc_commit(bar(B_KE + st));
        return true;
      };
      if (ok && nkv > 0) ok = issue_s(0);
      for (int kv = 0; kv < nkv && ok; ++kv) {
        if (kv + 1 < nkv && !issue_s(kv + 1)) {
          ok = false;
          break;
        }
        const int st = kv & 1;
        if (!mbar_wait(bar(B_VF + st), static_cast<uint32_t>((kv >> 1) & 1), wc)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int t = 0; t < QT; ++t) {
          if (kv >= nkv_t[t]) continue;
          if (!mbar_wait(bar(B_PF + 2 * t + st), static_cast<uint32_t>((kv >> 1) & 1), wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk) {
            const uint64_t bd = sdesc_sw128(sV(st) + kk * 2048, 8192, 1024);
            tc_mma_bf16_ts(tmem + 256 + t * 128, tmem + t * 128 + st * BKV + kk * 8, bd, ID_PV,
                           (kv > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar(B_PE + 2 * t + st));
        }
        if (!ok) break;
        tc_commit(bar(B_VE + st));
      }
      if (any) {
        tc_commit(bar(B_DR));
        mbar_wait(bar(B_DR), 0, wdrain);
      }
    }
  } else {
    // -------------------------------------------------------------- softmax / output
    const int t = warp >> 2;            // tile
    const int quad = warp & 3;          // TMEM lane quadrant
    const int r = quad * 32 + lane;     // row within the tile
    const int q = q0 + t * BQ + r;
    const int nk = nkv_t[t];
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(t * 128);
    const uint32_t tO = tmem + lane_off + static_cast<uint32_t>(256 + t * 128);
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int kv = 0; kv < nk; ++kv) {
      const int st = kv & 1;
      const uint32_t tSb = tS + static_cast<uint32_t>(st * BKV);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B_SF + 2 * t + st), static_cast<uint32_t>((kv >> 1) & 1), wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t v0[32], v1[32];
      tmem_ld32(tSb, v0);
      tmem_ld32(tSb + 32, v1);
      tmem_ld_wait(v0);
      tmem_ld_wait(v1);
      // keep the P V completion barriers in step (block kv-2: long done)
      if (kv >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B_PE + 2 * t + st), static_cast<uint32_t>(((kv - 2) >> 1) & 1), wc));
        if (!ok) break;
      }
      const int kbase = kv * BKV;
      const bool masked = (a.causal && kbase + BKV - 1 > q0 + t * BQ) || (kbase + BKV > a.S);
      float sv[64];
      float bmax = -INFINITY;
#pragma unroll
      for (int e = 0; e < 64; ++e) {
        float s = __uint_as_float(e < 32 ? v0[e] : v1[e - 32]) * scale_log2;
        if (masked) {
          const int key = kbase + e;
          if (key >= a.S || (a.causal && key > q)) s = -INFINITY;
        }
        sv[e] = s;
        bmax = fmaxf(bmax, s);
      }
      if (kv == 0) {
        m = bmax;
      } else {
        const bool need = bmax > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          // O must be quiescent: wait for the previous block's P V
          ok = __all_sync(0xffffffffu, mbar_wait(bar(B_PE + 2 * t + ((kv - 1) & 1)),
                                                 static_cast<uint32_t>(((kv - 1) >> 1) & 1), wc));
          if (!ok) break;
          tc_fence_after();
          const float alpha = need ? exp2f(m - bmax) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + 32 * c, o);
          }
          l *= alpha;
          if (need) m = bmax;
        }
      }
      const float m_use = (m == -INFINITY) ? 0.0f : m;
      float ls = 0.0f;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const uint32_t pp = pack_bf16x2(exp2f(sv[2 * c] - m_use), exp2f(sv[2 * c + 1] - m_use));
        ls += bf16lo_to_f32(pp) + bf16hi_to_f32(pp);
        pk[c] = pp;
      }
      tmem_st32(tSb, pk);  // P over the scores just read (this thread's row only)
      tmem_st_wait();
      l += ls;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PF + 2 * t + st));
    }
    if (ok && nk > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B_PE + 2 * t + ((nk - 1) & 1)),
                                             static_cast<uint32_t>(((nk - 1) >> 1) & 1), wc));
    if (ok && nk > 0) {
      tc_fence_after();
      // every P.V of this tile is complete (and every score product before it): the
      // tile's Qh buffer is free for staging O
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      const uint32_t stage = sQ(t, 0) + static_cast<uint32_t>(quad * C::CH * 4096);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_ld_wait(o);
        const uint32_t cb = static_cast<uint32_t>(c >> 1), g0 = static_cast<uint32_t>((c & 1) * 4);
#pragma unroll
        for (int g = 0; g < 4; ++g)
          st_shared_v4(stage + cb * 4096 + lane * 128 + (((g0 + g) ^ static_cast<uint32_t>(lane & 7)) << 4),
                       pack_bf16x2(__uint_as_float(o[8 * g + 0]) * inv, __uint_as_float(o[8 * g + 1]) * inv),
                       pack_bf16x2(__uint_as_float(o[8 * g + 2]) * inv, __uint_as_float(o[8 * g + 3]) * inv),
                       pack_bf16x2(__uint_as_float(o[8 * g + 4]) * inv, __uint_as_float(o[8 * g + 5]) * inv),
                       pack_bf16x2(__uint_as_float(o[8 * g + 6]) * inv, __uint_as_float(o[8 * g + 7]) * inv));
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int qrow0 = q0 + t * BQ + quad * 32;
      if (lane == 0 && qrow0 < a.S) {
#pragma unroll
        for (int cb = 0; cb < C::CH; ++cb) tma_store_4d(&tmO, stage + cb * 4096, jj * D + 64 * cb, qrow0, b, shard);
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
  if (warp == WARP_MMA) {
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
  CUtensorMap tq, tkv, to;
  const uint64_t qd[4] = {static_cast<uint64_t>(a.qkv_width()), static_cast<uint64_t>(a.S),
                          static_cast<uint64_t>(a.B), static_cast<uint64_t>(a.N)};
  const uint32_t qbox[4] = {64, 128, 1, 1};
  const uint32_t kbox[4] = {64, BKV, 1, 1};
  const uint64_t od[4] = {static_cast<uint64_t>(a.hN) * D, static_cast<uint64_t>(a.S), static_cast<uint64_t>(a.B),
                          static_cast<uint64_t>(a.N)};
  const uint32_t obox[4] = {64, 32, 1, 1};
  if (!encode_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, qkv, qd, qbox, CU_TENSOR_MAP_SWIZZLE_128B)) return 2;
  if (!encode_tmap(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, qkv, qd, kbox, CU_TENSOR_MAP_SWIZZLE_128B)) return 2;
  if (!encode_tmap(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, o, od, obox, CU_TENSOR_MAP_SWIZZLE_128B)) return 2;
  const int nqb = (a.S + QT * BQ - 1) / (QT * BQ);
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  dim3 grid(nqb, a.H, a.B);
  const int slot = timing_begin(kKAttnCore, st);
  k_attn_fwd<D><<<grid, NTHREADS, C::SMEM, st>>>(tq, tkv, to, a, lse, scale_log2, err, timeout_ns);
  const bool ok = cudaGetLastError() == cudaSuccess;
  timing_end(slot, st);
  return ok ? 0 : 2;
}

}  // namespace

int launch_attn_fwd(const AttnDims& a, const void* qkv, void* o, float* lse, unsigned* err,
                    unsigned long long timeout_ns, cudaStream_t st) {
  if (a.B < 1 || a.S < 1 || a.H < 1 || a.N < 1 || a.hN * a.N != a.H) return 1;
  if (a.Hkv < 1 || a.hkvN * a.N != a.Hkv || a.H % a.Hkv || a.hN % a.hkvN) return 1;
  if (a.H > 65535 || a.B > 65535) return 1;
  if (a.d == 128) return launch_fwd_d<128>(a, qkv, o, lse, err, timeout_ns, st);
  if (a.d == 64) return launch_fwd_d<64>(a, qkv, o, lse, err, timeout_ns, st);
  return 1;
}

}  // namespace tpb
