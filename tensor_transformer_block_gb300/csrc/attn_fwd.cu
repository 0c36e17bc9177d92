// Fused per-head attention forward on tcgen05:
//   O_j = softmax(mask(Q_j K_j^T / sqrt(d))) V_j,  LSE = log sum exp(scaled scores)
// (damodev 3D并行 §1.2.2 per-head attention; the blockwise online-softmax
// recurrence is the one sunjinbo 并行方式 §CP uses to combine per-block results).
//
// One CTA per (256 queries = two 128-query tiles, query head, batch), heaviest
// causal blocks first; the key/value tiles are those of the head's group.  Keys
// are processed in blocks of 128 (the score products are M=128, N=128 MMAs: an
// M=128 tcgen05 instruction costs about as much at N=64 as at N=128), K and V each
// with two shared-memory stages so that the copies of block kv+1 overlap block kv.
//   warp 8: TMA producer: both Q tiles once; K and V per key block
//   warp 9: MMA issuer: per block, O_t += P_t V for both tiles (P read from TMEM,
//           V from shared memory; fp16 P and V), then S_t = Q_t K^T of the next
//           block for each tile once that tile's P V has read its P (fp16 Q and K,
//           one MMA per 16 of the head dim)
//   warps 0-3 / 4-7: the softmax warpgroup of tile 0 / tile 1, one query row per
//           thread: masked row max over the block, exp2, P (fp16) written back
//           over the first half of the same TMEM columns.  The running max is only
//           moved (and the row of O rescaled in TMEM) when a block's max exceeds
//           it by more than 8 (log2 units); otherwise the stale max stays,
//           P <= 2^8, and the final O / l is unchanged because the max cancels.
//           While one warpgroup works on its softmax the tensor core works on the
//           other tile.
// TMEM (512 columns): tile t's scores at 256 t (128 columns; P, 128 fp16 per row,
// in the first 64 of them), its O at 256 t + 128.  O is written out as fp16 or
// bf16 (AttnDims::o_f16).  A tile's P V has completed
// before the next block's scores overwrite its P, so O is never being accumulated
// while the softmax warps read or rescale it.
#include <cmath>

#include "attn.cuh"
#include "host_util.cuh"
#include "ptx.cuh"

namespace tpb {
namespace {

constexpr int BQ = 128;    // queries per tile
constexpr int QT = 2;      // tiles per CTA
constexpr int BKV = 128;   // keys per block
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
  B_SF = 9,   // [tile]: scores ready
  B_PF = 11,  // [tile]: P written to TMEM (4 arrivals)
  B_PE = 13,  // [tile]: P V complete
  B_DR = 15, NBARS = 16
};

// max(a, b, c) in one instruction (the three-input form of max.f32)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// acc + lo + hi of an fp16 pair, each half widened exactly inside the add
__device__ __forceinline__ float add_f16x2_f32(float acc, uint32_t pk) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.f32.f16 %0, lo, %0;\n\tadd.f32.f16 %0, hi, %0;\n\t}"
      : "+f"(acc)
      : "r"(pk));
  return acc;
}

template <int D>
struct FwdCfg {
  static constexpr int CH = D / 64;
  static constexpr int TILE = CH * 16384;  // 128 rows x D 16-bit values in 64-column swizzled chunks
  static constexpr int OFF_Q = 0;          // [tile]
  static constexpr int OFF_K = QT * TILE;  // [stage]
  static constexpr int OFF_V = OFF_K + 2 * TILE;  // [stage]
  static constexpr int OFF_BAR = OFF_V + 2 * TILE;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int USED = OFF_MISC + 16;
  // at least 120 KB so that a second CTA (which would wait for the TMEM this one
  // holds) never shares the SM
  static constexpr int SMEM = (USED + 1024 > 122880) ? USED + 1024 : 122880;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(D <= 128, "head dim");
};

// S = A B^T over K = D: A and B 128-row K-major tiles (16 KB chunks of 64 columns).
template <int D>
__device__ __forceinline__ void mma_scores(uint32_t d_tmem, uint32_t sa, uint32_t sb, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>((kk >> 2) * 16384 + (kk & 3) * 32);
    tc_mma_bf16(d_tmem, sdesc_sw128(sa + off, 16, 1024), sdesc_sw128(sb + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
  }
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_attn_fwd(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmO, const AttnDims a,
               float* __restrict__ lse, const float scale_log2, const WorkOrder ord, unsigned* err,
               const unsigned long long timeout_ns) {
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
  auto sQ = [&](int t) { return sb + C::OFF_Q + static_cast<uint32_t>(t * C::TILE); };
  auto sK = [&](int st) { return sb + C::OFF_K + static_cast<uint32_t>(st * C::TILE); };
  auto sV = [&](int st) { return sb + C::OFF_V + static_cast<uint32_t>(st * C::TILE); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (a.S + QT * BQ - 1) / (QT * BQ);
  int unit, rank;
  ord.decode(static_cast<int>(blockIdx.x), unit, rank);
  const int qb = nqb - 1 - rank;  // the last query blocks have the most causal work
  const int j = unit % a.H, b = unit / a.H;
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
  const int cQ = a.col_q(jj), cK = a.col_k(kvh), cV = a.col_v(kvh);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBARS; ++i) mbar_init(bar(i), (i >= B_PF && i < B_PF + QT) ? 4 : 1);
    *abort_flag = 0;
    *never_flag = 0;
    fence_mbar_init();
  }
  if (warp == WARP_PRODUCER && lane == 0) {
    prefetch_tmap(&tmQKV);
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
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();
  const WaitCtx wc{err, abort_flag, timeout_ns};
  const WaitCtx wdrain{err, never_flag, timeout_ns};

  if (warp == WARP_PRODUCER) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int kiss = 0, viss = 0;  // key blocks whose K / V copies were issued
      // every copy's x coordinate is a head's column offset + 64 c (16-byte aligned)
      const bool coords_ok = TP_DCHECK(cQ % 8 == 0 && cK % 8 == 0 && cV % 8 == 0 && cV + D <= a.qkv_width() &&
                                           b < a.B && shard < a.N,
                                       err);
      if (coords_ok) mbar_arrive_expect_tx(bar(B_QF), QT * C::TILE);
#pragma unroll
      for (int t = 0; t < QT; ++t)
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          if (coords_ok) tma_load_4d(sQ(t) + c * 16384, &tmQKV, bar(B_QF), cQ + 64 * c, q0 + t * BQ, b, shard);
      for (int kv = 0; kv < nkv && coords_ok; ++kv) {
        const int st = kv & 1;
        const uint32_t ph = static_cast<uint32_t>((kv >> 1) & 1);
        if (!mbar_wait(bar(B_KE + st), ph ^ 1u, wc)) break;
        mbar_arrive_expect_tx(bar(B_KF + st), C::TILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          tma_load_4d(sK(st) + c * 16384, &tmQKV, bar(B_KF + st), cK + 64 * c, kv * BKV, b, shard);
        kiss = kv + 1;
        if (!mbar_wait(bar(B_VE + st), ph ^ 1u, wc)) break;
        mbar_arrive_expect_tx(bar(B_VF + st), C::TILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          tma_load_4d(sV(st) + c * 16384, &tmQKV, bar(B_VF + st), cV + 64 * c, kv * BKV, b, shard);
        viss = kv + 1;
      }
      // every issued copy lands before the CTA may exit
      if (coords_ok) mbar_wait(bar(B_QF), 0, wdrain);
      for (int k = (kiss > 2 ? kiss - 2 : 0); k < kiss; ++k)
        mbar_wait(bar(B_KF + (k & 1)), static_cast<uint32_t>((k >> 1) & 1), wdrain);
      for (int k = (viss > 2 ? viss - 2 : 0); k < viss; ++k)
        mbar_wait(bar(B_VF + (k & 1)), static_cast<uint32_t>((k >> 1) & 1), wdrain);
    }
  } else if (warp == WARP_MMA) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t ID_S = idesc_f16(128, BKV, false, false);
      constexpr uint32_t ID_PV = idesc_f16(128, D, false, true);
      bool ok = mbar_wait(bar(B_QF), 0, wc), any = false;
      // scores of key block 0 for every tile
      if (ok && nkv > 0) {
        ok = mbar_wait(bar(B_KF), 0, wc);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < QT; ++t) {
            if (nkv_t[t] == 0) continue;
            mma_scores<D>(tmem + static_cast<uint32_t>(t * 256), sQ(t), sK(0), ID_S);
            tc_commit(bar(B_SF + t));
          }
          any = true;
          tc_commit(bar(B_KE));
        }
      }
      // per block kv and tile t: O_t += P_t V (once the softmax wrote P_t), then, as
      // soon as that P V has read P_t, the tile's scores of block kv+1 into the same
      // columns; the other tile's softmax runs meanwhile
      for (int kv = 0; kv < nkv && ok; ++kv) {
        const int st = kv & 1, st1 = (kv + 1) & 1;
        const bool next = kv + 1 < nkv;
        if (!mbar_wait(bar(B_VF + st), static_cast<uint32_t>((kv >> 1) & 1), wc)) {
          ok = false;
          break;
        }
        if (next && !mbar_wait(bar(B_KF + st1), static_cast<uint32_t>(((kv + 1) >> 1) & 1), wc)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int t = 0; t < QT; ++t) {
          if (kv >= nkv_t[t]) continue;
          if (!mbar_wait(bar(B_PF + t), static_cast<uint32_t>(kv & 1), wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tS = tmem + static_cast<uint32_t>(t * 256);
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            tc_mma_bf16_ts(tS + 128, tS + kk * 8, sdesc_sw128(sV(st) + kk * 2048, 16384, 1024), ID_PV,
                           (kv > 0 || kk > 0) ? 1u : 0u);
          tc_commit(bar(B_PE + t));
          if (kv + 1 < nkv_t[t]) {
            // the P V just issued has read the P these columns hold
            if (!mbar_wait(bar(B_PE + t), static_cast<uint32_t>(kv & 1), wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_scores<D>(tS, sQ(t), sK(st1), ID_S);
            tc_commit(bar(B_SF + t));
          }
        }
        if (!ok) break;
        tc_commit(bar(B_VE + st));
        if (next) tc_commit(bar(B_KE + st1));
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
    const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(t * 256);
    const uint32_t tO = tS + 128;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int kv = 0; kv < nk; ++kv) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B_SF + t), static_cast<uint32_t>(kv & 1), wc));
      if (!ok) break;
      tc_fence_after();
      const int kbase = kv * BKV;
      const bool masked = (a.causal && kbase + BKV - 1 > q0 + t * BQ) || (kbase + BKV > a.S);
      const int klim = a.causal ? min(q, a.S - 1) : a.S - 1;  // last visible key
      // the block's 128 raw scores of this row, in registers
      uint32_t v[BKV / 32][32];
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) tmem_ld32(tS + 32 * c, v[c]);
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) tmem_ld_wait(v[c]);
      if (masked) {
#pragma unroll
        for (int c = 0; c < BKV / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (kbase + 32 * c + e > klim) v[c][e] = __float_as_uint(-INFINITY);
      }
      // row max (raw scores; the scale is positive), two scores per instruction
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          mx[(e >> 1) & 3] = fmax3(mx[(e >> 1) & 3], __uint_as_float(v[c][e]), __uint_as_float(v[c][e + 1]));
      const float bmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
      // the running max moves only when the block's exceeds it by the threshold; O
      // is then rescaled after P is written, when the score registers are dead
      float alpha = 1.0f;
      bool rescale = false;
      if (kv == 0) {
        m = bmax;
      } else {
        const bool need = bmax > m + kRescaleThreshold;
        rescale = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = exp2f(m - bmax);
          m = bmax;
        }
      }
      const float m_use = (m == -INFINITY) ? 0.0f : m;
      // P = exp2(s * scale - m) as fp16 (masked scores are -inf: exp2 gives 0; P <= 2^8,
      // and a P below fp16's normal range keeps an absolute error under 2^-25),
      // written over the first 64 of the columns just read
      // the exponent arguments s * scale - m two at a time (paired fp32 FMA)
      float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const uint64_t sc2 = f32x2(scale_log2, scale_log2), nm2 = f32x2(-m_use, -m_use);
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float x0, x1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(v[c][2 * e]), __uint_as_float(v[c][2 * e + 1])), sc2, nm2), x0,
                      x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          pk[e] = pack_f16x2(p0, p1);
          ls[e & 3] = add_f16x2_f32(ls[e & 3], pk[e]);
        }
        tmem_st16(tS + 16 * c, pk);
      }
      if (rescale) {
        // O is quiescent: this tile's previous P V completed before these scores, and
        // the next one waits for the P arrival below
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + 32 * c, o);
        }
      }
      tmem_st_wait();
      l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PF + t));
    }
    // the last P V (issued after this tile's previous ones had completed)
    if (ok && nk > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar(B_PE + t), static_cast<uint32_t>((nk - 1) & 1), wc));
    if (ok && nk > 0) {
      tc_fence_after();
      // every MMA of this tile is complete: its Q buffer is free for staging O
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      const uint32_t stage = sQ(t) + static_cast<uint32_t>(quad * C::CH * 4096);
      const bool of16 = a.o_f16 != 0;
      auto pk2 = [of16](float x, float y) { return of16 ? pack_f16x2(x, y) : pack_bf16x2(x, y); };
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_ld_wait(o);
        const uint32_t cb = static_cast<uint32_t>(c >> 1), g0 = static_cast<uint32_t>((c & 1) * 4);
#pragma unroll
        for (int g = 0; g < 4; ++g)
          st_shared_v4(stage + cb * 4096 + lane * 128 + (((g0 + g) ^ static_cast<uint32_t>(lane & 7)) << 4),
                       pk2(__uint_as_float(o[8 * g + 0]) * inv, __uint_as_float(o[8 * g + 1]) * inv),
                       pk2(__uint_as_float(o[8 * g + 2]) * inv, __uint_as_float(o[8 * g + 3]) * inv),
                       pk2(__uint_as_float(o[8 * g + 4]) * inv, __uint_as_float(o[8 * g + 5]) * inv),
                       pk2(__uint_as_float(o[8 * g + 6]) * inv, __uint_as_float(o[8 * g + 7]) * inv));
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int qrow0 = q0 + t * BQ + quad * 32;
      if (lane == 0 && qrow0 < a.S) {
#pragma unroll
        for (int cb = 0; cb < C::CH; ++cb) tma_store_4d(&tmO, stage + cb * 4096, jj * D + 64 * cb, qrow0, b, shard);
        bulk_commit();
      }
      const size_t li = (static_cast<size_t>(b) * a.H + j) * a.S + q;
      if (q < a.S && TP_DCHECK(li < static_cast<size_t>(a.B) * a.H * a.S, err))
        lse[li] = (m + log2f(l)) * 0.6931471805599453f;
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
  static std::atomic<bool> configured[kMaxDevices];
  if (!set_smem_limit_once(reinterpret_cast<const void*>(k_attn_fwd<D>), C::SMEM, configured)) return 2;
  CUtensorMap tqkv, to;
  const uint64_t qd[4] = {static_cast<uint64_t>(a.qkv_width()), static_cast<uint64_t>(a.S),
                          static_cast<uint64_t>(a.B), static_cast<uint64_t>(a.N)};
  const uint32_t box[4] = {64, 128, 1, 1};
  const uint64_t od[4] = {static_cast<uint64_t>(a.hN) * D, static_cast<uint64_t>(a.S), static_cast<uint64_t>(a.B),
                          static_cast<uint64_t>(a.N)};
  const uint32_t obox[4] = {64, 32, 1, 1};
  // 16-bit elements (fp16 Q, K and V; O fp16 or bf16): the copies do not interpret them
  if (!encode_tmap(&tqkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, qkv, qd, box, CU_TENSOR_MAP_SWIZZLE_128B)) return 2;
  if (!encode_tmap(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, o, od, obox, CU_TENSOR_MAP_SWIZZLE_128B)) return 2;
  const int nqb = (a.S + QT * BQ - 1) / (QT * BQ);
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  const WorkOrder ord = make_work_order(a.B * a.H, nqb, device_sm_count());
  const int slot = timing_begin(kKAttnCore, st);
  const bool ok = launch_k(k_attn_fwd<D>, dim3(ord.ctas()), dim3(NTHREADS), C::SMEM, st, 1, tqkv, to, a, lse,
                           scale_log2, ord, err, timeout_ns) == cudaSuccess;
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
