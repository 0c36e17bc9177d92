// tcgen05 GEMM with TMA multi-stage pipeline and fused epilogues (see gemm_tc.cuh).
//
// CTA = 10 warps, one CTA per SM, persistent over output tiles:
//   warp 8  TMA producer: fills a ring of (A 128x64, B 64-deep) bf16 stages,
//           128-byte swizzled, K-major or MN-major as the operand is stored; an
//           MN-major operand whose rows are whole 64-element chunks comes in one
//           copy per stage through a map with the chunk as an outer dimension;
//   warp 9  MMA issuer: 4 x tcgen05.mma (K=16) per stage into one of two TMEM
//           accumulators (2 x 256 fp32 columns), so the epilogue of tile t
//           overlaps the main loop of tile t+1;
//   warps 0-7 epilogue: warp w reads TMEM lanes 32*(w%4).. (its row quadrant) and
//           columns 128*(w/4).. (its half), so every SM sub-partition runs two
//           epilogue warps to hide the latency of the fused math; fused GeLU /
//           GeLU' / SwiGLU / residual in fp32, bf16 pack into a swizzled staging
//           box, TMA store.
// The main loop is fed by as many stages as shared memory holds next to the
// epilogue's staging: a k-block's loads take microseconds to arrive from L2, and
// with one stage fewer the MMA issuer measurably waits for data.  The epilogue
// stages 32 KB per CTA: the plain-store epilogues one box of 32 rows x 64 columns
// per warp (128-byte swizzle), the fused ones two boxes of 32 rows x 32 columns
// (64-byte swizzle; an input and an output, or two outputs).
// Two tilings:
//   single: one CTA per 128 x 256 tile (cta_group::1, M=128 N=256); 4 stages of 48 KB.
//   pair:   a cluster of two CTAs per 256 x 256 tile (cta_group::2, M=256 N=256):
//           each CTA stages its 128 rows of A and half (128 columns) of B, so each
//           SM moves 32 KB per k-block instead of 48; 6 stages.  The even CTA issues
//           the MMAs; both CTAs' TMA loads count on its full barrier; its commits
//           arrive on both CTAs' empty / accumulator-ready barriers; both CTAs'
//           epilogue warps release an accumulator on the even CTA's barrier.
// Every wait is bounded; on a timeout the CTA latches an error, drains its own
// copies and MMAs, frees TMEM and returns.
#include <cstdlib>

#include "gemm_tc.cuh"
#include "host_util.cuh"
#include "ptx.cuh"

namespace tpb {
namespace {

constexpr int BK = 64;
constexpr int BN = 256;  // MMA N (tile columns)
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 320;
constexpr int WARP_PRODUCER = 8;
constexpr int WARP_MMA = 9;
constexpr int TMEM_COLS = 512;
constexpr int GROUP_M = 16;

template <bool PAIR, int EPI>
struct Cfg {
  // staging boxes per warp
  static constexpr int EBUFS = (EPI == kEpiStore || EPI == kEpiSplit || EPI == kEpiPartial) ? 1 : 2;
  // epilogue chunk: 32 rows x CW columns of bf16 (one box): 64 columns with 128-byte
  // swizzle for the one-box epilogues, 32 columns with 64-byte swizzle for the fused
  // ones, so that either stages 32 KB per CTA
  static constexpr int CW = EBUFS == 1 ? 64 : 32;
  static constexpr int EBOX = 32 * CW * 2;
  static constexpr int BM = 128;                      // accumulator rows per CTA
  static constexpr int TILE_M = PAIR ? 256 : 128;     // rows per output tile
  static constexpr int BN_CTA = PAIR ? 128 : 256;     // B columns staged per CTA
  static constexpr int STAGES = PAIR ? 6 : 4;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN_CTA * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_FULL = 0;
  static constexpr int BAR_EMPTY = STAGES;
  static constexpr int BAR_TFULL = 2 * STAGES;
  static constexpr int BAR_TEMPTY = 2 * STAGES + 2;
  static constexpr int BAR_Y = 2 * STAGES + 4;
  static constexpr int BAR_DRAIN = BAR_Y + 2 * EPI_WARPS;
  static constexpr int NUM_BARS = BAR_DRAIN + 1;
  static constexpr int SMEM_EPI_OFF = STAGES * STAGE_BYTES;
  static constexpr int SMEM_BAR_OFF = SMEM_EPI_OFF + EPI_WARPS * EBUFS * EBOX;
  static constexpr int SMEM_MISC_OFF = SMEM_BAR_OFF + NUM_BARS * 8;
  static constexpr int SMEM_USED = SMEM_MISC_OFF + 16;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

// Tile order: GROUP_M consecutive M tiles sweep the N tiles together, so the
// operand panels they share are reused from L2.  With several output groups that
// share the A operand the groups are folded into the N sweep (g_mode 1), so an A
// panel is read once for all groups instead of once per group; g_mode 2 folds
// them into M instead.
__device__ __forceinline__ void decode_tile(int t, const GemmShape& p, int& g, int& mb, int& nb) {
  const int tm = p.g_mode == 2 ? p.G * p.tiles_m : p.tiles_m;
  const int tn = p.g_mode == 1 ? p.G * p.tiles_n : p.tiles_n;
  const int per_g = tm * tn;
  const int g0 = p.g_mode == 0 ? t / per_g : 0;
  const int r = t - g0 * per_g;
  const int span = GROUP_M * tn;
  const int grp = r / span;
  const int first_m = grp * GROUP_M;
  const int gm = min(tm - first_m, GROUP_M);
  const int rr = r - grp * span;
  int m = first_m + rr % gm, n = rr / gm;
  g = g0;
  if (p.g_mode == 1) {
    g = n / p.tiles_n;
    n -= g * p.tiles_n;
  } else if (p.g_mode == 2) {
    g = m / p.tiles_m;
    m -= g * p.tiles_m;
  }
  mb = m;
  nb = n;
}

// GeLU (tanh form) through the logistic identity 0.5 (1 + tanh u) = 1 / (1 + e^(-2u))
// with u = sqrt(2/pi) (x + 0.044715 x^3): with s = 1 / (1 + e^(-2u)), GeLU(x) = x s
// and, since 1 - tanh^2 u = 4 s (1 - s), GeLU'(x) = s (1 + x (1 - s) 2u').  One exp2
// and one reciprocal per element, no cancellation in 1 + tanh u for negative x.  The
// constants are folded (x2 = x^2):
//   -2u log2(e) = x (k1 + k3 x2),  k1 = -2 log2(e) sqrt(2/pi),  k3 = 0.044715 k1
//   2u'         = d0 + d2 x2,      d0 = 2 sqrt(2/pi),           d2 = 3 * 0.044715 d0
// The exponent is clamped so that e^(-2u) stays finite (s then underflows towards 0
// smoothly).  exp2 and the reciprocal are the special-function unit's approximations
// (about 1 ulp of fp32): the results are rounded to bf16, and the correctly rounded
// reciprocal cost ~2% of the fused GEMMs' time.
// Two values are computed at once: the fp32 arithmetic in paired instructions (each
// half rounded as the scalar instruction rounds it), the clamp, exponential and
// reciprocal per element.  That halves the issue cost of the fused epilogues' math,
// which shares its sub-partitions with the MMA and TMA warps.  s and oms = 1 - s
// (= e^(-2u) s, no cancellation) of the pair x (x2 = x^2):
__device__ __forceinline__ void gelu_sigmoid2(uint64_t x, uint64_t x2, uint64_t& s, uint64_t& oms) {
  const uint64_t k3 = f32x2(-0.1029432395800235f, -0.1029432395800235f);
  const uint64_t k1 = f32x2(-2.302208198144325f, -2.302208198144325f);
  float a0, a1;
  f32x2_split(mul_f32x2(x, fma_f32x2(k3, x2, k1)), a0, a1);
  const float e0 = ex2_approx(fminf(a0, 126.0f)), e1 = ex2_approx(fminf(a1, 126.0f));
  const uint64_t e = f32x2(e0, e1);
  float d0, d1;
  f32x2_split(add_f32x2(f32x2(1.0f, 1.0f), e), d0, d1);
  s = f32x2(rcp_approx(d0), rcp_approx(d1));
  oms = mul_f32x2(e, s);
}

// GeLU of two values (the pair (lo, hi) of ``x``)
__device__ __forceinline__ uint64_t gelu2(uint64_t x) {
  uint64_t s, oms;
  gelu_sigmoid2(x, mul_f32x2(x, x), s, oms);
  return mul_f32x2(x, s);
}

// da * GeLU'(y) for two values
__device__ __forceinline__ uint64_t dgelu2(uint64_t da, uint64_t y) {
  const uint64_t y2 = mul_f32x2(y, y);
  uint64_t s, oms;
  gelu_sigmoid2(y, y2, s, oms);
  const uint64_t d2 = f32x2(0.21406444881780076f, 0.21406444881780076f);
  const uint64_t d0 = f32x2(1.5957691216057308f, 1.5957691216057308f);
  const uint64_t g =
      mul_f32x2(s, fma_f32x2(mul_f32x2(y, oms), fma_f32x2(d2, y2, d0), f32x2(1.0f, 1.0f)));
  return mul_f32x2(da, g);
}

// Logistic sigmoid s = 1 / (1 + e^(-x)) and 1 - s = e^(-x) s (no cancellation) of
// a pair; silu(x) = x s, silu'(x) = s (1 + x (1 - s)).  Clamped and paired as above.
__device__ __forceinline__ void sigmoid2(uint64_t x, uint64_t& s, uint64_t& oms) {
  float a0, a1;
  f32x2_split(mul_f32x2(f32x2(-1.4426950408889634f, -1.4426950408889634f), x), a0, a1);  // -x log2(e)
  const float e0 = ex2_approx(fminf(a0, 126.0f)), e1 = ex2_approx(fminf(a1, 126.0f));
  const uint64_t e = f32x2(e0, e1);
  float d0, d1;
  f32x2_split(add_f32x2(f32x2(1.0f, 1.0f), e), d0, d1);
  s = f32x2(rcp_approx(d0), rcp_approx(d1));
  oms = mul_f32x2(e, s);
}

// Tile copies of an operand whose second coordinate c1 may be a token of a
// sequence-sharded tensor (spS > 0): token b*spS + s lives at [s / spL][b][s % spL].
// Tiles never straddle a shard or a batch (spL is a multiple of every box height).
__device__ __forceinline__ void tok_coords(int t, int spS, int spL, int& sl, int& bb, int& cc) {
  bb = t / spS;
  const int s = t - bb * spS;
  cc = s / spL;
  sl = s - cc * spL;
}
// Position of a token in the sequence-sharded layout (tracked incrementally by the
// producer, so the K loop does no integer division).
struct TokPos {
  int sl, b, c;
};
template <bool PAIR>
__device__ __forceinline__ void op_load_at(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1, int z,
                                           bool sp, const TokPos& tp) {
  if (sp) {
    if (PAIR)
      tma_load_4d_pair(dst, m, bar, c0, tp.sl, tp.b, tp.c);
    else
      tma_load_4d(dst, m, bar, c0, tp.sl, tp.b, tp.c);
  } else {
    if (PAIR)
      tma_load_3d_pair(dst, m, bar, c0, c1, z);
    else
      tma_load_3d(dst, m, bar, c0, c1, z);
  }
}
template <bool PAIR>
__device__ __forceinline__ void op_load(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1, int z, int spS,
                                        int spL) {
  TokPos tp{0, 0, 0};
  if (spS > 0) tok_coords(c1, spS, spL, tp.sl, tp.b, tp.c);
  op_load_at<PAIR>(dst, m, bar, c0, c1, z, spS > 0, tp);
}
// One copy of an MN-major operand's stage through a chunked map: {64, K, chunks, z}
// (or {64, L, chunks, B, S/L} for sequence-sharded K); chunk0 = first 64-wide chunk.
template <bool PAIR>
__device__ __forceinline__ void mn_load(uint32_t dst, const CUtensorMap* m, uint32_t bar, int chunk0, int k, int z,
                                        bool sp, const TokPos& tp) {
  if (sp) {
    if (PAIR)
      tma_load_5d_pair(dst, m, bar, 0, tp.sl, chunk0, tp.b, tp.c);
    else
      tma_load_5d(dst, m, bar, 0, tp.sl, chunk0, tp.b, tp.c);
  } else {
    if (PAIR)
      tma_load_4d_pair(dst, m, bar, 0, k, chunk0, z);
    else
      tma_load_4d(dst, m, bar, 0, k, chunk0, z);
  }
}
__device__ __forceinline__ void out_store(const CUtensorMap* m, uint32_t src, int c0, int row, int z, int spS, int spL) {
  if (spS > 0) {
    int sl, bb, cc;
    tok_coords(row, spS, spL, sl, bb, cc);
    tma_store_4d(m, src, c0, sl, bb, cc);
  } else {
    tma_store_3d(m, src, c0, row, z);
  }
}

template <bool PAIR, bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmY, const GemmShape p) {
  using C = Cfg<PAIR, EPI>;
  // output columns per tile: the gated forward spends half the MMA's N on the up part
  constexpr int TILE_N = EPI == kEpiSwiGLU ? BN / 2 : BN;
  constexpr int WARP_COLS = TILE_N / 2;  // output columns per epilogue warp
  constexpr bool LOADS_Y = EPI == kEpiDGelu || EPI == kEpiDSwiGLU || EPI == kEpiResidual;
  constexpr int BM = C::BM, STAGES = C::STAGES, A_BYTES = C::A_BYTES, STAGE_BYTES = C::STAGE_BYTES;
  constexpr int BAR_FULL = C::BAR_FULL, BAR_EMPTY = C::BAR_EMPTY, BAR_TFULL = C::BAR_TFULL;
  constexpr int BAR_TEMPTY = C::BAR_TEMPTY, BAR_Y = C::BAR_Y, BAR_DRAIN = C::BAR_DRAIN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const uint32_t bar0 = sbase + C::SMEM_BAR_OFF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SMEM_MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::SMEM_MISC_OFF + 4);
  volatile int* never_flag = reinterpret_cast<volatile int*>(smem + C::SMEM_MISC_OFF + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int CL = PAIR ? 2 : 1;                     // CTAs per cluster
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // position in the CTA pair
  const uint32_t lead = 0u;                            // the pair's even CTA
  const bool leader = rank == 0;
  const int unit = static_cast<int>(blockIdx.x) / CL;
  const int nunits = static_cast<int>(gridDim.x) / CL;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bar0 + 8u * (BAR_FULL + i), 1);
      mbar_init(bar0 + 8u * (BAR_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar0 + 8u * (BAR_TFULL + i), 1);
      mbar_init(bar0 + 8u * (BAR_TEMPTY + i), PAIR ? 2 * EPI_WARPS : EPI_WARPS);
    }
    for (int i = 0; i < 2 * EPI_WARPS; ++i) mbar_init(bar0 + 8u * (BAR_Y + i), 1);
    mbar_init(bar0 + 8u * BAR_DRAIN, 1);
    *abort_flag = 0;
    *never_flag = 0;
    fence_mbar_init();
  }
  if (warp == WARP_PRODUCER && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
    if (EPI != kEpiStore && EPI != kEpiSplit) prefetch_tmap(&tmY);
  }
  if (warp == WARP_MMA) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers are initialised before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();

  const WaitCtx wc{p.err, abort_flag, p.timeout_ns};
  const WaitCtx wdrain{p.err, never_flag, p.timeout_ns};
  const int tiles = p.G * p.tiles_m * p.tiles_n;
  const int total = tiles * p.ksplit;  // work units: (split, tile), split-major
  const int nk = p.S * p.kb_per_seg;
  // K blocks [kbeg, kend) of the unit's split
  auto krange = [&](int t, int& kbeg, int& kend) {
    const int split = t / tiles;
    kbeg = split * p.kps;
    kend = min(nk, kbeg + p.kps);
  };

  if (warp == WARP_PRODUCER) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      // sequence-sharded token axes: the rows of a K-major A (one position per
      // tile) and the K axis of MN-major A / B (advanced by 64 per k-block)
      const bool a_rows_sp = !A_MN && p.a_spS > 0;
      const bool a_k_sp = A_MN && p.a_spS > 0, b_k_sp = B_MN && p.b_spS > 0;
      const int k_spL = a_k_sp ? p.a_spL : p.b_spL;
      const int k_nc = (a_k_sp || b_k_sp) ? (a_k_sp ? p.a_spS : p.b_spS) / k_spL : 1;
      for (int t = unit; t < total && ok; t += nunits) {
        int g, mb, nb, kbeg, kend;
        decode_tile(t % tiles, p, g, mb, nb);
        krange(t, kbeg, kend);
        const int arow = mb * C::TILE_M + static_cast<int>(rank) * BM;
        const int bcol = EPI == kEpiSwiGLU ? nb * TILE_N : nb * BN + static_cast<int>(rank) * C::BN_CTA;
        TokPos apos{0, 0, 0};
        if (a_rows_sp) tok_coords(arow, p.a_spS, p.a_spL, apos.sl, apos.b, apos.c);
        // the segments the split's K blocks fall in (a split starts inside a segment only
        // without sequence-sharded K, where kpos is unused)
        for (int s = kbeg / p.kb_per_seg; s < p.S && s * p.kb_per_seg < kend && ok; ++s) {
          const int az = g * p.a_zg + s * p.a_zs;
          const int bz = g * p.b_zg + s * p.b_zs;
          TokPos kpos{0, 0, 0};
          const int kb_lo = max(0, kbeg - s * p.kb_per_seg), kb_hi = min(p.kb_per_seg, kend - s * p.kb_per_seg);
          for (int kb = kb_lo; kb < kb_hi; ++kb) {
            if (!mbar_wait(bar0 + 8u * (BAR_EMPTY + stage), phase ^ 1u, wc)) {
              ok = false;
              break;
            }
            const uint32_t fb_local = bar0 + 8u * (BAR_FULL + stage);
            const uint32_t sa = sbase + stage * STAGE_BYTES;
            const uint32_t sb = sa + A_BYTES;
            const int kc = kb * BK;
            // every x coordinate below is kc, arow + 64 j or bcol + 64 j (or 0): a copy
            // must start on a 16-byte boundary and inside the operand's extent
            if (!TP_DCHECK(kc % 8 == 0 && arow % 8 == 0 && bcol % 8 == 0 && arow >= 0 && bcol >= 0 &&
                               arow < p.tiles_m * C::TILE_M && az >= 0 && bz >= 0,
                           p.err)) {
              ok = false;
              break;
            }
            if (PAIR) {
              const uint32_t fb = mapa_shared(fb_local, lead);  // the even CTA's full barrier counts both
              if (leader) mbar_arrive_expect_tx(fb_local, 2 * STAGE_BYTES);
              if (A_MN && p.a_chunked) {
                mn_load<true>(sa, &tmA, fb, arow / 64, kc, az, a_k_sp, kpos);
              } else if (A_MN) {
#pragma unroll
                for (int j = 0; j < BM / 64; ++j)
                  op_load_at<true>(sa + j * (BK * 128), &tmA, fb, arow + j * 64, kc, az, a_k_sp, kpos);
              } else {
                op_load_at<true>(sa, &tmA, fb, kc, arow, az, a_rows_sp, apos);
              }
              // B: each CTA stages half of the tile's columns
              if (EPI == kEpiSwiGLU) {
                // the even CTA stages the tile's gate columns, the odd CTA its up columns
                if (p.b_chunked) {
                  tma_load_5d_pair(sb, &tmB, fb, 0, kc, bcol / 64, static_cast<int>(rank), bz);
                } else {
#pragma unroll
                  for (int j = 0; j < C::BN_CTA / 64; ++j)
                    tma_load_4d_pair(sb + j * (BK * 128), &tmB, fb, bcol + j * 64, static_cast<int>(rank), kc, bz);
                }
              } else if (B_MN && p.b_chunked) {
                if (b_k_sp)
                  tma_load_5d_pair(sb, &tmB, fb, 0, kpos.sl, bcol / 64, kpos.b, kpos.c);
                else
                  tma_load_4d_pair(sb, &tmB, fb, 0, kc, bcol / 64, bz);
              } else if (B_MN) {
#pragma unroll
                for (int j = 0; j < C::BN_CTA / 64; ++j) {
                  if (b_k_sp)
                    tma_load_4d_pair(sb + j * (BK * 128), &tmB, fb, bcol + j * 64, kpos.sl, kpos.b, kpos.c);
                  else
                    tma_load_3d_pair(sb + j * (BK * 128), &tmB, fb, bcol + j * 64, kc, bz);
                }
              } else {
                tma_load_3d_pair(sb, &tmB, fb, kc, bcol, bz);
              }
            } else {
              mbar_arrive_expect_tx(fb_local, STAGE_BYTES);
              if (A_MN && p.a_chunked) {
                mn_load<false>(sa, &tmA, fb_local, arow / 64, kc, az, a_k_sp, kpos);
              } else if (A_MN) {
#pragma unroll
                for (int j = 0; j < BM / 64; ++j)
                  op_load_at<false>(sa + j * (BK * 128), &tmA, fb_local, arow + j * 64, kc, az, a_k_sp, kpos);
              } else {
                op_load_at<false>(sa, &tmA, fb_local, kc, arow, az, a_rows_sp, apos);
              }
              if (EPI == kEpiSwiGLU) {
                // atoms 0-1: gate columns, atoms 2-3: the same columns of the up part
                if (p.b_chunked) {
                  tma_load_5d(sb, &tmB, fb_local, 0, kc, bcol / 64, 0, bz);
                  tma_load_5d(sb + 2 * (BK * 128), &tmB, fb_local, 0, kc, bcol / 64, 1, bz);
                } else {
#pragma unroll
                  for (int j = 0; j < C::BN_CTA / 64; ++j)
                    tma_load_4d(sb + j * (BK * 128), &tmB, fb_local, bcol + (j & 1) * 64, j >> 1, kc, bz);
                }
              } else if (B_MN && p.b_chunked) {
                mn_load<false>(sb, &tmB, fb_local, bcol / 64, kc, bz, b_k_sp, kpos);
              } else if (B_MN) {
#pragma unroll
                for (int j = 0; j < C::BN_CTA / 64; ++j)
                  op_load_at<false>(sb + j * (BK * 128), &tmB, fb_local, bcol + j * 64, kc, bz, b_k_sp, kpos);
              } else {
                tma_load_3d(sb, &tmB, fb_local, kc, bcol, bz);
              }
            }
            if (a_k_sp || b_k_sp) {  // next 64 tokens of the K axis
              kpos.sl += BK;
              if (kpos.sl >= k_spL) {
                kpos.sl = 0;
                if (++kpos.c >= k_nc) {
                  kpos.c = 0;
                  ++kpos.b;
                }
              }
            }
            issued |= 1u << stage;
            last_par = (last_par & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // every issued copy must land before the CTA may exit: the even CTA watches
      // its full barriers; the odd CTA the empty barriers the even CTA's MMAs
      // release after consuming those copies
      for (int s2 = 0; s2 < STAGES; ++s2)
        if (issued & (1u << s2)) {
          const uint32_t par = (last_par >> s2) & 1u;
          if (!PAIR || leader)
            mbar_wait(bar0 + 8u * (BAR_FULL + s2), par, wdrain);
          else
            mbar_wait(bar0 + 8u * (BAR_EMPTY + s2), par, wdrain);
        }
    }
  } else if (warp == WARP_MMA) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------------- MMA issuer
      const uint32_t IDESC =
          p.ab_f16 ? idesc_f16(C::TILE_M, BN, A_MN, B_MN) : idesc_bf16(C::TILE_M, BN, A_MN, B_MN);
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true, any = false;
      for (int t = unit; t < total && ok; t += nunits, ++it) {
        const int buf = it & 1;
        const uint32_t tph = (it >> 1) & 1;
        int kbeg, kend;
        krange(t, kbeg, kend);
        if (!mbar_wait(bar0 + 8u * (BAR_TEMPTY + buf), tph ^ 1u, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int k = kbeg; k < kend; ++k) {
          if (!mbar_wait(bar0 + 8u * (BAR_FULL + stage), phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(sa + kk * 2048, BK * 128, 1024) : sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(sb + kk * 2048, BK * 128, 1024) : sdesc_sw128(sb + kk * 32, 16, 1024);
            const uint32_t acc = ((k - kbeg) | kk) != 0 ? 1u : 0u;
            if (PAIR)
              tc_mma_bf16_pair(dt, ad, bd, IDESC, acc);
            else
              tc_mma_bf16(dt, ad, bd, IDESC, acc);
          }
          any = true;
          if (PAIR)
            tc_commit_pair(bar0 + 8u * (BAR_EMPTY + stage), 3);
          else
            tc_commit(bar0 + 8u * (BAR_EMPTY + stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR)
          tc_commit_pair(bar0 + 8u * (BAR_TFULL + buf), 3);
        else
          tc_commit(bar0 + 8u * (BAR_TFULL + buf));
      }
      if (any) {
        if (PAIR)
          tc_commit_pair(bar0 + 8u * BAR_DRAIN, 1);
        else
          tc_commit(bar0 + 8u * BAR_DRAIN);
        mbar_wait(bar0 + 8u * BAR_DRAIN, 0, wdrain);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int ew = warp;                 // staging buffers and Y barriers
    const int quad = warp & 3;           // TMEM lanes 32*quad .. 32*quad+31
    const int half = warp >> 2;          // tile columns 128*half .. 128*half+127
    constexpr int CW = C::CW, EBOX = C::EBOX;
    const uint32_t ebuf[2] = {sbase + C::SMEM_EPI_OFF + ew * C::EBUFS * EBOX,
                              sbase + C::SMEM_EPI_OFF + ew * C::EBUFS * EBOX + (C::EBUFS - 1) * EBOX};
    const uint32_t ybar[2] = {bar0 + 8u * (BAR_Y + 2 * ew), bar0 + 8u * (BAR_Y + 2 * ew + 1)};
    // byte offset of this lane's 16-byte unit c in a swizzled staging box (row = lane):
    // 128-byte rows XOR row % 8, or 64-byte rows XOR (row / 2) % 4
    auto soff = [lane](uint32_t c) -> uint32_t {
      const uint32_t r = static_cast<uint32_t>(lane);
      return CW == 64 ? r * 128 + ((c ^ (r & 7)) << 4) : r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
    };
    uint32_t yph = 0;      // bit b: parity of the next completion of ybar[b]
    uint32_t ypend = 0;    // bit b: a Y load into ebuf[b] is in flight
    uint32_t ecount = 0;   // chunks staged so far (buffer alternation for kEpiStore / kEpiDGelu)
    int it = 0;
    bool ok = true;
    for (int t = unit; t < total && ok; t += nunits, ++it) {
      int g, mb, nb;
      decode_tile(t % tiles, p, g, mb, nb);
      const int split = t / tiles;
      const int buf = it & 1;
      const uint32_t tph = (it >> 1) & 1;
      const int row0 = mb * C::TILE_M + static_cast<int>(rank) * BM + quad * 32;
      const int col0 = nb * TILE_N + half * WARP_COLS;
      int nch = col0 < p.N ? (p.N - col0 + CW - 1) / CW : 0;
      if (nch > WARP_COLS / CW) nch = WARP_COLS / CW;
      // the staged boxes start at x = col0 + CW j (16-byte aligned) in group g < G;
      // the condition is the same for every lane of the warp
      const bool rows_valid =
          row0 < p.M && nch > 0 && TP_DCHECK(col0 % 8 == 0 && row0 >= 0 && g >= 0 && g < p.G, p.err);
      if ((EPI == kEpiDGelu || EPI == kEpiResidual) && rows_valid) {
        const uint32_t b = ecount & 1u;
        if (lane == 0) {
          bulk_wait_read0();
          mbar_arrive_expect_tx(ybar[b], EBOX);
          op_load<false>(ebuf[b], &tmY, ybar[b], col0, row0, g, p.c_spS, p.c_spL);
        }
        ypend |= 1u << b;
      }
      if (EPI == kEpiDSwiGLU && rows_valid) {
        // G and U of the warp's first chunk, fetched while the main loop runs
        if (lane == 0) {
          bulk_wait_read0();
          mbar_arrive_expect_tx(ybar[0], 2 * EBOX);
          tma_load_4d(ebuf[0], &tmY, ybar[0], col0, 0, row0, g);
          tma_load_4d(ebuf[1], &tmY, ybar[0], col0, 1, row0, g);
        }
        ypend |= 1u;
      }

      ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8u * (BAR_TFULL + buf), tph, wc));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                          static_cast<uint32_t>(buf * BN + half * WARP_COLS);

      if (rows_valid) {
        for (int j = 0; j < nch && ok; ++j) {
          const int ccol = col0 + j * CW;
          const uint32_t tcol = tl + j * CW;
          // The fused epilogues run as a rolled loop of 16-column TMEM loads: a
          // fully unrolled 64-column body is large enough to evict the MMA
          // warp's instructions from the cache the SM sub-partition shares.
          if (EPI == kEpiPartial) {
            // fp32 partial sums: two boxes of 32 rows x 32 columns (128-byte rows,
            // the same swizzle as the bf16 boxes), group split * G + g of the partials
            uint32_t r0[32], r1[32];
            tmem_ld32(tcol, r0);
            tmem_ld32(tcol + 32, r1);
            tmem_ld_wait(r0);
            tmem_ld_wait(r1);
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              if (ccol + 32 * hb >= p.N) break;  // no box that starts past the last column
              const uint32_t* v = hb ? r1 : r0;
              const uint32_t sb = ebuf[0];
              if (lane == 0) bulk_wait_read0();
              __syncwarp();
#pragma unroll
              for (int c = 0; c < 8; ++c) st_shared_v4(sb + soff(c), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&tmC, sb, ccol + 32 * hb, row0, split * p.G + g);
                bulk_commit();
              }
            }
          } else if (EPI == kEpiStore || EPI == kEpiSplit) {
            // fp16 for the columns before split_cols (whole 64-column chunks)
            const bool f16 = ccol < p.split_cols;
            uint32_t r0[32], r1[32];
            tmem_ld32(tcol, r0);
            tmem_ld32(tcol + 32, r1);
            tmem_ld_wait(r0);
            tmem_ld_wait(r1);
            const uint32_t sb = ebuf[ecount & 1u];
            // one staging box: the previous chunk's store must have read it
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t* v = (c < 4) ? &r0[8 * c] : &r1[8 * (c - 4)];
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = f16 ? pack_f16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]))
                           : pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
              st_shared_v4(sb + soff(c), w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              out_store(&tmC, sb, ccol, row0, g, p.c_spS, p.c_spL);
              bulk_commit();
            }
            ++ecount;
          } else if (EPI == kEpiGelu) {
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
#pragma unroll 1
            for (int q = 0; q < CW / 16; ++q) {
              uint32_t v[16];
              tmem_ld16(tcol + q * 16, v);
              tmem_ld_wait16(v);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const uint32_t c = static_cast<uint32_t>(2 * q + hh);
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(v[8 * hh + e]);
                const uint32_t off = soff(c);
                uint32_t gq[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  float g0, g1;
                  f32x2_split(gelu2(f32x2(x[2 * e], x[2 * e + 1])), g0, g1);
                  gq[e] = pack_bf16x2(g0, g1);
                }
                st_shared_v4(ebuf[0] + off, gq[0], gq[1], gq[2], gq[3]);
                if (p.store_y)
                  st_shared_v4(ebuf[1] + off, pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                               pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmC, ebuf[0], ccol, row0, g);
              if (p.store_y) tma_store_3d(&tmY, ebuf[1], ccol, row0, g);
              bulk_commit();
            }
          } else if (EPI == kEpiSwiGLU) {
            // gate at TMEM columns tcol.., up at tcol + 128..
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
#pragma unroll 1
            for (int q = 0; q < CW / 16; ++q) {
              uint32_t vg[16], vu[16];
              tmem_ld16(tcol + q * 16, vg);
              tmem_ld16(tcol + 128 + q * 16, vu);
              tmem_ld_wait16(vg);
              tmem_ld_wait16(vu);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const uint32_t c = static_cast<uint32_t>(2 * q + hh);
                uint32_t a[4], gg[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float g0 = __uint_as_float(vg[8 * hh + 2 * e]), g1 = __uint_as_float(vg[8 * hh + 2 * e + 1]);
                  const uint64_t g2 = f32x2(g0, g1);
                  uint64_t s2, o2;
                  sigmoid2(g2, s2, o2);
                  float a0, a1;
                  f32x2_split(mul_f32x2(mul_f32x2(g2, s2), f32x2(__uint_as_float(vu[8 * hh + 2 * e]),
                                                                 __uint_as_float(vu[8 * hh + 2 * e + 1]))),
                              a0, a1);
                  a[e] = pack_bf16x2(a0, a1);
                  gg[e] = pack_bf16x2(g0, g1);
                }
                const uint32_t off = soff(c);
                st_shared_v4(ebuf[0] + off, a[0], a[1], a[2], a[3]);
                if (p.store_y) st_shared_v4(ebuf[1] + off, gg[0], gg[1], gg[2], gg[3]);
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmC, ebuf[0], ccol, row0, g);
              bulk_commit();
              if (p.store_y) {
                tma_store_4d(&tmY, ebuf[1], ccol, 0, row0, g);
                bulk_commit();
              }
            }
            if (p.store_y) {
              // the up part goes out through ebuf[0] once the activation store has read it
              if (lane == 0) bulk_wait_read1();
              __syncwarp();
#pragma unroll 1
              for (int q = 0; q < CW / 16; ++q) {
                uint32_t vu[16];
                tmem_ld16(tcol + 128 + q * 16, vu);
                tmem_ld_wait16(vu);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  const uint32_t c = static_cast<uint32_t>(2 * q + hh);
                  const uint32_t* v = &vu[8 * hh];
                  st_shared_v4(ebuf[0] + soff(c),
                               pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                               pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                               pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                               pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
                }
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_4d(&tmY, ebuf[0], ccol, 1, row0, g);
                bulk_commit();
              }
            }
          } else if (EPI == kEpiDSwiGLU) {
            // ebuf[0] <- G, ebuf[1] <- U of this chunk; dG, dU written over them in place
            if (j > 0) {
              if (lane == 0) {
                bulk_wait_read0();
                mbar_arrive_expect_tx(ybar[0], 2 * EBOX);
                tma_load_4d(ebuf[0], &tmY, ybar[0], ccol, 0, row0, g);
                tma_load_4d(ebuf[1], &tmY, ybar[0], ccol, 1, row0, g);
              }
              ypend |= 1u;
            }
            ok = __all_sync(0xffffffffu, mbar_wait(ybar[0], yph & 1u, wc));
            if (!ok) break;
            yph ^= 1u;
            ypend &= ~1u;
#pragma unroll 1
            for (int q = 0; q < CW / 16; ++q) {
              uint32_t v[16];
              tmem_ld16(tcol + q * 16, v);
              tmem_ld_wait16(v);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const uint32_t c = static_cast<uint32_t>(2 * q + hh);
                const uint32_t off = soff(c);
                uint32_t gq[4], uq[4], dg[4], du[4];
                ld_shared_v4(ebuf[0] + off, gq[0], gq[1], gq[2], gq[3]);
                ld_shared_v4(ebuf[1] + off, uq[0], uq[1], uq[2], uq[3]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const uint64_t gv = f32x2(bf16lo_to_f32(gq[e]), bf16hi_to_f32(gq[e]));
                  const uint64_t uv = f32x2(bf16lo_to_f32(uq[e]), bf16hi_to_f32(uq[e]));
                  const uint64_t da = f32x2(__uint_as_float(v[8 * hh + 2 * e]), __uint_as_float(v[8 * hh + 2 * e + 1]));
                  uint64_t sg, om;
                  sigmoid2(gv, sg, om);
                  float r0, r1, q0, q1;
                  // dG = dA U silu'(G), dU = dA silu(G)
                  f32x2_split(mul_f32x2(mul_f32x2(da, uv), mul_f32x2(sg, fma_f32x2(gv, om, f32x2(1.0f, 1.0f)))), r0,
                              r1);
                  f32x2_split(mul_f32x2(mul_f32x2(da, gv), sg), q0, q1);
                  dg[e] = pack_bf16x2(r0, r1);
                  du[e] = pack_bf16x2(q0, q1);
                }
                st_shared_v4(ebuf[0] + off, dg[0], dg[1], dg[2], dg[3]);
                st_shared_v4(ebuf[1] + off, du[0], du[1], du[2], du[3]);
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_4d(&tmC, ebuf[0], ccol, 0, row0, g);
              tma_store_4d(&tmC, ebuf[1], ccol, 1, row0, g);
              bulk_commit();
            }
          } else {  // kEpiDGelu, kEpiResidual: Y / R chunks double-buffered through ebuf
            const uint32_t cb = ecount & 1u, nb2 = cb ^ 1u;
            if (j + 1 < nch) {
              if (lane == 0) {
                bulk_wait_read0();
                mbar_arrive_expect_tx(ybar[nb2], EBOX);
                op_load<false>(ebuf[nb2], &tmY, ybar[nb2], ccol + CW, row0, g, p.c_spS, p.c_spL);
              }
              ypend |= 1u << nb2;
            }
            ok = __all_sync(0xffffffffu, mbar_wait(ybar[cb], (yph >> cb) & 1u, wc));
            if (!ok) break;
            yph ^= 1u << cb;
            ypend &= ~(1u << cb);
#pragma unroll 1
            for (int q = 0; q < CW / 16; ++q) {
              uint32_t v[16];
              tmem_ld16(tcol + q * 16, v);
              tmem_ld_wait16(v);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const uint32_t c = static_cast<uint32_t>(2 * q + hh);
                const uint32_t addr = ebuf[cb] + soff(c);
                uint32_t y0, y1, y2, y3;
                ld_shared_v4(addr, y0, y1, y2, y3);
                const uint32_t yy[4] = {y0, y1, y2, y3};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float a0 = __uint_as_float(v[8 * hh + 2 * e]), a1 = __uint_as_float(v[8 * hh + 2 * e + 1]);
                  const float y0 = bf16lo_to_f32(yy[e]), y1 = bf16hi_to_f32(yy[e]);
                  float r0, r1;
                  if (EPI == kEpiResidual) {
                    r0 = a0 + y0;
                    r1 = a1 + y1;
                  } else {
                    f32x2_split(dgelu2(f32x2(a0, a1), f32x2(y0, y1)), r0, r1);
                  }
                  o[e] = p.c_f16 ? pack_f16x2(r0, r1) : pack_bf16x2(r0, r1);
                }
                st_shared_v4(addr, o[0], o[1], o[2], o[3]);
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              out_store(&tmC, ebuf[cb], ccol, row0, g, p.c_spS, p.c_spL);
              bulk_commit();
            }
            ++ecount;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(mapa_shared(bar0 + 8u * (BAR_TEMPTY + buf), lead));
        else
          mbar_arrive(bar0 + 8u * (BAR_TEMPTY + buf));
      }
    }
    // drain: Y loads still in flight (only after an abort), then the stores
    if (LOADS_Y) {
      for (int b = 0; b < 2; ++b)
        if (ypend & (1u << b)) mbar_wait(ybar[b], (yph >> b) & 1u, wdrain);
    }
    __syncwarp();
    if (lane == 0) bulk_wait0();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // neither CTA leaves while the pair's MMAs or signals may touch it
  if (warp == WARP_MMA) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, GemmShape);

template <bool PAIR, bool A_MN, bool B_MN, int EPI>
KernelFn get_kernel() {
  static std::atomic<bool> configured[kMaxDevices];
  auto fn = &k_gemm<PAIR, A_MN, B_MN, EPI>;
  if (!set_smem_limit_once(reinterpret_cast<const void*>(fn), Cfg<PAIR, EPI>::SMEM_ALLOC, configured)) return nullptr;
  return fn;
}

template <bool PAIR>
KernelFn pick_kernel(bool a_mn, bool b_mn, int epi) {
  if (!a_mn && b_mn && epi == kEpiGelu) return get_kernel<PAIR, false, true, kEpiGelu>();
  if (!a_mn && b_mn && epi == kEpiStore) return get_kernel<PAIR, false, true, kEpiStore>();
  if (!a_mn && b_mn && epi == kEpiSplit) return get_kernel<PAIR, false, true, kEpiSplit>();
  if (!a_mn && !b_mn && epi == kEpiDGelu) return get_kernel<PAIR, false, false, kEpiDGelu>();
  if (!a_mn && !b_mn && epi == kEpiStore) return get_kernel<PAIR, false, false, kEpiStore>();
  if (a_mn && b_mn && epi == kEpiStore) return get_kernel<PAIR, true, true, kEpiStore>();
  if (!a_mn && b_mn && epi == kEpiSwiGLU) return get_kernel<PAIR, false, true, kEpiSwiGLU>();
  if (!a_mn && !b_mn && epi == kEpiDSwiGLU) return get_kernel<PAIR, false, false, kEpiDSwiGLU>();
  if (!a_mn && b_mn && epi == kEpiResidual) return get_kernel<PAIR, false, true, kEpiResidual>();
  if (!a_mn && b_mn && epi == kEpiPartial) return get_kernel<PAIR, false, true, kEpiPartial>();
  if (!a_mn && !b_mn && epi == kEpiPartial) return get_kernel<PAIR, false, false, kEpiPartial>();
  if (a_mn && b_mn && epi == kEpiPartial) return get_kernel<PAIR, true, true, kEpiPartial>();
  return nullptr;
}

// C[r][c] = fp(sum_{j=0}^{ksplit-1} part[j][r][c] (+ R[r][c])) over the G*M rows of N
// columns, the splits added in index order (deterministic); 8 columns per thread,
// 16-byte loads and stores; C and R are [G*M][ldc] 16-bit tensors (R bf16).
__global__ void __launch_bounds__(256) k_splitk_reduce(const float* __restrict__ part, int ksplit, long long rows,
                                                       int N, long long ldc, const uint4* __restrict__ R,
                                                       uint4* __restrict__ C, int c_f16) {
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();
  const long long per_row = N / 8, n8 = rows * per_row, plane = rows * N;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8; i += stride) {
    const long long row = i / per_row;
    const int col = static_cast<int>(i - row * per_row) * 8;
    const float* src = part + row * N + col;
    float4 a = *reinterpret_cast<const float4*>(src), b = *reinterpret_cast<const float4*>(src + 4);
    for (int j = 1; j < ksplit; ++j) {
      const float4 x = *reinterpret_cast<const float4*>(src + j * plane);
      const float4 y = *reinterpret_cast<const float4*>(src + j * plane + 4);
      a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
      b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
    }
    float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const long long o = (row * ldc + col) / 8;
    if (R) {
      const uint4 r = R[o];
      const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[2 * e] += bf16lo_to_f32(rw[e]);
        v[2 * e + 1] += bf16hi_to_f32(rw[e]);
      }
    }
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = c_f16 ? pack_f16x2(v[2 * e], v[2 * e + 1]) : pack_bf16x2(v[2 * e], v[2 * e + 1]);
    C[o] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// split-K is worth its second kernel when the tiles leave most of the GPU idle and
// the K loop is long
constexpr int64_t kSplitMaxTiles = 76;
constexpr int64_t kSplitMinKBlocks = 32;
constexpr int kSplit = 2;

// An MN-major operand whose d0 is a multiple of 64: the 64-element chunks of a row
// become an outer dimension, so a box {64, BK, chunks} lands in shared memory as the
// chunk-major 128-byte-swizzled layout the MMA descriptors read (chunk c at c * 8 KB).
bool chunked_map(CUtensorMap* m, const GemmOperand& o, uint32_t rows) {
  const uint64_t d0 = static_cast<uint64_t>(o.d0), e = 2;
  const uint32_t nch = o.parts == 2 ? 2u : rows / 64u;
  if (o.sp_S > 0) {  // [S/L][B][L][d0] -> {64, L, d0/64, B, S/L}
    const uint64_t L = static_cast<uint64_t>(o.sp_L), Bn = static_cast<uint64_t>(o.d1 / o.sp_S);
    const uint64_t dims[5] = {64u, L, d0 / 64, Bn, static_cast<uint64_t>(o.sp_S / o.sp_L)};
    const uint64_t gs[4] = {d0 * e, 128u, L * d0 * e, Bn * L * d0 * e};
    const uint32_t box[5] = {64u, static_cast<uint32_t>(BK), nch, 1u, 1u};
    return encode_tmap_strided(m, 5, o.ptr, dims, gs, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const uint64_t d1 = static_cast<uint64_t>(o.d1), d2 = static_cast<uint64_t>(o.d2);
  if (o.parts == 2) {  // [d2][d1][2][d0] -> {64, d1, d0/64, 2, d2}
    const uint64_t dims[5] = {64u, d1, d0 / 64, 2u, d2};
    const uint64_t gs[4] = {2 * d0 * e, 128u, d0 * e, d1 * 2 * d0 * e};
    const uint32_t box[5] = {64u, static_cast<uint32_t>(BK), nch, 1u, 1u};
    return encode_tmap_strided(m, 5, o.ptr, dims, gs, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const uint64_t dims[4] = {64u, d1, d0 / 64, d2};  // [d2][d1][d0] -> {64, d1, d0/64, d2}
  const uint64_t gs[3] = {d0 * e, 128u, d1 * d0 * e};
  const uint32_t box[4] = {64u, static_cast<uint32_t>(BK), nch, 1u};
  return encode_tmap_strided(m, 4, o.ptr, dims, gs, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool operand_map(CUtensorMap* m, const GemmOperand& o, uint32_t rows) {
  const uint32_t r = o.mn_major ? static_cast<uint32_t>(BK) : rows;
  if (o.sp_S > 0) {  // [S/L][B][L][d0]
    const uint64_t dims[4] = {static_cast<uint64_t>(o.d0), static_cast<uint64_t>(o.sp_L),
                              static_cast<uint64_t>(o.d1 / o.sp_S), static_cast<uint64_t>(o.sp_S / o.sp_L)};
    const uint32_t box[4] = {64u, r, 1u, 1u};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, o.ptr, dims, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (o.parts == 2) {  // [d2][d1][2][d0]: the part is the second coordinate
    const uint64_t dims[4] = {static_cast<uint64_t>(o.d0), 2u, static_cast<uint64_t>(o.d1),
                              static_cast<uint64_t>(o.d2)};
    const uint32_t box[4] = {64u, 1u, r, 1u};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, o.ptr, dims, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const uint64_t dims[3] = {static_cast<uint64_t>(o.d0), static_cast<uint64_t>(o.d1), static_cast<uint64_t>(o.d2)};
  const uint32_t box[3] = {64u, r, 1u};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o.ptr, dims, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// [G][M][2][N] output or auxiliary tensor of the gated epilogues, 32-row x cw boxes
bool two_part_map(CUtensorMap* m, const void* ptr, int64_t N, int64_t M, int G, uint32_t cw, CUtensorMapSwizzle swz) {
  const uint64_t dims[4] = {static_cast<uint64_t>(N), 2u, static_cast<uint64_t>(M), static_cast<uint64_t>(G)};
  const uint32_t box[4] = {cw, 1u, 32u, 1u};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims, box, swz);
}

int g_tiling_mode = 0;  // 0 automatic, 1 single CTA per tile, 2 CTA pairs

}  // namespace

size_t gemm_splitk_bytes(int64_t M, int64_t N, int G, int S, int64_t Ks) {
  if (M < 1 || N < 1 || G < 1 || S < 1 || Ks < 1) return 0;
  const int64_t tiles = static_cast<int64_t>(G) * ((M + 127) / 128) * ((N + 255) / 256);
  const int64_t nk = static_cast<int64_t>(S) * ((Ks + BK - 1) / BK);
  if (tiles > kSplitMaxTiles || nk < kSplitMinKBlocks) return 0;
  return static_cast<size_t>(kSplit) * static_cast<size_t>(G) * static_cast<size_t>(M) * static_cast<size_t>(N) * 4;
}

bool set_gemm_tiling_mode(int mode) {
  if (mode < 0 || mode > 2) return false;
  g_tiling_mode = mode;
  return true;
}

int launch_gemm_bf16(int epi, const GemmOperand& A, const GemmOperand& B, void* C, const void* Yaux,
                     bool store_y, int64_t M, int64_t N, int G, int S, int64_t Ks, unsigned* err,
                     unsigned long long timeout_ns, cudaStream_t stream, int kind, const GemmExtra& extra) {
  // returns 0 on success, 1 for bad arguments, 2 for a CUDA failure
  if (M < 1 || N < 1 || G < 1 || S < 1 || Ks < 1) return 1;
  const int64_t ldc = extra.ldc > 0 ? extra.ldc : N;
  if ((A.d0 % 8) || (B.d0 % 8) || (N % 8) || (ldc % 8) || ldc < N) return 1;
  if (ldc != N && (N % 64)) return 1;  // a partial last chunk would not be clipped at N
  if (epi == kEpiSplit && (extra.split_cols % 64)) return 1;
  // fp16 outputs: the plain store, the dGeLU and the residual epilogues
  if (extra.c_f16 && epi != kEpiStore && epi != kEpiDGelu && epi != kEpiResidual) return 1;
  const bool gated = epi == kEpiSwiGLU || epi == kEpiDSwiGLU;
  // sequence-sharded operands: the token axis is d1 (A, B) or M (C), d2 = 1, and
  // every box height (128, 64, 32 rows) divides the shard length L
  auto sp_ok = [](int S, int L, int64_t rows, int64_t d2) {
    return S == 0 || (L > 0 && L % 128 == 0 && S % L == 0 && rows % S == 0 && d2 == 1);
  };
  if (!sp_ok(A.sp_S, A.sp_L, A.d1, A.d2) || !sp_ok(B.sp_S, B.sp_L, B.d1, B.d2) ||
      !sp_ok(extra.c_sp_S, extra.c_sp_L, M, G))
    return 1;
  if (B.sp_S > 0 && !B.mn_major) return 1;  // a K-major B operand's rows are not tokens
  if (A.sp_S > 0 && A.mn_major && B.sp_S > 0 && (A.sp_S != B.sp_S || A.sp_L != B.sp_L)) return 1;
  if (extra.c_sp_S > 0 && ((epi != kEpiStore && epi != kEpiResidual) || ldc != N)) return 1;
  if ((A.sp_S > 0 && A.parts != 1) || (B.sp_S > 0 && B.parts != 1)) return 1;
  if (gated && ldc != N) return 1;
  if ((epi == kEpiSwiGLU) != (B.parts == 2) || A.parts != 1) return 1;
  if (epi == kEpiSwiGLU && !B.mn_major) return 1;
  if ((epi == kEpiDSwiGLU || epi == kEpiResidual || epi == kEpiDGelu) && !Yaux) return 1;
  const int64_t tile_n = epi == kEpiSwiGLU ? BN / 2 : BN;
  const int sms = device_sm_count();
  if (sms <= 0) return 2;
  // CTA pairs unless M fits one 128-row tile: a pair stages 32 KB per SM and k-block
  // against 48 KB for a single CTA's 128 x 256 tile, and the SMs' L2 read bandwidth
  // (about 64 bytes per clock each) is what a k-block's copies contend for; for a
  // launch with few tiles both tilings occupy the same number of SMs
  const long long pair_tiles = static_cast<long long>(G) * ((M + 255) / 256) * ((N + tile_n - 1) / tile_n);
  bool pair = g_tiling_mode >= 2 || (g_tiling_mode == 0 && M > 128);
  if (sms < 2) pair = false;
  // split-K for launches whose tiles leave most SMs idle: the K loop in two halves,
  // fp32 partials in the caller's scratch, added in fixed order by k_splitk_reduce
  // (its units: pair tiles on #SM/2 pairs, or single tiles on #SM CTAs)
  const size_t split_bytes = gemm_splitk_bytes(M, N, G, S, Ks);
  const int64_t units1 = pair ? pair_tiles : static_cast<int64_t>(G) * ((M + 127) / 128) * ((N + 255) / 256);
  const bool split = split_bytes > 0 && extra.part_ws && extra.part_ws_bytes >= split_bytes &&
                     (reinterpret_cast<uintptr_t>(extra.part_ws) & 255u) == 0 &&
                     (epi == kEpiStore || epi == kEpiResidual) && extra.c_sp_S == 0 && A.sp_S == 0 && B.sp_S == 0 &&
                     units1 * kSplit <= (pair ? sms / 2 : sms) &&
                     (pair ? pick_kernel<true>(A.mn_major, B.mn_major, kEpiPartial)
                           : pick_kernel<false>(A.mn_major, B.mn_major, kEpiPartial)) != nullptr;
  const int kepi = split ? static_cast<int>(kEpiPartial) : epi;
  KernelFn fn = pair ? pick_kernel<true>(A.mn_major, B.mn_major, kepi) : pick_kernel<false>(A.mn_major, B.mn_major, kepi);
  if (!fn) return 2;
  const uint32_t a_rows = 128, b_rows = pair ? Cfg<true, kEpiStore>::BN_CTA : Cfg<false, kEpiStore>::BN_CTA;
  const bool one_box = epi == kEpiStore || epi == kEpiSplit;
  const int smem = pair ? (one_box ? Cfg<true, kEpiStore>::SMEM_ALLOC : Cfg<true, kEpiGelu>::SMEM_ALLOC)
                        : (one_box ? Cfg<false, kEpiStore>::SMEM_ALLOC : Cfg<false, kEpiGelu>::SMEM_ALLOC);
  CUtensorMap ta, tb, tc, ty;
  // MN-major operands with whole 64-element chunks: one copy per stage
  const bool a_ch = A.mn_major && A.d0 % 64 == 0, b_ch = B.mn_major && B.d0 % 64 == 0;
  if (!(a_ch ? chunked_map(&ta, A, a_rows) : operand_map(&ta, A, a_rows)) ||
      !(b_ch ? chunked_map(&tb, B, b_rows) : operand_map(&tb, B, b_rows)))
    return 2;
  const uint64_t cdims[3] = {static_cast<uint64_t>(ldc), static_cast<uint64_t>(M), static_cast<uint64_t>(G)};
  // staging boxes: 64 columns (128-byte swizzle) for one-box epilogues, 32 (64-byte) for fused ones
  const uint32_t cw = one_box ? 64u : 32u;
  const CUtensorMapSwizzle swz = one_box ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const uint32_t cbox[3] = {cw, 32u, 1u};
  const uint64_t sdims[4] = {static_cast<uint64_t>(ldc), static_cast<uint64_t>(extra.c_sp_L),
                             static_cast<uint64_t>(extra.c_sp_S > 0 ? M / extra.c_sp_S : 1),
                             static_cast<uint64_t>(extra.c_sp_S > 0 ? extra.c_sp_S / extra.c_sp_L : 1)};
  const uint32_t sbox[4] = {cw, 32u, 1u, 1u};
  auto out_map = [&](CUtensorMap* m, const void* ptr) {
    if (extra.c_sp_S > 0)
      return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, sdims, sbox, swz);
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, cdims, cbox, swz);
  };
  if (split) {  // fp32 partials [kSplit][G][M][N], 32 x 32 boxes (128-byte rows)
    const uint64_t pdims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                               static_cast<uint64_t>(kSplit) * static_cast<uint64_t>(G)};
    const uint32_t pbox[3] = {32u, 32u, 1u};
    if (!encode_tmap(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, extra.part_ws, pdims, pbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return 2;
  } else if (epi == kEpiDSwiGLU) {
    if (!two_part_map(&tc, C, N, M, G, cw, swz)) return 2;
  } else if (!out_map(&tc, C)) {
    return 2;
  }
  if (Yaux && gated) {
    if (!two_part_map(&ty, Yaux, N, M, G, cw, swz)) return 2;
  } else if (Yaux) {
    if (!out_map(&ty, Yaux)) return 2;
  } else {
    ty = tc;
  }
  GemmShape p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.G = G;
  p.S = S;
  p.kb_per_seg = static_cast<int>((Ks + BK - 1) / BK);
  p.tiles_m = static_cast<int>((M + (pair ? 255 : 127)) / (pair ? 256 : 128));
  p.tiles_n = static_cast<int>((N + tile_n - 1) / tile_n);
  p.a_zg = A.zg;
  p.a_zs = A.zs;
  p.b_zg = B.zg;
  p.b_zs = B.zs;
  p.store_y = (store_y && Yaux) ? 1 : 0;
  // kEpiStore with c_f16: every column fp16 (N < 2^31)
  p.split_cols = epi == kEpiSplit ? static_cast<int>(extra.split_cols)
                                  : (epi == kEpiStore && extra.c_f16 ? 0x7fffffff : 0);
  p.ab_f16 = extra.ab_f16 ? 1 : 0;
  p.c_f16 = extra.c_f16 ? 1 : 0;
  {
    const int nkb = S * static_cast<int>((Ks + BK - 1) / BK);
    p.ksplit = split ? kSplit : 1;
    p.kps = (nkb + p.ksplit - 1) / p.ksplit;
  }
  p.a_spS = A.sp_S;
  p.a_spL = A.sp_L;
  p.b_spS = B.sp_S;
  p.b_spL = B.sp_L;
  p.c_spS = extra.c_sp_S;
  p.c_spL = extra.c_sp_L;
  // fold the groups into N when they share A (the column-parallel GEMMs' X or dZ);
  // folding into M for a shared B measured slower (more L2 misses) and is not used
  p.g_mode = (G > 1 && A.zg == 0) ? 1 : 0;
  p.a_chunked = a_ch ? 1 : 0;
  p.b_chunked = b_ch ? 1 : 0;
  p.err = err;
  p.timeout_ns = timeout_ns;
  const long long total = static_cast<long long>(G) * p.tiles_m * p.tiles_n * p.ksplit;
  // with split-K the kind's time covers both kernels (one product per launch)
  const int slot = timing_begin(kind, stream);
  bool ok;
  if (pair) {
    // persistent pairs: one per two SMs
    long long units = sms / 2;
    if (units > total) units = total;
    ok = launch_k(fn, dim3(static_cast<unsigned>(2 * units)), dim3(NUM_THREADS), static_cast<size_t>(smem), stream, 2,
                  ta, tb, tc, ty, p) == cudaSuccess;
  } else {
    const int grid = static_cast<int>(total < sms ? total : sms);
    ok = launch_k(fn, dim3(static_cast<unsigned>(grid)), dim3(NUM_THREADS), static_cast<size_t>(smem), stream, 1, ta,
                  tb, tc, ty, p) == cudaSuccess;
  }
  if (ok && split) {
    const long long rows = static_cast<long long>(G) * M, n8 = rows * (N / 8);
    long long blocks = (n8 + 255) / 256;
    if (blocks > static_cast<long long>(sms) * 8) blocks = static_cast<long long>(sms) * 8;
    const int rslot = timing_begin(kKSplitReduce, stream);
    ok = launch_k(k_splitk_reduce, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1,
                  static_cast<const float*>(extra.part_ws), kSplit, rows, static_cast<int>(N), ldc,
                  epi == kEpiResidual ? static_cast<const uint4*>(Yaux) : nullptr, static_cast<uint4*>(C),
                  p.c_f16) == cudaSuccess;
    timing_end(rslot, stream);
  }
  timing_end(slot, stream);
  return ok ? 0 : 2;
}

}  // namespace tpb
