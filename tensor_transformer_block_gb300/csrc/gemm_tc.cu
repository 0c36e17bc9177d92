// tcgen05 GEMM with TMA multi-stage pipeline and fused epilogues (see gemm_tc.cuh).
//
// CTA = 6 warps, one CTA per SM, persistent over output tiles of 128 x 256:
//   warp 4  TMA producer: fills a 4-stage ring of (A 128x64, B 256x64) bf16 tiles,
//           128-byte swizzled, K-major or MN-major as the operand is stored;
//   warp 5  MMA issuer: 4 x tcgen05.mma (M=128, N=256, K=16) per stage into one of
//           two TMEM accumulators (2 x 256 fp32 columns), so the epilogue of tile t
//           overlaps the main loop of tile t+1;
//   warps 0-3 epilogue: tcgen05.ld 32 rows each, fused GeLU / GeLU' in fp32,
//           bf16 pack into a swizzled staging box, TMA store (coalesced 128-byte rows).
// Every wait is bounded; on a timeout the CTA latches an error, drains its own
// copies and MMAs, frees TMEM and returns.
#include "gemm_tc.cuh"
#include "host_util.cuh"
#include "ptx.cuh"

namespace tpb {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 4;
constexpr int EPI_BUF = 32 * 128;  // one 32-row x 64-column bf16 box
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int GROUP_M = 16;

constexpr int BAR_FULL = 0;
constexpr int BAR_EMPTY = STAGES;
constexpr int BAR_TFULL = 2 * STAGES;
constexpr int BAR_TEMPTY = 2 * STAGES + 2;
constexpr int BAR_Y = 2 * STAGES + 4;
constexpr int BAR_DRAIN = BAR_Y + 2 * EPI_WARPS;
constexpr int NUM_BARS = BAR_DRAIN + 1;

constexpr int SMEM_EPI_OFF = STAGES * STAGE_BYTES;
constexpr int SMEM_BAR_OFF = SMEM_EPI_OFF + EPI_WARPS * 2 * EPI_BUF;
constexpr int SMEM_MISC_OFF = SMEM_BAR_OFF + NUM_BARS * 8;
constexpr int SMEM_USED = SMEM_MISC_OFF + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

__device__ __forceinline__ void decode_tile(int t, const GemmShape& p, int& g, int& mb, int& nb) {
  const int per_g = p.tiles_m * p.tiles_n;
  g = t / per_g;
  const int r = t - g * per_g;
  const int span = GROUP_M * p.tiles_n;
  const int grp = r / span;
  const int first_m = grp * GROUP_M;
  const int gm = min(p.tiles_m - first_m, GROUP_M);
  const int rr = r - grp * span;
  mb = first_m + rr % gm;
  nb = rr / gm;
}

__device__ __forceinline__ float gelu_f(float x) {
  const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
  return 0.5f * x * (1.0f + tanhf(u));
}

__device__ __forceinline__ float gelu_grad_f(float x) {
  const float x2 = x * x;
  const float u = 0.7978845608028654f * (x + 0.044715f * x2 * x);
  const float t = tanhf(u);
  return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * 0.7978845608028654f * (1.0f + 0.134145f * x2);
}

template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmY, const GemmShape p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const uint32_t bar0 = sbase + SMEM_BAR_OFF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SMEM_MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SMEM_MISC_OFF + 4);
  volatile int* never_flag = reinterpret_cast<volatile int*>(smem + SMEM_MISC_OFF + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bar0 + 8u * (BAR_FULL + i), 1);
      mbar_init(bar0 + 8u * (BAR_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar0 + 8u * (BAR_TFULL + i), 1);
      mbar_init(bar0 + 8u * (BAR_TEMPTY + i), EPI_WARPS);
    }
    for (int i = 0; i < 2 * EPI_WARPS; ++i) mbar_init(bar0 + 8u * (BAR_Y + i), 1);
    mbar_init(bar0 + 8u * BAR_DRAIN, 1);
    *abort_flag = 0;
    *never_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
    if (EPI != kEpiStore) prefetch_tmap(&tmY);
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const WaitCtx wc{p.err, abort_flag, p.timeout_ns};
  const WaitCtx wdrain{p.err, never_flag, p.timeout_ns};
  const int total = p.G * p.tiles_m * p.tiles_n;
  const int nk = p.S * p.kb_per_seg;

  if (warp == 4) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int g, mb, nb;
        decode_tile(t, p, g, mb, nb);
        for (int s = 0; s < p.S && ok; ++s) {
          const int az = g * p.a_zg + s * p.a_zs;
          const int bz = g * p.b_zg + s * p.b_zs;
          for (int kb = 0; kb < p.kb_per_seg; ++kb) {
            if (!mbar_wait(bar0 + 8u * (BAR_EMPTY + stage), phase ^ 1u, wc)) {
              ok = false;
              break;
            }
            const uint32_t fb = bar0 + 8u * (BAR_FULL + stage);
            mbar_arrive_expect_tx(fb, STAGE_BYTES);
            const uint32_t sa = sbase + stage * STAGE_BYTES;
            const uint32_t sb = sa + A_BYTES;
            const int kc = kb * BK;
            if (A_MN) {
#pragma unroll
              for (int j = 0; j < BM / 64; ++j) tma_load_3d(sa + j * (BK * 128), &tmA, fb, mb * BM + j * 64, kc, az);
            } else {
              tma_load_3d(sa, &tmA, fb, kc, mb * BM, az);
            }
            if (B_MN) {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tma_load_3d(sb + j * (BK * 128), &tmB, fb, nb * BN + j * 64, kc, bz);
            } else {
              tma_load_3d(sb, &tmB, fb, kc, nb * BN, bz);
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
      // every issued copy must land before the CTA may exit
      for (int s2 = 0; s2 < STAGES; ++s2)
        if (issued & (1u << s2)) mbar_wait(bar0 + 8u * (BAR_FULL + s2), (last_par >> s2) & 1u, wdrain);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t IDESC = idesc_bf16(BM, BN, A_MN, B_MN);
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true, any = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t tph = (it >> 1) & 1;
        if (!mbar_wait(bar0 + 8u * (BAR_TEMPTY + buf), tph ^ 1u, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int k = 0; k < nk; ++k) {
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
            tc_mma_bf16(dt, ad, bd, IDESC, (k | kk) != 0 ? 1u : 0u);
          }
          any = true;
          tc_commit(bar0 + 8u * (BAR_EMPTY + stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(bar0 + 8u * (BAR_TFULL + buf));
      }
      if (any) {
        tc_commit(bar0 + 8u * BAR_DRAIN);
        mbar_wait(bar0 + 8u * BAR_DRAIN, 0, wdrain);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int ew = warp;  // TMEM lanes 32*ew .. 32*ew+31
    const uint32_t ebuf[2] = {sbase + SMEM_EPI_OFF + ew * 2 * EPI_BUF, sbase + SMEM_EPI_OFF + ew * 2 * EPI_BUF + EPI_BUF};
    const uint32_t ybar[2] = {bar0 + 8u * (BAR_Y + 2 * ew), bar0 + 8u * (BAR_Y + 2 * ew + 1)};
    const uint32_t rsw = static_cast<uint32_t>(lane & 7);
    uint32_t yph = 0;      // bit b: parity of the next completion of ybar[b]
    uint32_t ypend = 0;    // bit b: a Y load into ebuf[b] is in flight
    uint32_t ecount = 0;   // chunks staged so far (buffer alternation for kEpiStore / kEpiDGelu)
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
      int g, mb, nb;
      decode_tile(t, p, g, mb, nb);
      const int buf = it & 1;
      const uint32_t tph = (it >> 1) & 1;
      const int row0 = mb * BM + ew * 32;
      const int col0 = nb * BN;
      int nch = (p.N - col0 + 63) / 64;
      if (nch > BN / 64) nch = BN / 64;
      const bool rows_valid = row0 < p.M;

      if (EPI == kEpiDGelu && rows_valid) {
        const uint32_t b = ecount & 1u;
        if (lane == 0) {
          bulk_wait_read0();
          mbar_arrive_expect_tx(ybar[b], EPI_BUF);
          tma_load_3d(ebuf[b], &tmY, ybar[b], col0, row0, g);
        }
        ypend |= 1u << b;
      }

      ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8u * (BAR_TFULL + buf), tph, wc));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(buf * BN);

      if (rows_valid) {
        for (int j = 0; j < nch && ok; ++j) {
          uint32_t r0[32], r1[32];
          tmem_ld32(tl + j * 64, r0);
          tmem_ld32(tl + j * 64 + 32, r1);
          tmem_ld_wait(r0);
          tmem_ld_wait(r1);
          const int ccol = col0 + j * 64;

          if (EPI == kEpiStore) {
            const uint32_t sb = ebuf[ecount & 1u];
            if (lane == 0) bulk_wait_read1();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t* v = (c < 4) ? &r0[8 * c] : &r1[8 * (c - 4)];
              st_shared_v4(sb + lane * 128 + ((c ^ rsw) << 4),
                           pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                           pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                           pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                           pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmC, sb, ccol, row0, g);
              bulk_commit();
            }
            ++ecount;
          } else if (EPI == kEpiSplit) {
            const bool with_lo = ccol < p.split_cols;
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t* v = (c < 4) ? &r0[8 * c] : &r1[8 * (c - 4)];
              uint32_t hi[4], lo[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float x0 = __uint_as_float(v[2 * e]), x1 = __uint_as_float(v[2 * e + 1]);
                hi[e] = pack_bf16x2(x0, x1);
                lo[e] = pack_bf16x2(x0 - bf16lo_to_f32(hi[e]), x1 - bf16hi_to_f32(hi[e]));
              }
              const uint32_t off = lane * 128 + ((c ^ rsw) << 4);
              st_shared_v4(ebuf[0] + off, hi[0], hi[1], hi[2], hi[3]);
              if (with_lo) st_shared_v4(ebuf[1] + off, lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmC, ebuf[0], ccol, row0, g);
              if (with_lo) tma_store_3d(&tmC, ebuf[1], ccol + p.lo_off, row0, g);
              bulk_commit();
            }
          } else if (EPI == kEpiGelu) {
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t* v = (c < 4) ? &r0[8 * c] : &r1[8 * (c - 4)];
              float x[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(v[e]);
              const uint32_t off = lane * 128 + ((c ^ rsw) << 4);
              st_shared_v4(ebuf[0] + off, pack_bf16x2(gelu_f(x[0]), gelu_f(x[1])),
                           pack_bf16x2(gelu_f(x[2]), gelu_f(x[3])), pack_bf16x2(gelu_f(x[4]), gelu_f(x[5])),
                           pack_bf16x2(gelu_f(x[6]), gelu_f(x[7])));
              if (p.store_y)
                st_shared_v4(ebuf[1] + off, pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                             pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmC, ebuf[0], ccol, row0, g);
              if (p.store_y) tma_store_3d(&tmY, ebuf[1], ccol, row0, g);
              bulk_commit();
            }
          } else {  // kEpiDGelu
            const uint32_t cb = ecount & 1u, nb2 = cb ^ 1u;
            if (j + 1 < nch) {
              if (lane == 0) {
                bulk_wait_read0();
                mbar_arrive_expect_tx(ybar[nb2], EPI_BUF);
                tma_load_3d(ebuf[nb2], &tmY, ybar[nb2], ccol + 64, row0, g);
              }
              ypend |= 1u << nb2;
            }
            ok = __all_sync(0xffffffffu, mbar_wait(ybar[cb], (yph >> cb) & 1u, wc));
            if (!ok) break;
            yph ^= 1u << cb;
            ypend &= ~(1u << cb);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t* v = (c < 4) ? &r0[8 * c] : &r1[8 * (c - 4)];
              const uint32_t addr = ebuf[cb] + lane * 128 + ((c ^ rsw) << 4);
              uint32_t y0, y1, y2, y3;
              ld_shared_v4(addr, y0, y1, y2, y3);
              const uint32_t yy[4] = {y0, y1, y2, y3};
              uint32_t o[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float lo = __uint_as_float(v[2 * e]) * gelu_grad_f(bf16lo_to_f32(yy[e]));
                const float hi = __uint_as_float(v[2 * e + 1]) * gelu_grad_f(bf16hi_to_f32(yy[e]));
                o[e] = pack_bf16x2(lo, hi);
              }
              st_shared_v4(addr, o[0], o[1], o[2], o[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmC, ebuf[cb], ccol, row0, g);
              bulk_commit();
            }
            ++ecount;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar0 + 8u * (BAR_TEMPTY + buf));
    }
    // drain: Y loads still in flight (only after an abort), then the stores
    if (EPI == kEpiDGelu) {
      for (int b = 0; b < 2; ++b)
        if (ypend & (1u << b)) mbar_wait(ybar[b], (yph >> b) & 1u, wdrain);
    }
    __syncwarp();
    if (lane == 0) bulk_wait0();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, GemmShape);

template <bool A_MN, bool B_MN, int EPI>
KernelFn get_kernel() {
  static bool configured = false;
  auto fn = &k_gemm<A_MN, B_MN, EPI>;
  if (!configured) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC) != cudaSuccess)
      return nullptr;
    configured = true;
  }
  return reinterpret_cast<KernelFn>(fn);
}

KernelFn pick_kernel(bool a_mn, bool b_mn, int epi) {
  if (!a_mn && b_mn && epi == kEpiGelu) return get_kernel<false, true, kEpiGelu>();
  if (!a_mn && b_mn && epi == kEpiStore) return get_kernel<false, true, kEpiStore>();
  if (!a_mn && b_mn && epi == kEpiSplit) return get_kernel<false, true, kEpiSplit>();
  if (!a_mn && !b_mn && epi == kEpiDGelu) return get_kernel<false, false, kEpiDGelu>();
  if (!a_mn && !b_mn && epi == kEpiStore) return get_kernel<false, false, kEpiStore>();
  if (a_mn && b_mn && epi == kEpiStore) return get_kernel<true, true, kEpiStore>();
  return nullptr;
}

bool operand_map(CUtensorMap* m, const GemmOperand& o, bool is_a) {
  const uint64_t dims[3] = {static_cast<uint64_t>(o.d0), static_cast<uint64_t>(o.d1), static_cast<uint64_t>(o.d2)};
  const uint32_t rows = is_a ? BM : BN;
  const uint32_t box[3] = {64u, o.mn_major ? static_cast<uint32_t>(BK) : rows, 1u};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o.ptr, dims, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

int launch_gemm_bf16(int epi, const GemmOperand& A, const GemmOperand& B, void* C, const void* Yaux,
                     bool store_y, int64_t M, int64_t N, int G, int S, int64_t Ks, unsigned* err,
                     unsigned long long timeout_ns, cudaStream_t stream, int kind, const GemmExtra& extra) {
  // returns 0 on success, 1 for bad arguments, 2 for a CUDA failure
  if (M < 1 || N < 1 || G < 1 || S < 1 || Ks < 1) return 1;
  const int64_t ldc = extra.ldc > 0 ? extra.ldc : N;
  if ((A.d0 % 8) || (B.d0 % 8) || (N % 8) || (ldc % 8) || ldc < N) return 1;
  if (ldc != N && (N % 64)) return 1;  // a partial last chunk would not be clipped at N
  if (epi == kEpiSplit && ((extra.split_cols % 64) || extra.lo_off < N || extra.lo_off + extra.split_cols > ldc))
    return 1;
  KernelFn fn = pick_kernel(A.mn_major, B.mn_major, epi);
  if (!fn) return 2;
  CUtensorMap ta, tb, tc, ty;
  if (!operand_map(&ta, A, true) || !operand_map(&tb, B, false)) return 2;
  const uint64_t cdims[3] = {static_cast<uint64_t>(ldc), static_cast<uint64_t>(M), static_cast<uint64_t>(G)};
  const uint32_t cbox[3] = {64u, 32u, 1u};
  if (!encode_tmap(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, C, cdims, cbox, CU_TENSOR_MAP_SWIZZLE_128B)) return 2;
  if (Yaux) {
    if (!encode_tmap(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, Yaux, cdims, cbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return 2;
  } else {
    ty = tc;
  }
  GemmShape p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.G = G;
  p.S = S;
  p.kb_per_seg = static_cast<int>((Ks + BK - 1) / BK);
  p.tiles_m = static_cast<int>((M + BM - 1) / BM);
  p.tiles_n = static_cast<int>((N + BN - 1) / BN);
  p.a_zg = A.zg;
  p.a_zs = A.zs;
  p.b_zg = B.zg;
  p.b_zs = B.zs;
  p.store_y = (store_y && Yaux) ? 1 : 0;
  p.split_cols = static_cast<int>(extra.split_cols);
  p.lo_off = static_cast<int>(extra.lo_off);
  p.err = err;
  p.timeout_ns = timeout_ns;
  const long long total = static_cast<long long>(G) * p.tiles_m * p.tiles_n;
  const int sms = device_sm_count();
  if (sms <= 0) return 2;
  const int grid = static_cast<int>(total < sms ? total : sms);
  const int slot = timing_begin(kind, stream);
  fn<<<grid, NUM_THREADS, SMEM_ALLOC, stream>>>(ta, tb, tc, ty, p);
  const bool ok = cudaGetLastError() == cudaSuccess;
  timing_end(slot, stream);
  return ok ? 0 : 2;
}

}  // namespace tpb
