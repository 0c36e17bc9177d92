// FP32 GEMM on the CUDA cores (FFMA, no TF32) for the fp32 MLP forward, whose
// tolerance (1e-5 relative) rules out reduced-precision tensor-core inputs.
//   C[g] = sum_{s} A(g,s) * B(g,s)   (row-major, [in x out] weights)
// optionally followed by A_out = GeLU_tanh(C) with the pre-activation kept.
// 64x64 output tile per 256-thread CTA, 4x4 outputs per thread, 16-deep K slices
// staged in double-buffered shared memory; the next slice's global loads are in
// flight while the current one is multiplied.
//
// The K loop of a tile (the S shards x the K slices of each, in that order) is split
// over the KS CTAs of a thread-block cluster when the tiles alone would leave most
// SMs idle (the small token counts this path serves).  Each CTA adds its contiguous
// range of slices into a 64x64 fp32 partial in its shared memory; after a cluster
// barrier CTA r finishes rows [r*64/KS, (r+1)*64/KS) of the tile, adding the KS
// partials in rank order through distributed shared memory, and applies the
// epilogue.  The summation order is fixed by the shape and KS alone: results are
// deterministic, and no workspace is needed.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_simt.cuh"
#include "host_util.cuh"
#include "ptx.cuh"

namespace tpb {
namespace {

constexpr int TM = 64, TN = 64, TK = 16, KS_MAX = 8;

__device__ __forceinline__ float gelu32(float x) {
  const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
  return 0.5f * x * (1.0f + tanhf(u));
}

// C = v, or with the GeLU epilogue Y = v (when kept) and C = GeLU(v).
__device__ __forceinline__ void store_out(float* C, float* Y, int64_t ldc, bool gelu, int gm, int gn, float v) {
  const int64_t o = static_cast<int64_t>(gm) * ldc + gn;
  if (gelu) {
    if (Y) Y[o] = v;
    C[o] = gelu32(v);
  } else {
    C[o] = v;
  }
}

struct SliceRegs {
  float a[4], b[4];
};

// Global -> registers for slice ``sl`` (shard sl / nks, K offset (sl % nks) * TK):
// thread i holds A rows m0 + (i + 256 e) / TK, column (i % TK), and B row
// (i + 256 e) / TN, column (i % TN), zero outside the matrices.
__device__ __forceinline__ void load_slice(const SimtArgs& a, int g, int m0, int n0, int sl, int nks, SliceRegs& r) {
  const int s = sl / nks, k0 = (sl % nks) * TK;
  const float* A = a.A + g * a.a_sg + s * a.a_ss;
  const float* B = a.B + g * a.b_sg + s * a.b_ss;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int i = threadIdx.x + 256 * e;
    const int gm = m0 + i / TK, gk = k0 + i % TK;
    r.a[e] = (gm < a.M && gk < a.K) ? A[static_cast<int64_t>(gm) * a.lda + gk] : 0.0f;
    const int bk = k0 + i / TN, gn = n0 + i % TN;
    r.b[e] = (bk < a.K && gn < a.N) ? B[static_cast<int64_t>(bk) * a.ldb + gn] : 0.0f;
  }
}

__global__ void __launch_bounds__(256, 2) k_gemm_f32(SimtArgs a, int KS) {
  __shared__ __align__(16) float sA[2][TK][TM + 4];
  __shared__ __align__(16) float sB[2][TK][TN + 4];
  __shared__ __align__(16) float part[TM][TN];  // this CTA's partial tile (cluster split)
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();
  const int g = blockIdx.z;
  const int rank = static_cast<int>(blockIdx.x) % KS;  // the cluster spans KS consecutive x
  const int m0 = blockIdx.y * TM, n0 = (static_cast<int>(blockIdx.x) / KS) * TN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int nks = (a.K + TK - 1) / TK;
  const int nsl = a.S * nks;
  const int per = (nsl + KS - 1) / KS;
  const int sl0 = rank * per, sl1 = min(nsl, sl0 + per);

  float acc[4][4] = {};
  SliceRegs r;
  if (sl0 < sl1) load_slice(a, g, m0, n0, sl0, nks, r);
  int buf = 0;
  for (int sl = sl0; sl < sl1; ++sl) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = threadIdx.x + 256 * e;
      sA[buf][i % TK][i / TK] = r.a[e];
      sB[buf][i / TN][i % TN] = r.b[e];
    }
    __syncthreads();
    if (sl + 1 < sl1) load_slice(a, g, m0, n0, sl + 1, nks, r);  // in flight during the products
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&sA[buf][kk][ty * 4]);
      const float4 bv = *reinterpret_cast<const float4*>(&sB[buf][kk][tx * 4]);
      const float ai[4] = {av.x, av.y, av.z, av.w}, bj[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ai[i], bj[j], acc[i][j]);
    }
    buf ^= 1;
  }

  float* C = a.C + g * a.c_sg;
  float* Y = a.Yout ? a.Yout + g * a.c_sg : nullptr;
  const int64_t ldc = a.ldc;
  const bool gelu = a.gelu != 0;
  if (KS == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int gm = m0 + ty * 4 + i;
      if (gm >= a.M) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int gn = n0 + tx * 4 + j;
        if (gn < a.N) store_out(C, Y, ldc, gelu, gm, gn, acc[i][j]);
      }
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(&part[ty * 4 + i][tx * 4]) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  cluster_sync();  // every partial is written and visible to the cluster
  const int rows = TM / KS;
  const uint32_t base = smem_u32(&part[0][0]);
  for (int e = threadIdx.x; e < rows * TN; e += 256) {
    const int row = rank * rows + e / TN, col = e % TN;
    const uint32_t off = base + static_cast<uint32_t>((row * TN + col) * 4);
    float v = 0.0f;
    for (int j = 0; j < KS; ++j) v += ld_dsmem_f32(mapa_shared(off, static_cast<uint32_t>(j)));
    const int gm = m0 + row, gn = n0 + col;
    if (gm < a.M && gn < a.N) store_out(C, Y, ldc, gelu, gm, gn, v);
  }
  cluster_sync();  // no CTA leaves while a peer still reads its partial
}

}  // namespace

int launch_gemm_f32(const SimtArgs& a, cudaStream_t stream, int kind) {
  if (a.M < 1 || a.N < 1 || a.K < 1 || a.G < 1 || a.S < 1) return 1;
  const int tn = (a.N + TN - 1) / TN, tm = (a.M + TM - 1) / TM;
  if (tm > 65535 || a.G > 65535) return 1;
  // split K over a cluster while the tiles fill fewer than two CTAs per SM
  const long long tiles = static_cast<long long>(tn) * tm * a.G;
  const long long nsl = static_cast<long long>(a.S) * ((a.K + TK - 1) / TK);
  const int sms = device_sm_count();
  int KS = 1;
  while (KS < KS_MAX && tiles * KS * 2 <= 2LL * sms && 2 * KS <= nsl) KS *= 2;
  if (static_cast<long long>(tn) * KS > 0x7fffffffLL) return 1;
  const dim3 grid(static_cast<unsigned>(tn * KS), static_cast<unsigned>(tm), static_cast<unsigned>(a.G));
  const int slot = timing_begin(kind, stream);
  const bool ok = launch_k(k_gemm_f32, grid, dim3(256), 0, stream, KS, a, KS) == cudaSuccess;
  timing_end(slot, stream);
  return ok ? 0 : 2;
}

}  // namespace tpb
