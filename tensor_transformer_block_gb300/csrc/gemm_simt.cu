// FP32 GEMM on the CUDA cores (FFMA, no TF32) for the fp32 MLP forward, whose
// tolerance (1e-5 relative) rules out reduced-precision tensor-core inputs.
//   C[g] = sum_{s} A(g,s) * B(g,s)   (row-major, [in x out] weights)
// optionally followed by A_out = GeLU_tanh(C) with the pre-activation kept.
// 64x64 output tile per 256-thread block, 4x4 outputs per thread, 16-deep K slices
// staged in shared memory.  The row-parallel case (S = N shards) accumulates all
// shards in the same registers in order s = 0..S-1.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_simt.cuh"
#include "host_util.cuh"

namespace tpb {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

__device__ __forceinline__ float gelu32(float x) {
  const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
  return 0.5f * x * (1.0f + tanhf(u));
}

__global__ void __launch_bounds__(256) k_gemm_f32(SimtArgs a) {
  __shared__ float sA[TK][TM + 4];
  __shared__ float sB[TK][TN + 4];
  const int g = blockIdx.z;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int s = 0; s < a.S; ++s) {
    const float* A = a.A + g * a.a_sg + s * a.a_ss;
    const float* B = a.B + g * a.b_sg + s * a.b_ss;
    for (int k0 = 0; k0 < a.K; k0 += TK) {
      for (int i = threadIdx.x; i < TM * TK; i += 256) {
        const int r = i / TK, c = i % TK;
        const int gm = m0 + r, gk = k0 + c;
        sA[c][r] = (gm < a.M && gk < a.K) ? A[static_cast<int64_t>(gm) * a.lda + gk] : 0.0f;
      }
      for (int i = threadIdx.x; i < TK * TN; i += 256) {
        const int r = i / TN, c = i % TN;
        const int gk = k0 + r, gn = n0 + c;
        sB[r][c] = (gk < a.K && gn < a.N) ? B[static_cast<int64_t>(gk) * a.ldb + gn] : 0.0f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < TK; ++kk) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = sA[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = sB[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      __syncthreads();
    }
  }
  float* C = a.C + g * a.c_sg;
  float* Y = a.Yout ? a.Yout + g * a.c_sg : nullptr;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= a.N) continue;
      const int64_t o = static_cast<int64_t>(gm) * a.ldc + gn;
      if (a.gelu) {
        if (Y) Y[o] = acc[i][j];
        C[o] = gelu32(acc[i][j]);
      } else {
        C[o] = acc[i][j];
      }
    }
  }
}

}  // namespace

int launch_gemm_f32(const SimtArgs& a, cudaStream_t stream, int kind) {
  if (a.M < 1 || a.N < 1 || a.K < 1 || a.G < 1 || a.S < 1) return 1;
  dim3 grid((a.N + TN - 1) / TN, (a.M + TM - 1) / TM, a.G);
  if (grid.y > 65535 || grid.z > 65535) return 1;
  const int slot = timing_begin(kind, stream);
  k_gemm_f32<<<grid, 256, 0, stream>>>(a);
  const bool ok = cudaGetLastError() == cudaSuccess;
  timing_end(slot, stream);
  return ok ? 0 : 2;
}

}  // namespace tpb
