#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace tpb {

// C[g] (M x N, ldc) = sum_{s<S} A[g*a_sg + s*a_ss] (M x K, lda) * B[g*b_sg + s*b_ss] (K x N, ldb)
// If gelu: C = GeLU_tanh(acc) and, when Yout is not NULL, Yout = acc (same strides as C).
struct SimtArgs {
  const float* A;
  const float* B;
  float* C;
  float* Yout;
  int M, N, K, G, S;
  int64_t a_sg, a_ss, b_sg, b_ss, c_sg;
  int64_t lda, ldb, ldc;
  int gelu;
};

int launch_gemm_f32(const SimtArgs& a, cudaStream_t stream, int kind);

}  // namespace tpb
