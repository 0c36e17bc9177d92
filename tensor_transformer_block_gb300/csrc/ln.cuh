// LayerNorm launchers (layernorm.cu).  Rows are [T][h] of 16-bit values, bf16
// unless the ``io`` flags below make a tensor fp16; gamma / beta bf16 [h],
// statistics fp32 [T].  Each launcher returns 0 on success, 1 for bad sizes and 2
// for a CUDA launch failure.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace tpb {

constexpr int64_t kLnMaxH = 16384;  // a row is held in the registers of one CTA (<= 1024 x 2 x 8)

// ``err``: the device error word that a debug build's bounds checks latch into.
// ``io`` bits: which row tensors hold fp16 values (the others bf16)
constexpr int kLnXF16 = 1;   // X (forward and backward input)
constexpr int kLnYF16 = 2;   // Y (forward output)
constexpr int kLnDyF16 = 4;  // dY (backward input)
constexpr int kLnDrF16 = 8;  // dR (backward residual gradient)
constexpr int kLnDxF16 = 16; // dX (backward output)

bool ln_shape_ok(int64_t T, int64_t h);

// fp32 scratch of launch_ln_bwd: one [2][h] partial row (dgamma, dbeta) per CTA.
size_t ln_partial_bytes(int64_t T, int64_t h);

// Y = gamma * (X - mean) * rstd + beta per row; mean and rstd = 1/sqrt(var + eps) saved.
int launch_ln_fwd(const void* X, const void* gamma, const void* beta, void* Y, float* mean, float* rstd, int64_t T,
                  int64_t h, float eps, cudaStream_t st, int io = 0, unsigned* err = nullptr);

// dX = rstd (g - mean(g) - xhat mean(g xhat)) + dR with g = dY * gamma (dR may be
// NULL); dgamma = sum_rows dY * xhat, dbeta = sum_rows dY (bf16), finished from
// fp32 per-CTA partial rows in ``part`` (ln_partial_bytes) added in CTA order.
int launch_ln_bwd(const void* X, const void* gamma, const float* mean, const float* rstd, const void* dY,
                  const void* dR, void* dX, void* dgamma, void* dbeta, float* part, int64_t T, int64_t h,
                  cudaStream_t st, int io = 0, unsigned* err = nullptr);

}  // namespace tpb
