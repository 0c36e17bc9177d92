// Per-head fused causal attention on tcgen05 (forward and backward cores).
//
// Tensors are in the shard-major layouts of the boundary:
//   QKV  [N][B][S][5][H/N][d]   planes: Q, K, V, then the bf16 residuals
//                               Q - bf16(Q) and K - bf16(K) of the projection
//   O    [N][B][S][H/N][d]
//   LSE  [B][H][S] fp32          natural-log sum of exp of the scaled scores
// Global head j lives in shard i = j / (H/N) as local head jj = j % (H/N)
// (io.zouht.com 张量并行 §2.2.1: each shard owns whole heads).
//
// Scores are computed split-bf16: S = Qh Kh^T + Qh Kl^T + Ql Kh^T with Qh =
// bf16(Q), Ql = bf16(Q - Qh) (same for K), which carries Q K^T to ~2^-16
// relative instead of bf16's 2^-9; the softmax exponentiates scores whose range
// reaches tens of units, where bf16 Q and K would move the largest weights by
// several percent.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace tpb {

struct AttnDims {
  int B, S, H, hN, N, d, causal;
};

// Number of d-wide planes per (token, local head) in QKV.
constexpr int kQkvPlanes = 5;

// Forward: O and LSE from QKV (returns 0, 1 bad arguments, 2 CUDA failure).
int launch_attn_fwd(const AttnDims& a, const void* qkv, void* o, float* lse, unsigned* err,
                    unsigned long long timeout_ns, cudaStream_t st);

// Backward cores.  Dsum[b][j][s] = sum_e dO * O over the head dim; dqkv
// [N][B][S][3][H/N][d] gets dQ, dK, dV.
int launch_attn_bwd(const AttnDims& a, const void* qkv, const void* o, const void* dout, const float* lse,
                    float* dsum, void* dqkv, unsigned* err, unsigned long long timeout_ns, cudaStream_t st);

}  // namespace tpb
