// bf16 -> fp16 copies of weight matrices (cast.cu).
#pragma once

#include <cuda_runtime.h>

namespace tpb {

// out[i] = fp16(in[i]) for n 16-bit elements; n a multiple of 8, both pointers
// 16-byte aligned.  Returns 0, 1 for bad arguments, 2 for a CUDA failure.
int launch_bf16_to_f16(const void* in, void* out, long long n, cudaStream_t st);

}  // namespace tpb
