// bf16 -> fp16 copy of a weight matrix, for the products whose other operand is
// an fp16 activation (one tcgen05 MMA takes A and B of one type).  Every bf16
// value of magnitude 2^-17 .. 65504 is exactly representable in fp16 (bf16 has 8
// significant bits, fp16 11, and fp16 subnormals reach 2^-24), so the copy is
// exact there; smaller magnitudes round to the nearest multiple of 2^-24 (an
// absolute error of at most 2^-25); larger ones overflow to infinity.
//
// HBM-bound: one 16-byte load and one 16-byte store per thread and iteration,
// a grid of resident CTAs striding over the tensor.
#include <cuda_fp16.h>

#include <cstdint>

#include "cast.cuh"
#include "host_util.cuh"
#include "ptx.cuh"

namespace tpb {
namespace {

__global__ void __launch_bounds__(256) k_bf16_to_f16(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                     long long n8) {
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8; i += stride) {
    const uint4 v = in[i];
    uint4 r;
    r.x = pack_f16x2(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x));
    r.y = pack_f16x2(bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
    r.z = pack_f16x2(bf16lo_to_f32(v.z), bf16hi_to_f32(v.z));
    r.w = pack_f16x2(bf16lo_to_f32(v.w), bf16hi_to_f32(v.w));
    out[i] = r;
  }
}

}  // namespace

int launch_bf16_to_f16(const void* in, void* out, long long n, cudaStream_t st) {
  if (n < 0 || (n % 8) || (reinterpret_cast<uintptr_t>(in) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u))
    return 1;
  if (n == 0) return 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 2;
  const long long n8 = n / 8;
  long long blocks = (n8 + 255) / 256;
  if (blocks > static_cast<long long>(sms) * 8) blocks = static_cast<long long>(sms) * 8;  // 8 x 256 threads per SM
  const int slot = timing_begin(kKCast, st);
  const bool ok = launch_k(k_bf16_to_f16, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1,
                           static_cast<const uint4*>(in), static_cast<uint4*>(out), n8) == cudaSuccess;
  timing_end(slot, st);
  return ok ? 0 : 2;
}

}  // namespace tpb
