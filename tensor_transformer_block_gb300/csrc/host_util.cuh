// Host-side helpers shared by the launchers: TMA tensor-map encoding through the
// driver entry point (no link-time dependency on libcuda), device properties.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <atomic>
#include <utility>

namespace tpb {

// Encodes a tiled TMA map over a row-major tensor of rank 2..5 with bf16 or fp32
// elements.  dims[0] is the contiguous dimension; box[i] <= 256; the
// innermost box extent times the element size must be <= 128 bytes for the
// 128-byte swizzle.  Returns true on success.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint32_t* box, CUtensorMapSwizzle swizzle);
// The same for a bf16 tensor whose dimensions are not packed: gstride[i] is the
// byte stride of dimension i+1 (a multiple of 16), dimension 0 being contiguous.
bool encode_tmap_strided(CUtensorMap* map, int rank, const void* base, const uint64_t* dims, const uint64_t* gstride,
                         const uint32_t* box, CUtensorMapSwizzle swizzle);

// Streaming-multiprocessor count of the current device (cached per device).
int device_sm_count();

// Raises a kernel's dynamic shared-memory limit to ``bytes`` on the current device,
// once per device (the attribute belongs to the device's context); ``done`` is the
// kernel's own per-device flag array.  False if the device or the call fails.
constexpr int kMaxDevices = 64;
bool set_smem_limit_once(const void* fn, int bytes, std::atomic<bool> (&done)[kMaxDevices]);

// Current device's compute capability as major*10+minor, or -1.
int device_cc();

// Programmatic dependent launch (process-wide, on by default): every kernel is
// launched with programmatic stream serialisation, so that its prologue overlaps
// the tail of the kernel before it in the stream (grid_dep_wait in ptx.cuh).  Off,
// each kernel starts after the previous one has completed; results are the same.
void set_launch_overlap(bool on);
bool launch_overlap();

// fn<<<grid, block, smem, st>>>(args...) through cudaLaunchKernelEx, with
// programmatic stream serialisation while launch_overlap() and, for cluster > 1,
// clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*fn)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (launch_overlap()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, std::forward<Args>(args)...);
  if (e != cudaSuccess) (void)cudaGetLastError();  // returned here; not left for a later check
  return e;
}

// Kernel launch registry.  Every launch is counted per kernel kind; while
// timing is on, a pair of CUDA events is recorded on the launch stream around
// it, and timing_read() sums the elapsed times per kind.
enum KernelKind : int {
  kKMlpFc1 = 0,     // column-parallel GEMM + GeLU (Y_i = X W1_i)
  kKMlpFc2,         // row-parallel GEMM, shard sum in the accumulator (Z = sum_i A_i W2_i)
  kKMlpDgelu,       // dY_i = (dZ W2_i^T) * GeLU'(Y_i)
  kKMlpDw2,         // dW2_i = A_i^T dZ
  kKMlpDw1,         // dW1_i = X^T dY_i
  kKMlpDx,          // dX = sum_i dY_i W1_i^T
  kKMlpF32Fc1,      // fp32 column GEMM + GeLU
  kKMlpF32Fc2,      // fp32 row GEMM
  kKAttnQkv,        // [Q K V]_i = X Wqkv_i
  kKAttnCore,       // per-head causal attention forward
  kKAttnOut,        // Z = sum_i O_i Wo_i
  kKAttnDo,         // dO_i = dZ Wo_i^T
  kKAttnDwo,        // dWo_i = O_i^T dZ
  kKAttnDsum,       // rowsum(dO * O)
  kKAttnDkdv,       // dK, dV per key block
  kKAttnDq,         // dQ per query block
  kKAttnDwqkv,      // dWqkv_i = X^T dQKV_i
  kKAttnDx,         // dX = sum_i dQKV_i Wqkv_i^T
  kKGmlpFc1,        // [G_i U_i] = X Wgu_i, A_i = silu(G_i) * U_i
  kKGmlpFc2,        // Z = sum_i A_i Wd_i
  kKGmlpDswiglu,    // dA_i = dZ Wd_i^T -> dG_i, dU_i
  kKGmlpDwd,        // dWd_i = A_i^T dZ
  kKGmlpDwgu,       // dWgu_i = X^T [dG_i dU_i]
  kKGmlpDx,         // dX = sum_i [dG_i dU_i] Wgu_i^T
  kKLnFwd,          // LayerNorm forward
  kKLnBwd,          // LayerNorm backward (+ residual gradient), per-CTA partial dgamma / dbeta
  kKLnColsum,       // fixed-order sum of the partial rows -> dgamma, dbeta
  kKProbe,          // timeout probe
  kKCast,           // bf16 -> fp16 copy of a weight matrix
  kKSplitReduce,    // fixed-order sum of split-K partials (+ residual), 16-bit output
  kNumKernelKinds
};
const char* kernel_kind_name(int k);
int timing_begin(int kind, cudaStream_t st);  // returns a slot (or -1)
void timing_end(int slot, cudaStream_t st);
void timing_enable(bool on);                   // also clears counts and times
bool timing_read(int kind, long long* launches, double* total_ms);

}  // namespace tpb
