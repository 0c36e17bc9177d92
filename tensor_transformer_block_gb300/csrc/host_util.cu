#include "host_util.cuh"

#include <atomic>
#include <mutex>
#include <vector>

namespace tpb {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
}

int g_sms[kMaxDevices] = {0};

}  // namespace

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode || rank < 1 || rank > 5) return false;
  const uint64_t esz = (dtype == CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ? 4 : 2;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  uint64_t stride = esz;
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i > 0) gstride[i - 1] = stride;
    stride *= dims[i];
  }
  CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gdim, gstride, bdim,
                        estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_strided(CUtensorMap* map, int rank, const void* base, const uint64_t* dims, const uint64_t* gstride,
                         const uint32_t* box, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode || rank < 1 || rank > 5) return false;
  cuuint64_t gdim[5], gs[4];
  cuuint32_t bdim[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i > 0) gs[i - 1] = gstride[i - 1];
  }
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                        gdim, gs, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices && g_sms[dev] > 0) return g_sms[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) g_sms[dev] = n;
  return n;
}

int device_cc() {
  int dev = 0, ma = 0, mi = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return -1;
  return ma * 10 + mi;
}

namespace {

const char* const kKindNames[kNumKernelKinds] = {
    "mlp.fc1_col_gemm_gelu", "mlp.fc2_row_gemm_shard_sum", "mlp.bwd_dA_gemm_dgelu", "mlp.bwd_dW2_gemm",
    "mlp.bwd_dW1_gemm", "mlp.bwd_dX_row_gemm_shard_sum", "mlp.f32_fc1_col_gemm_gelu", "mlp.f32_fc2_row_gemm",
    "attn.qkv_col_gemm", "attn.core_fwd", "attn.out_row_gemm_shard_sum", "attn.bwd_dO_gemm", "attn.bwd_dWo_gemm",
    "attn.bwd_dsum", "attn.bwd_core_dkdv", "attn.bwd_core_dq", "attn.bwd_dWqkv_gemm",
    "attn.bwd_dX_row_gemm_shard_sum", "gmlp.fc1_col_gemm_swiglu", "gmlp.fc2_row_gemm_shard_sum",
    "gmlp.bwd_dA_gemm_dswiglu", "gmlp.bwd_dWd_gemm", "gmlp.bwd_dWgu_gemm", "gmlp.bwd_dX_row_gemm_shard_sum",
    "ln.fwd", "ln.bwd_residual", "ln.bwd_colsum", "debug.timeout_probe", "cast.bf16_to_f16",
    "gemm.splitk_reduce"};

struct Slot {
  int kind;
  cudaEvent_t a, b;
};

std::mutex g_tmu;
bool g_timing = false;
long long g_launches[kNumKernelKinds] = {0};
std::vector<Slot> g_slots;      // recorded this timing window
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

namespace {
std::atomic<bool> g_overlap{true};
}  // namespace

bool set_smem_limit_once(const void* fn, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  if (done[dev].load()) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  done[dev].store(true);
  return true;
}

void set_launch_overlap(bool on) { g_overlap.store(on); }
bool launch_overlap() { return g_overlap.load(); }

const char* kernel_kind_name(int k) { return (k >= 0 && k < kNumKernelKinds) ? kKindNames[k] : nullptr; }

int timing_begin(int kind, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_tmu);
  if (kind < 0 || kind >= kNumKernelKinds) return -1;
  ++g_launches[kind];
  if (!g_timing) return -1;
  Slot s{kind, take_event(), take_event()};
  if (!s.a || !s.b || cudaEventRecord(s.a, st) != cudaSuccess) return -1;
  g_slots.push_back(s);
  return static_cast<int>(g_slots.size()) - 1;
}

void timing_end(int slot, cudaStream_t st) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_tmu);
  if (slot < static_cast<int>(g_slots.size())) cudaEventRecord(g_slots[slot].b, st);
}

void timing_enable(bool on) {
  std::lock_guard<std::mutex> lk(g_tmu);
  for (auto& s : g_slots) {
    cudaEventSynchronize(s.b);
    g_pool.push_back(s.a);
    g_pool.push_back(s.b);
  }
  g_slots.clear();
  for (auto& c : g_launches) c = 0;
  g_timing = on;
}

bool timing_read(int kind, long long* launches, double* total_ms) {
  std::lock_guard<std::mutex> lk(g_tmu);
  if (kind < 0 || kind >= kNumKernelKinds) return false;
  double t = 0.0;
  for (auto& s : g_slots) {
    if (s.kind != kind) continue;
    if (cudaEventSynchronize(s.b) != cudaSuccess) return false;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, s.a, s.b) != cudaSuccess) return false;
    t += ms;
  }
  if (launches) *launches = g_launches[kind];
  if (total_ms) *total_ms = t;
  return true;
}

}  // namespace tpb
