// C-ABI entry points of libtpblock (declared in include/tpblock.h): argument
// validation, workspace carving and the kernel sequence of each call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/tpblock.h"
#include "attn.cuh"
#include "cast.cuh"
#include "gemm_simt.cuh"
#include "gemm_tc.cuh"
#include "host_util.cuh"
#include "ln.cuh"
#include "ptx.cuh"

// Device error word: kernels latch bits here (atomicOr); tp_sync_status reads and clears it.
__device__ unsigned g_tp_error_word;

namespace {

constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // bounded waits give up after 2 s
constexpr int kMaxDev = 64;
int g_dev_ok[kMaxDev];            // 0 unknown, 1 ok, -1 not sm_103
unsigned* g_err_ptr[kMaxDev];

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDev) return -1;
  return d;
}

int check_device(unsigned** err) {
  const int d = current_device();
  if (d < 0) return TP_ERR_CUDA;
  if (g_dev_ok[d] == 0) {
    const int cc = tpb::device_cc();
    if (cc < 0) return TP_ERR_CUDA;
    if (cc != 103) {
      g_dev_ok[d] = -1;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_tp_error_word) != cudaSuccess) return TP_ERR_CUDA;
      g_err_ptr[d] = static_cast<unsigned*>(p);
      g_dev_ok[d] = 1;
    }
  }
  if (g_dev_ok[d] < 0) return TP_ERR_DEVICE;
  if (err) *err = g_err_ptr[d];
  return TP_OK;
}

// An NVTX range (domain "libtpblock") around every C-ABI call, named after the
// call: a profiler attached to the process sees each call and the kernels it
// launched inside it.  With no tool attached a range costs a function-pointer
// check.  NVTX v3 is header-only; a tool is found through the environment.
nvtxDomainHandle_t trace_domain() {
  static const nvtxDomainHandle_t d = nvtxDomainCreateA("libtpblock");
  return d;
}
struct TraceRange {
  explicit TraceRange(const char* name) {
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    nvtxDomainRangePushEx(trace_domain(), &a);
  }
  ~TraceRange() { nvtxDomainRangePop(trace_domain()); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};
#define TP_TRACE const TraceRange tp_trace_range_(__func__)

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int gemm_status(int rc) { return rc == 0 ? TP_OK : (rc == 1 ? TP_ERR_SHAPE : TP_ERR_CUDA); }

// Sequence-sharded activations (zouht 张量并行 §2.2.2, 与序列并行结合): outside the
// tensor-parallel blocks an activation of B x S tokens is split along the sequence
// into N shards [N][B][S/N][h].  S = 0: the plain token-major [B*S][h] layout.
struct Sp {
  int S = 0, L = 0;
};
tpb::GemmOperand with_sp(tpb::GemmOperand o, Sp sp) {
  o.sp_S = sp.S;
  o.sp_L = sp.L;
  return o;
}
tpb::GemmExtra out_sp(Sp sp) {
  tpb::GemmExtra e;
  e.c_sp_S = sp.S;
  e.c_sp_L = sp.L;
  return e;
}

__global__ void k_timeout_probe(unsigned* err, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tpb::mbar_init(tpb::smem_u32(&bar), 1);
    abort_flag = 0;
    tpb::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const tpb::WaitCtx w{err, &abort_flag, timeout_ns};
    tpb::mbar_wait(tpb::smem_u32(&bar), 0, w);  // nothing arrives: runs out, latches kErrTimeout
  }
}

// Shape rules of the MLP block (bf16 needs 16-byte rows for TMA).
int mlp_shape_check(int dtype, int64_t T, int64_t h, int64_t f, int N) {
  if (dtype != TP_F32 && dtype != TP_BF16) return TP_ERR_DTYPE;
  if (T < 1 || h < 1 || f < 1 || N < 1) return TP_ERR_SHAPE;
  if (f % N) return TP_ERR_SHAPE;
  if (T > (1ll << 31) - 1 || h > (1ll << 31) - 1 || f > (1ll << 31) - 1) return TP_ERR_SHAPE;
  if (dtype == TP_BF16 && ((h % 8) || ((f / N) % 8))) return TP_ERR_SHAPE;
  return TP_OK;
}

// Shape rules of the attention block (H query heads, Hkv key/value heads).
int attn_shape_check(int dtype, int64_t B, int64_t S, int64_t h, int H, int Hkv, int d, int N) {
  if (dtype != TP_BF16) return TP_ERR_DTYPE;
  if (B < 1 || S < 1 || h < 1 || H < 1 || Hkv < 1 || d < 1 || N < 1) return TP_ERR_SHAPE;
  if (H % N || H % Hkv || Hkv % N) return TP_ERR_SHAPE;
  if (d != 64 && d != 128) return TP_ERR_SHAPE;
  if (h % 8) return TP_ERR_SHAPE;
  if (B > 65535 || H > 65535 || B * S > (1ll << 31) - 1 || h > (1ll << 31) - 1) return TP_ERR_SHAPE;
  return TP_OK;
}

// Workspace of the attention block: [QKV (fp16 Q, K, V) | O | LSE] in the
// forward; [dQKV | dO | Dsum | dS tiles] in the backward, the first three in the
// same regions.  The dS tiles (128 x 128 fp16 per query head, query block and key
// block) are sized for all block pairs, causal or not: the size queries take no
// mask flag.
struct AttnWs {
  size_t qkv, o, lse, ds, total;
};
AttnWs attn_ws(int64_t B, int64_t S, int H, int Hkv, int d) {
  const size_t T = static_cast<size_t>(B) * static_cast<size_t>(S);
  const size_t nb = (static_cast<size_t>(S) + 127) / 128;
  AttnWs w;
  w.qkv = round_up(T * (static_cast<size_t>(H) + 2 * static_cast<size_t>(Hkv)) * static_cast<size_t>(d) * 2, 256);
  w.o = round_up(T * static_cast<size_t>(H) * static_cast<size_t>(d) * 2, 256);
  w.lse = round_up(T * static_cast<size_t>(H) * 4, 256);
  w.ds = static_cast<size_t>(B) * static_cast<size_t>(H) * nb * nb * 128 * 128 * 2;
  w.total = w.qkv + w.o + w.lse + w.ds;
  return w;
}

}  // namespace

extern "C" {

int tp_version(void) { return (0 << 16) | 7; }

const char* tp_status_string(int s) {
  switch (s) {
    case TP_OK: return "ok";
    case TP_ERR_NULL: return "a required pointer is NULL";
    case TP_ERR_SHAPE: return "invalid shape (size < 1, N does not divide f or H, or row length not a multiple of 8)";
    case TP_ERR_DTYPE: return "dtype not supported by this call";
    case TP_ERR_WORKSPACE: return "workspace missing or too small";
    case TP_ERR_CUDA: return "CUDA error";
    case TP_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
    case TP_ERR_ALIGN: return "pointer not aligned (16 bytes; workspace 256 bytes)";
    case TP_ERR_DEVICE: return "current device is not an sm_103 GPU";
    case TP_ERR_BOUNDS: return "a debug build's device-side bounds or alignment check failed";
    default: return "unknown status";
  }
}

int tp_device_check(void) { return check_device(nullptr); }

int tp_sync_status(void* stream) {
  TP_TRACE;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TP_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tp_error_word, sizeof(v)) != cudaSuccess) return TP_ERR_CUDA;
  if (v) {
    const unsigned z = 0;
    if (cudaMemcpyToSymbol(g_tp_error_word, &z, sizeof(z)) != cudaSuccess) return TP_ERR_CUDA;
  }
  if (v & tpb::kErrTimeout) return TP_ERR_TIMEOUT;
  if (v & tpb::kErrBounds) return TP_ERR_BOUNDS;
  return TP_OK;
}

int tp_debug_timeout_probe(int64_t timeout_ns, void* stream) {
  TP_TRACE;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  if (timeout_ns < 1) return TP_ERR_SHAPE;
  const int slot = tpb::timing_begin(tpb::kKProbe, static_cast<cudaStream_t>(stream));
  k_timeout_probe<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, static_cast<unsigned long long>(timeout_ns));
  const bool ok = cudaGetLastError() == cudaSuccess;
  tpb::timing_end(slot, static_cast<cudaStream_t>(stream));
  return ok ? TP_OK : TP_ERR_CUDA;
}

}  // extern "C"

namespace {
// bf16 MLP forward kernels: a1 then a2.  With ``residual`` (a [T][h] tensor) the
// row-parallel GEMM's epilogue adds it: Z = residual + sum_i A_i W2_i.  With
// ``W1_16`` (an fp16 copy of W1s) X holds fp16 values and a1 is an fp16 product.
int mlp_fwd_seq(int64_t T, int64_t h, int64_t f, int N, const void* X, const void* W1s, const void* W2s,
                void* Y_save, void* Abuf, void* Z, const void* residual, unsigned* err, cudaStream_t st, Sp sp = Sp(),
                const void* W1_16 = nullptr, void* part_ws = nullptr, size_t part_bytes = 0) {
  const int64_t fN = f / N;
  // a1: Y_i = X W1_i, A_i = GeLU(Y_i)   (column-parallel, one group per shard; with
  // sequence-sharded X the copies gather the shards: the pages' all-gather g)
  const tpb::GemmOperand opX = with_sp(tpb::GemmOperand{X, h, T, 1, false, 0, 0}, sp);
  const tpb::GemmOperand opW1{W1_16 ? W1_16 : W1s, fN, h, N, true, 1, 0};
  tpb::GemmExtra e1;
  e1.ab_f16 = W1_16 != nullptr;
  int rc = tpb::launch_gemm_bf16(tpb::kEpiGelu, opX, opW1, Abuf, Y_save, Y_save != nullptr, T, fN, N, 1, h, err,
                                 kWaitTimeoutNs, st, tpb::kKMlpFc1, e1);
  if (rc) return gemm_status(rc);
  // a2: Z = sum_i A_i W2_i   (row-parallel, shards reduced in the accumulator, order 0..N-1)
  const tpb::GemmOperand opA{Abuf, fN, T, N, false, 0, 1};
  const tpb::GemmOperand opW2{W2s, h, fN, N, true, 0, 1};
  // (sequence-sharded Z: the stores scatter the summed rows to their shards, the
  // pages' reduce-scatter g*).  With ``part_ws`` a launch too small to fill the GPU
  // splits its K loop (the shards) in two halves added in fixed order.
  tpb::GemmExtra e2 = out_sp(sp);
  e2.part_ws = part_ws;
  e2.part_ws_bytes = part_bytes;
  rc = tpb::launch_gemm_bf16(residual ? tpb::kEpiResidual : tpb::kEpiStore, opA, opW2, Z, residual, false, T, h, 1,
                             N, fN, err, kWaitTimeoutNs, st, tpb::kKMlpFc2, e2);
  return gemm_status(rc);
}

tpb::AttnDims attn_dims(int64_t B, int64_t S, int H, int Hkv, int d, int N, int causal) {
  return tpb::AttnDims{static_cast<int>(B), static_cast<int>(S), H, H / N, N, d, causal ? 1 : 0, Hkv, Hkv / N};
}

// bf16 MLP backward kernels a3..a6 (dY in ``dY``, an activation-sized scratch).
// With sequence-sharded X, dZ and dX (``sp``) the GEMMs read and write those
// tensors in their shards.  With ``W1_16`` (an fp16 copy of W1s; X then holds
// fp16 values) dY is stored in fp16, dW1 and dX are fp16 products and dX is
// written in fp16.
int mlp_bwd_seq(int64_t T, int64_t h, int64_t f, int N, const void* X, const void* W1s, const void* W2s,
                const void* Y_save, const void* A_save, const void* dZ, void* dX, void* dW1s, void* dW2s, void* dY,
                unsigned* err, cudaStream_t st, Sp sp, const void* W1_16 = nullptr, void* part_ws = nullptr,
                size_t part_bytes = 0) {
  const int64_t fN = f / N;
  const bool h16 = W1_16 != nullptr;
  tpb::GemmExtra e16;
  e16.ab_f16 = h16;

  // a3: dY_i = (dZ W2_i^T) * GeLU'(Y_i)   (the row-split backward needs no reduction)
  const tpb::GemmOperand opdZk = with_sp(tpb::GemmOperand{dZ, h, T, 1, false, 0, 0}, sp);
  const tpb::GemmOperand opW2k{W2s, h, fN, N, false, 1, 0};
  tpb::GemmExtra e3;
  e3.c_f16 = h16;
  int rc = tpb::launch_gemm_bf16(tpb::kEpiDGelu, opdZk, opW2k, dY, Y_save, false, T, fN, N, 1, h, err,
                                 kWaitTimeoutNs, st, tpb::kKMlpDgelu, e3);
  if (rc) return gemm_status(rc);
  // a4: dW2_i = A_i^T dZ
  const tpb::GemmOperand opAt{A_save, fN, T, N, true, 1, 0};
  const tpb::GemmOperand opdZn = with_sp(tpb::GemmOperand{dZ, h, T, 1, true, 0, 0}, sp);
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opAt, opdZn, dW2s, nullptr, false, fN, h, N, 1, T, err, kWaitTimeoutNs,
                             st, tpb::kKMlpDw2);
  if (rc) return gemm_status(rc);
  // a5: dW1_i = X^T dY_i
  const tpb::GemmOperand opXt = with_sp(tpb::GemmOperand{X, h, T, 1, true, 0, 0}, sp);
  const tpb::GemmOperand opdYn{dY, fN, T, N, true, 1, 0};
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opXt, opdYn, dW1s, nullptr, false, h, fN, N, 1, T, err, kWaitTimeoutNs,
                             st, tpb::kKMlpDw1, e16);
  if (rc) return gemm_status(rc);
  // a6: dX = sum_i dY_i W1_i^T   (the column split's backward all-reduce, done in the accumulator)
  const tpb::GemmOperand opdYk{dY, fN, T, N, false, 0, 1};
  const tpb::GemmOperand opW1k{h16 ? W1_16 : W1s, fN, h, N, false, 0, 1};
  tpb::GemmExtra e6 = out_sp(sp);
  e6.ab_f16 = h16;
  e6.c_f16 = h16;
  e6.part_ws = part_ws;
  e6.part_ws_bytes = part_bytes;
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opdYk, opW1k, dX, nullptr, false, T, h, 1, N, fN, err, kWaitTimeoutNs,
                             st, tpb::kKMlpDx, e6);
  return gemm_status(rc);
}


// Attention forward kernels: a7, a8, a9 (H query heads, Hkv key/value heads).
// With ``residual`` ([T][h]) the output projection's epilogue adds it:
// Z = residual + sum_i O_i Wo_i.  With ``Wo16`` (an fp16 copy of Wo) O is stored
// in fp16 and a9 is an fp16 product; ``z_f16`` writes Z in fp16.  With ``Wqkv16``
// (an fp16 copy of Wqkv) X holds fp16 values and a7 is an fp16 product.
int attn_fwd_seq(int64_t B, int64_t S, int64_t h, int H, int Hkv, int d, int N, int causal, const void* X,
                 const void* Wqkv, const void* Wo, void* QKV, void* Ob, float* LSE, void* Z, const void* residual,
                 unsigned* err, cudaStream_t st, Sp sp = Sp(), const void* Wo16 = nullptr, bool z_f16 = false,
                 const void* Wqkv16 = nullptr) {
  tpb::AttnDims ad = attn_dims(B, S, H, Hkv, d, N, causal);
  ad.o_f16 = Wo16 != nullptr;
  const int64_t T = B * S, hNd = static_cast<int64_t>(ad.hN) * d, kvd = static_cast<int64_t>(ad.hkvN) * d;
  // a7: [Q_i K_i V_i] = X Wqkv_i  (column-parallel by head); Q, K and V stored fp16
  const tpb::GemmOperand opX = with_sp(tpb::GemmOperand{X, h, T, 1, false, 0, 0}, sp);
  const tpb::GemmOperand opW{Wqkv16 ? Wqkv16 : Wqkv, hNd + 2 * kvd, h, N, true, 1, 0};
  tpb::GemmExtra split;
  split.split_cols = hNd + 2 * kvd;
  split.ab_f16 = Wqkv16 != nullptr;
  int rc = tpb::launch_gemm_bf16(tpb::kEpiSplit, opX, opW, QKV, nullptr, false, T, hNd + 2 * kvd, N, 1, h, err,
                                 kWaitTimeoutNs, st, tpb::kKAttnQkv, split);
  if (rc) return gemm_status(rc);
  // a8: per-head causal attention
  rc = tpb::launch_attn_fwd(ad, QKV, Ob, LSE, err, kWaitTimeoutNs, st);
  if (rc) return gemm_status(rc);
  // a9: Z = sum_i O_i Wo_i  (row-parallel, shard sum in the accumulator)
  const tpb::GemmOperand opO{Ob, hNd, T, N, false, 0, 1};
  const tpb::GemmOperand opWo{Wo16 ? Wo16 : Wo, h, hNd, N, true, 0, 1};
  tpb::GemmExtra e9 = out_sp(sp);
  e9.ab_f16 = Wo16 != nullptr;
  e9.c_f16 = z_f16;
  rc = tpb::launch_gemm_bf16(residual ? tpb::kEpiResidual : tpb::kEpiStore, opO, opWo, Z, residual, false, T, h, 1,
                             N, hNd, err, kWaitTimeoutNs, st, tpb::kKAttnOut, e9);
  return gemm_status(rc);
}
// Attention backward kernels (scratch [dQKV | dO | Dsum] carved from ``wsb`` per
// ``w``).  With sequence-sharded X, dZ and dX (``sp``) the GEMMs read and write
// those tensors in their shards.  With ``Wo16`` (the fp16 copy of Wo the forward
// used) O and dZ hold fp16 values and dO, dWo are fp16 products.  With
// ``Wqkv16`` (the fp16 copy of Wqkv) X holds fp16 values: dQKV is stored in fp16,
// dWqkv and dX are fp16 products and dX is written in fp16.
int attn_bwd_seq(int64_t B, int64_t S, int64_t h, int H, int Hkv, int d, int N, int causal, const void* X,
                 const void* Wqkv, const void* Wo, const void* QKV_save, const void* O_save, const float* LSE_save,
                 const void* dZ, void* dX, void* dWqkv, void* dWo, char* wsb, const AttnWs& w, unsigned* err,
                 cudaStream_t st, Sp sp, const void* Wo16 = nullptr, const void* Wqkv16 = nullptr) {
  tpb::AttnDims ad = attn_dims(B, S, H, Hkv, d, N, causal);
  ad.o_f16 = Wo16 != nullptr;
  ad.dqkv_f16 = Wqkv16 != nullptr;
  tpb::GemmExtra eq;  // the products with X or Wqkv
  eq.ab_f16 = Wqkv16 != nullptr;
  const int64_t T = B * S, hNd = static_cast<int64_t>(ad.hN) * d, gw = ad.dqkv_width();
  void* dQKV = wsb;
  void* dO = wsb + w.qkv;
  float* dsum = reinterpret_cast<float*>(wsb + w.qkv + w.o);
  void* dsbuf = wsb + w.qkv + w.o + w.lse;

  // dO_i = dZ Wo_i^T   (row-parallel backward: every shard sees the whole dZ); fp16
  const tpb::GemmOperand opdZk = with_sp(tpb::GemmOperand{dZ, h, T, 1, false, 0, 0}, sp);
  const tpb::GemmOperand opWok{Wo16 ? Wo16 : Wo, h, hNd, N, false, 1, 0};
  tpb::GemmExtra edo;
  edo.ab_f16 = Wo16 != nullptr;
  edo.c_f16 = true;
  int rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opdZk, opWok, dO, nullptr, false, T, hNd, N, 1, h, err,
                                 kWaitTimeoutNs, st, tpb::kKAttnDo, edo);
  if (rc) return gemm_status(rc);
  // dWo_i = O_i^T dZ
  const tpb::GemmOperand opOt{O_save, hNd, T, N, true, 1, 0};
  const tpb::GemmOperand opdZn = with_sp(tpb::GemmOperand{dZ, h, T, 1, true, 0, 0}, sp);
  tpb::GemmExtra ewo;
  ewo.ab_f16 = Wo16 != nullptr;
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opOt, opdZn, dWo, nullptr, false, hNd, h, N, 1, T, err, kWaitTimeoutNs,
                             st, tpb::kKAttnDwo, ewo);
  if (rc) return gemm_status(rc);
  // attention core backward -> dQKV
  rc = tpb::launch_attn_bwd(ad, QKV_save, O_save, dO, LSE_save, dsum, dsbuf, dQKV, err, kWaitTimeoutNs, st);
  if (rc) return gemm_status(rc);
  // dWqkv_i = X^T dQKV_i
  const tpb::GemmOperand opXt = with_sp(tpb::GemmOperand{X, h, T, 1, true, 0, 0}, sp);
  const tpb::GemmOperand opdQn{dQKV, gw, T, N, true, 1, 0};
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opXt, opdQn, dWqkv, nullptr, false, h, gw, N, 1, T, err, kWaitTimeoutNs,
                             st, tpb::kKAttnDwqkv, eq);
  if (rc) return gemm_status(rc);
  // dX = sum_i dQKV_i Wqkv_i^T  (the column split's backward all-reduce, in the accumulator)
  const tpb::GemmOperand opdQk{dQKV, gw, T, N, false, 0, 1};
  const tpb::GemmOperand opWk{Wqkv16 ? Wqkv16 : Wqkv, gw, h, N, false, 0, 1};
  tpb::GemmExtra edx = out_sp(sp);
  edx.ab_f16 = eq.ab_f16;
  edx.c_f16 = eq.ab_f16;
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opdQk, opWk, dX, nullptr, false, T, h, 1, N, gw, err, kWaitTimeoutNs, st,
                             tpb::kKAttnDx, edx);
  return gemm_status(rc);
}

}  // namespace

extern "C" {

// ------------------------------------------------------------------ MLP block
}  // extern "C"

namespace {
// The MLP workspace: [A (forward, when not saved) or dY (backward) | split-K
// partials of the two row-parallel GEMMs (Z, dX), for shapes too small to fill
// the GPU otherwise].
size_t mlp_act_bytes(int dtype, int64_t T, int64_t f) {
  return round_up(static_cast<size_t>(T) * static_cast<size_t>(f) * (dtype == TP_F32 ? 4 : 2), 256);
}
size_t mlp_part_bytes(int dtype, int64_t T, int64_t h, int64_t f, int N) {
  return dtype == TP_BF16 ? round_up(tpb::gemm_splitk_bytes(T, h, 1, N, f / N), 256) : 0;
}
}  // namespace

extern "C" {

size_t tp_mlp_workspace_bytes(int dtype, int64_t T, int64_t h, int64_t f, int N) {
  if (mlp_shape_check(dtype, T, h, f, N) != TP_OK) return 0;
  return mlp_act_bytes(dtype, T, f) + mlp_part_bytes(dtype, T, h, f, N);
}

int tp_mlp_fwd(int dtype, int64_t T, int64_t h, int64_t f, int N, const void* X, const void* W1s,
               const void* W2s, void* Y_save, void* A_save, void* Z, void* ws, size_t ws_bytes, void* stream) {
  TP_TRACE;
  const int sc = mlp_shape_check(dtype, T, h, f, N);
  if (sc != TP_OK) return sc;
  if (!X || !W1s || !W2s || !Z) return TP_ERR_NULL;
  if (!al16(X) || !al16(W1s) || !al16(W2s) || !al16(Z) || !al16(Y_save) || !al16(A_save)) return TP_ERR_ALIGN;
  void* Abuf = A_save;
  if (!Abuf) {  // A in the workspace: at least its bytes
    if (!ws || ws_bytes < mlp_act_bytes(dtype, T, f)) return TP_ERR_WORKSPACE;
    if (!al256(ws)) return TP_ERR_ALIGN;
    Abuf = ws;
  }
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t fN = f / N;

  if (dtype == TP_F32) {
    tpb::SimtArgs a1{};
    a1.A = static_cast<const float*>(X);
    a1.B = static_cast<const float*>(W1s);
    a1.C = static_cast<float*>(Abuf);
    a1.Yout = static_cast<float*>(Y_save);
    a1.M = static_cast<int>(T);
    a1.N = static_cast<int>(fN);
    a1.K = static_cast<int>(h);
    a1.G = N;
    a1.S = 1;
    a1.b_sg = h * fN;
    a1.c_sg = T * fN;
    a1.lda = h;
    a1.ldb = fN;
    a1.ldc = fN;
    a1.gelu = 1;
    int rc = tpb::launch_gemm_f32(a1, st, tpb::kKMlpF32Fc1);
    if (rc) return gemm_status(rc);
    tpb::SimtArgs a2{};
    a2.A = static_cast<const float*>(Abuf);
    a2.B = static_cast<const float*>(W2s);
    a2.C = static_cast<float*>(Z);
    a2.M = static_cast<int>(T);
    a2.N = static_cast<int>(h);
    a2.K = static_cast<int>(fN);
    a2.G = 1;
    a2.S = N;
    a2.a_ss = T * fN;
    a2.b_ss = fN * h;
    a2.lda = fN;
    a2.ldb = h;
    a2.ldc = h;
    return gemm_status(tpb::launch_gemm_f32(a2, st, tpb::kKMlpF32Fc2));
  }

  // the partials region of the workspace, when the caller gave one that holds it
  void* part = nullptr;
  const size_t act = mlp_act_bytes(dtype, T, f), pb = mlp_part_bytes(dtype, T, h, f, N);
  if (pb && ws && al256(ws) && ws_bytes >= act + pb) part = static_cast<char*>(ws) + act;
  return mlp_fwd_seq(T, h, f, N, X, W1s, W2s, Y_save, Abuf, Z, nullptr, err, st, Sp(), nullptr, part, pb);
}

int tp_mlp_bwd(int dtype, int64_t T, int64_t h, int64_t f, int N, const void* X, const void* W1s,
               const void* W2s, const void* Y_save, const void* A_save, const void* dZ, void* dX, void* dW1s,
               void* dW2s, void* ws, size_t ws_bytes, void* stream) {
  TP_TRACE;
  const int sc = mlp_shape_check(dtype, T, h, f, N);
  if (sc != TP_OK) return sc;
  if (dtype != TP_BF16) return TP_ERR_DTYPE;
  if (!X || !W1s || !W2s || !Y_save || !A_save || !dZ || !dX || !dW1s || !dW2s) return TP_ERR_NULL;
  if (!al16(X) || !al16(W1s) || !al16(W2s) || !al16(Y_save) || !al16(A_save) || !al16(dZ) || !al16(dX) ||
      !al16(dW1s) || !al16(dW2s))
    return TP_ERR_ALIGN;
  if (!ws || ws_bytes < mlp_act_bytes(dtype, T, f)) return TP_ERR_WORKSPACE;  // dY
  if (!al256(ws)) return TP_ERR_ALIGN;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  // the split-K partials region, when the workspace holds it
  const size_t act = mlp_act_bytes(dtype, T, f), pb = mlp_part_bytes(dtype, T, h, f, N);
  void* part = (pb && ws_bytes >= act + pb) ? static_cast<char*>(ws) + act : nullptr;
  return mlp_bwd_seq(T, h, f, N, X, W1s, W2s, Y_save, A_save, dZ, dX, dW1s, dW2s, ws, err,
                     static_cast<cudaStream_t>(stream), Sp(), nullptr, part, pb);
}

}  // extern "C"

// ---------------------------------------------------------- gated MLP block
namespace {
int gmlp_shape_check(int dtype, int64_t T, int64_t h, int64_t f, int N) {
  if (dtype != TP_BF16) return TP_ERR_DTYPE;
  return mlp_shape_check(dtype, T, h, f, N);
}
}  // namespace

extern "C" {

size_t tp_gmlp_workspace_bytes(int dtype, int64_t T, int64_t h, int64_t f, int N) {
  if (gmlp_shape_check(dtype, T, h, f, N) != TP_OK) return 0;
  return round_up(static_cast<size_t>(T) * static_cast<size_t>(f) * 2 * 2, 256);
}

int tp_gmlp_fwd(int dtype, int64_t T, int64_t h, int64_t f, int N, const void* X, const void* Wgus,
                const void* Wds, void* GU_save, void* A_save, void* Z, void* ws, size_t ws_bytes, void* stream) {
  TP_TRACE;
  const int sc = gmlp_shape_check(dtype, T, h, f, N);
  if (sc != TP_OK) return sc;
  if (!X || !Wgus || !Wds || !Z) return TP_ERR_NULL;
  if (!al16(X) || !al16(Wgus) || !al16(Wds) || !al16(Z) || !al16(GU_save) || !al16(A_save)) return TP_ERR_ALIGN;
  void* Abuf = A_save;
  if (!Abuf) {
    if (!ws || ws_bytes < tp_gmlp_workspace_bytes(dtype, T, h, f, N)) return TP_ERR_WORKSPACE;
    if (!al256(ws)) return TP_ERR_ALIGN;
    Abuf = ws;
  }
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t fN = f / N;
  // [G_i U_i] = X [Wg_i Wu_i] in one product per shard; A_i = silu(G_i) * U_i in the epilogue
  const tpb::GemmOperand opX{X, h, T, 1, false, 0, 0};
  const tpb::GemmOperand opWgu{Wgus, fN, h, N, true, 1, 0, 2};
  int rc = tpb::launch_gemm_bf16(tpb::kEpiSwiGLU, opX, opWgu, Abuf, GU_save, GU_save != nullptr, T, fN, N, 1, h,
                                 err, kWaitTimeoutNs, st, tpb::kKGmlpFc1);
  if (rc) return gemm_status(rc);
  // Z = sum_i A_i Wd_i  (row-parallel, shard sum in the accumulator, order 0..N-1)
  const tpb::GemmOperand opA{Abuf, fN, T, N, false, 0, 1};
  const tpb::GemmOperand opWd{Wds, h, fN, N, true, 0, 1};
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opA, opWd, Z, nullptr, false, T, h, 1, N, fN, err, kWaitTimeoutNs, st,
                             tpb::kKGmlpFc2);
  return gemm_status(rc);
}

int tp_gmlp_bwd(int dtype, int64_t T, int64_t h, int64_t f, int N, const void* X, const void* Wgus,
                const void* Wds, const void* GU_save, const void* A_save, const void* dZ, void* dX, void* dWgus,
                void* dWds, void* ws, size_t ws_bytes, void* stream) {
  TP_TRACE;
  const int sc = gmlp_shape_check(dtype, T, h, f, N);
  if (sc != TP_OK) return sc;
  if (!X || !Wgus || !Wds || !GU_save || !A_save || !dZ || !dX || !dWgus || !dWds) return TP_ERR_NULL;
  if (!al16(X) || !al16(Wgus) || !al16(Wds) || !al16(GU_save) || !al16(A_save) || !al16(dZ) || !al16(dX) ||
      !al16(dWgus) || !al16(dWds))
    return TP_ERR_ALIGN;
  if (!ws || ws_bytes < tp_gmlp_workspace_bytes(dtype, T, h, f, N)) return TP_ERR_WORKSPACE;
  if (!al256(ws)) return TP_ERR_ALIGN;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t fN = f / N;
  void* dGU = ws;  // [N][T][2][f/N]

  // dA_i = dZ Wd_i^T; epilogue: dG_i = dA_i * U_i * silu'(G_i), dU_i = dA_i * silu(G_i)
  const tpb::GemmOperand opdZk{dZ, h, T, 1, false, 0, 0};
  const tpb::GemmOperand opWdk{Wds, h, fN, N, false, 1, 0};
  int rc = tpb::launch_gemm_bf16(tpb::kEpiDSwiGLU, opdZk, opWdk, dGU, GU_save, false, T, fN, N, 1, h, err,
                                 kWaitTimeoutNs, st, tpb::kKGmlpDswiglu);
  if (rc) return gemm_status(rc);
  // dWd_i = A_i^T dZ
  const tpb::GemmOperand opAt{A_save, fN, T, N, true, 1, 0};
  const tpb::GemmOperand opdZn{dZ, h, T, 1, true, 0, 0};
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opAt, opdZn, dWds, nullptr, false, fN, h, N, 1, T, err, kWaitTimeoutNs,
                             st, tpb::kKGmlpDwd);
  if (rc) return gemm_status(rc);
  // [dWg_i dWu_i] = X^T [dG_i dU_i]  (one product per shard over the fused columns)
  const tpb::GemmOperand opXt{X, h, T, 1, true, 0, 0};
  const tpb::GemmOperand opdGUn{dGU, 2 * fN, T, N, true, 1, 0};
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opXt, opdGUn, dWgus, nullptr, false, h, 2 * fN, N, 1, T, err,
                             kWaitTimeoutNs, st, tpb::kKGmlpDwgu);
  if (rc) return gemm_status(rc);
  // dX = sum_i [dG_i dU_i] [Wg_i Wu_i]^T  (the column split's backward all-reduce, in the accumulator)
  const tpb::GemmOperand opdGUk{dGU, 2 * fN, T, N, false, 0, 1};
  const tpb::GemmOperand opWguk{Wgus, 2 * fN, h, N, false, 0, 1};
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opdGUk, opWguk, dX, nullptr, false, T, h, 1, N, 2 * fN, err,
                             kWaitTimeoutNs, st, tpb::kKGmlpDx);
  return gemm_status(rc);
}

}  // extern "C"

// ------------------------------------------------------------ attention block
extern "C" {

size_t tp_gqa_workspace_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int Hkv, int d, int N) {
  if (attn_shape_check(dtype, B, S, h, H, Hkv, d, N) != TP_OK) return 0;
  return attn_ws(B, S, H, Hkv, d).total;
}

size_t tp_attn_workspace_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int N) {
  return tp_gqa_workspace_bytes(dtype, B, S, h, H, H, d, N);
}

int tp_gqa_fwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int Hkv, int d, int N, int causal, const void* X,
               const void* Wqkv, const void* Wo, void* QKV_save, void* O_save, float* LSE_save, void* Z, void* ws,
               size_t ws_bytes, void* stream) {
  TP_TRACE;
  const int sc = attn_shape_check(dtype, B, S, h, H, Hkv, d, N);
  if (sc != TP_OK) return sc;
  if (!X || !Wqkv || !Wo || !Z) return TP_ERR_NULL;
  if (!al16(X) || !al16(Wqkv) || !al16(Wo) || !al16(Z) || !al16(QKV_save) || !al16(O_save) || !al16(LSE_save))
    return TP_ERR_ALIGN;
  const AttnWs w = attn_ws(B, S, H, Hkv, d);
  char* wsb = static_cast<char*>(ws);
  if (!QKV_save || !O_save || !LSE_save) {
    if (!ws || ws_bytes < w.total) return TP_ERR_WORKSPACE;
    if (!al256(ws)) return TP_ERR_ALIGN;
  }
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* QKV = QKV_save ? QKV_save : static_cast<void*>(wsb);
  void* Ob = O_save ? O_save : static_cast<void*>(wsb + w.qkv);
  float* LSE = LSE_save ? LSE_save : reinterpret_cast<float*>(wsb + w.qkv + w.o);
  return attn_fwd_seq(B, S, h, H, Hkv, d, N, causal, X, Wqkv, Wo, QKV, Ob, LSE, Z, nullptr, err, st);
}

int tp_attn_fwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int N, int causal, const void* X,
                const void* Wqkv, const void* Wo, void* QKV_save, void* O_save, float* LSE_save, void* Z, void* ws,
                size_t ws_bytes, void* stream) {
  TP_TRACE;
  return tp_gqa_fwd(dtype, B, S, h, H, H, d, N, causal, X, Wqkv, Wo, QKV_save, O_save, LSE_save, Z, ws, ws_bytes,
                    stream);
}

int tp_gqa_bwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int Hkv, int d, int N, int causal, const void* X,
               const void* Wqkv, const void* Wo, const void* QKV_save, const void* O_save, const float* LSE_save,
               const void* dZ, void* dX, void* dWqkv, void* dWo, void* ws, size_t ws_bytes, void* stream) {
  TP_TRACE;
  const int sc = attn_shape_check(dtype, B, S, h, H, Hkv, d, N);
  if (sc != TP_OK) return sc;
  if (!X || !Wqkv || !Wo || !QKV_save || !O_save || !LSE_save || !dZ || !dX || !dWqkv || !dWo) return TP_ERR_NULL;
  if (!al16(X) || !al16(Wqkv) || !al16(Wo) || !al16(QKV_save) || !al16(O_save) || !al16(LSE_save) || !al16(dZ) ||
      !al16(dX) || !al16(dWqkv) || !al16(dWo))
    return TP_ERR_ALIGN;
  const AttnWs w = attn_ws(B, S, H, Hkv, d);
  if (!ws || ws_bytes < w.total) return TP_ERR_WORKSPACE;
  if (!al256(ws)) return TP_ERR_ALIGN;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  return attn_bwd_seq(B, S, h, H, Hkv, d, N, causal, X, Wqkv, Wo, QKV_save, O_save, LSE_save, dZ, dX, dWqkv, dWo,
                      static_cast<char*>(ws), w, err, static_cast<cudaStream_t>(stream), Sp());
}

int tp_attn_bwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int N, int causal, const void* X,
                const void* Wqkv, const void* Wo, const void* QKV_save, const void* O_save, const float* LSE_save,
                const void* dZ, void* dX, void* dWqkv, void* dWo, void* ws, size_t ws_bytes, void* stream) {
  TP_TRACE;
  return tp_gqa_bwd(dtype, B, S, h, H, H, d, N, causal, X, Wqkv, Wo, QKV_save, O_save, LSE_save, dZ, dX, dWqkv, dWo,
                    ws, ws_bytes, stream);
}

}  // extern "C"

// ------------------------------------------- attention block then MLP block
namespace {
// The saved tensors of tp_attn_mlp_fwd, carved from the caller's ``save`` buffer
// in this order (each region 256-byte aligned): the attention block's QKV (fp16),
// O (fp16) and LSE; the fp16 copy of Wo; the block output H (fp16), which is the
// MLP's input; the fp16 copy of W1s; the MLP's Y and A (bf16).
struct AmSave {
  size_t qkv, o, lse, wo16, h16, w1_16, y, a, total;
};
AmSave am_save(int64_t B, int64_t S, int64_t h, int H, int d, int64_t f) {
  const size_t T = static_cast<size_t>(B) * static_cast<size_t>(S);
  const AttnWs aw = attn_ws(B, S, H, H, d);
  const size_t hs = static_cast<size_t>(h), fs = static_cast<size_t>(f), hd = static_cast<size_t>(H) * d;
  AmSave L;
  size_t o = 0;
  L.qkv = o;   o += aw.qkv;
  L.o = o;     o += aw.o;
  L.lse = o;   o += aw.lse;
  L.wo16 = o;  o += round_up(hd * hs * 2, 256);
  L.h16 = o;   o += round_up(T * hs * 2, 256);
  L.w1_16 = o; o += round_up(hs * fs * 2, 256);
  L.y = o;     o += round_up(T * fs * 2, 256);
  L.a = o;     o += round_up(T * fs * 2, 256);
  L.total = o;
  return L;
}
// Backward scratch: [block scratch (the MLP's dY, then the attention block's
// dQKV | dO | Dsum) | dH (fp16)].
struct AmWs {
  size_t blk, dh, total;
};
AmWs am_ws(int64_t B, int64_t S, int64_t h, int H, int d, int64_t f) {
  const size_t T = static_cast<size_t>(B) * static_cast<size_t>(S);
  const size_t a = attn_ws(B, S, H, H, d).total, m = round_up(T * static_cast<size_t>(f) * 2, 256);
  AmWs w;
  w.blk = 0;
  w.dh = a > m ? a : m;
  w.total = w.dh + round_up(T * static_cast<size_t>(h) * 2, 256);
  return w;
}
int am_check(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N) {
  const int c = attn_shape_check(dtype, B, S, h, H, H, d, N);
  return c != TP_OK ? c : mlp_shape_check(dtype, B * S, h, f, N);
}
}  // namespace

extern "C" {

size_t tp_attn_mlp_save_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N) {
  if (am_check(dtype, B, S, h, H, d, f, N) != TP_OK) return 0;
  return am_save(B, S, h, H, d, f).total;
}

size_t tp_attn_mlp_workspace_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N) {
  if (am_check(dtype, B, S, h, H, d, f, N) != TP_OK) return 0;
  return am_ws(B, S, h, H, d, f).total;
}

int tp_attn_mlp_fwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N, int causal,
                    const void* X, const void* Wqkv, const void* Wo, const void* W1s, const void* W2s, void* save,
                    size_t save_bytes, void* Z, void* stream) {
  TP_TRACE;
  const int sc = am_check(dtype, B, S, h, H, d, f, N);
  if (sc != TP_OK) return sc;
  if (!X || !Wqkv || !Wo || !W1s || !W2s || !save || !Z) return TP_ERR_NULL;
  if (!al16(X) || !al16(Wqkv) || !al16(Wo) || !al16(W1s) || !al16(W2s) || !al16(Z)) return TP_ERR_ALIGN;
  const AmSave L = am_save(B, S, h, H, d, f);
  if (save_bytes < L.total) return TP_ERR_WORKSPACE;
  if (!al256(save)) return TP_ERR_ALIGN;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* sv = static_cast<char*>(save);
  // fp16 copies of the two weights whose other operand is an fp16 activation
  int rc = tpb::launch_bf16_to_f16(Wo, sv + L.wo16, static_cast<long long>(H) * d * h, st);
  if (rc) return gemm_status(rc);
  rc = tpb::launch_bf16_to_f16(W1s, sv + L.w1_16, static_cast<long long>(h) * f, st);
  if (rc) return gemm_status(rc);
  // H = Attn(X), written in fp16
  rc = attn_fwd_seq(B, S, h, H, H, d, N, causal, X, Wqkv, Wo, sv + L.qkv, sv + L.o,
                    reinterpret_cast<float*>(sv + L.lse), sv + L.h16, nullptr, err, st, Sp(), sv + L.wo16, true);
  if (rc) return rc;
  // Z = MLP(H)
  return mlp_fwd_seq(B * S, h, f, N, sv + L.h16, W1s, W2s, sv + L.y, sv + L.a, Z, nullptr, err, st, Sp(),
                     sv + L.w1_16);
}

int tp_attn_mlp_bwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N, int causal,
                    const void* X, const void* Wqkv, const void* Wo, const void* W1s, const void* W2s,
                    const void* save, size_t save_bytes, const void* dZ, void* dX, void* dWqkv, void* dWo,
                    void* dW1s, void* dW2s, void* ws, size_t ws_bytes, void* stream) {
  TP_TRACE;
  const int sc = am_check(dtype, B, S, h, H, d, f, N);
  if (sc != TP_OK) return sc;
  if (!X || !Wqkv || !Wo || !W1s || !W2s || !save || !dZ || !dX || !dWqkv || !dWo || !dW1s || !dW2s)
    return TP_ERR_NULL;
  if (!al16(X) || !al16(Wqkv) || !al16(Wo) || !al16(W1s) || !al16(W2s) || !al16(dZ) || !al16(dX) || !al16(dWqkv) ||
      !al16(dWo) || !al16(dW1s) || !al16(dW2s))
    return TP_ERR_ALIGN;
  const AmSave L = am_save(B, S, h, H, d, f);
  const AmWs W = am_ws(B, S, h, H, d, f);
  if (save_bytes < L.total || !ws || ws_bytes < W.total) return TP_ERR_WORKSPACE;
  if (!al256(save) || !al256(ws)) return TP_ERR_ALIGN;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* sv = static_cast<const char*>(save);
  char* wb = static_cast<char*>(ws);
  // MLP block backward on H: dH (fp16) and the MLP's weight gradients
  int rc = mlp_bwd_seq(B * S, h, f, N, sv + L.h16, W1s, W2s, sv + L.y, sv + L.a, dZ, wb + W.dh, dW1s, dW2s,
                       wb + W.blk, err, st, Sp(), sv + L.w1_16);
  if (rc) return rc;
  // attention block backward with upstream dH
  return attn_bwd_seq(B, S, h, H, H, d, N, causal, X, Wqkv, Wo, sv + L.qkv, sv + L.o,
                      reinterpret_cast<const float*>(sv + L.lse), wb + W.dh, dX, dWqkv, dWo, wb + W.blk,
                      attn_ws(B, S, H, H, d), err, st, Sp(), sv + L.wo16);
}

}  // extern "C"

// ------------------------------------------------------ LayerNorm + residual
namespace {
constexpr float kEpsMin = 0.0f;

// The pre-norm layer's saved tensors, carved from the caller's ``save`` buffer in
// this order (each region 256-byte aligned): LN1(X) (fp16) and its statistics;
// the attention block's QKV, O (fp16) and LSE; H1 (bf16); LN2(H1) (fp16) and its
// statistics; the MLP's Y and A (bf16); the fp16 copies of Wqkv, Wo and W1s.
struct LayerSave {
  size_t ln1, mean1, rstd1, qkv, o, lse, h1, ln2, mean2, rstd2, y, a, wqkv16, wo16, w1_16, total;
};
LayerSave layer_save(int64_t B, int64_t S, int64_t h, int H, int d, int64_t f) {
  const size_t T = static_cast<size_t>(B) * static_cast<size_t>(S);
  const size_t th = round_up(T * static_cast<size_t>(h) * 2, 256), tv = round_up(T * 4, 256);
  const size_t hd = static_cast<size_t>(H) * static_cast<size_t>(d), hs = static_cast<size_t>(h);
  const AttnWs aw = attn_ws(B, S, H, H, d);
  LayerSave L;
  size_t o = 0;
  L.ln1 = o;   o += th;
  L.mean1 = o; o += tv;
  L.rstd1 = o; o += tv;
  L.qkv = o;   o += aw.qkv;
  L.o = o;     o += aw.o;
  L.lse = o;   o += aw.lse;
  L.h1 = o;    o += th;
  L.ln2 = o;   o += th;
  L.mean2 = o; o += tv;
  L.rstd2 = o; o += tv;
  L.y = o;     o += round_up(T * static_cast<size_t>(f) * 2, 256);
  L.a = o;     o += round_up(T * static_cast<size_t>(f) * 2, 256);
  L.wqkv16 = o; o += round_up(hs * 3 * hd * 2, 256);
  L.wo16 = o;   o += round_up(hd * hs * 2, 256);
  L.w1_16 = o;  o += round_up(hs * static_cast<size_t>(f) * 2, 256);
  L.total = o;
  return L;
}

// Backward scratch: [block scratch (attention or MLP, used in turn) | dLN | dH1 | LN partials].
struct LayerWs {
  size_t blk, dln, dh1, part, total;
};
LayerWs layer_ws(int64_t B, int64_t S, int64_t h, int H, int d, int64_t f) {
  const size_t T = static_cast<size_t>(B) * static_cast<size_t>(S);
  const size_t th = round_up(T * static_cast<size_t>(h) * 2, 256);
  const size_t a = attn_ws(B, S, H, H, d).total, m = round_up(T * static_cast<size_t>(f) * 2, 256);
  LayerWs w;
  w.blk = 0;
  w.dln = a > m ? a : m;
  w.dh1 = w.dln + th;
  w.part = w.dh1 + th;
  w.total = w.part + round_up(tpb::ln_partial_bytes(static_cast<int64_t>(T), h), 256);
  return w;
}

int layer_check(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N) {
  int c = attn_shape_check(dtype, B, S, h, H, H, d, N);
  if (c != TP_OK) return c;
  c = mlp_shape_check(dtype, B * S, h, f, N);
  if (c != TP_OK) return c;
  return tpb::ln_shape_ok(B * S, h) ? TP_OK : TP_ERR_SHAPE;
}
}  // namespace

extern "C" {

size_t tp_layernorm_workspace_bytes(int dtype, int64_t T, int64_t h) {
  if (dtype != TP_BF16 || !tpb::ln_shape_ok(T, h)) return 0;
  return round_up(tpb::ln_partial_bytes(T, h), 256);
}

int tp_layernorm_fwd(int dtype, int64_t T, int64_t h, float eps, const void* X, const void* gamma, const void* beta,
                     void* Y, float* mean, float* rstd, void* stream) {
  TP_TRACE;
  if (dtype != TP_BF16) return TP_ERR_DTYPE;
  if (!tpb::ln_shape_ok(T, h) || !(eps >= kEpsMin)) return TP_ERR_SHAPE;
  if (!X || !gamma || !beta || !Y || !mean || !rstd) return TP_ERR_NULL;
  if (!al16(X) || !al16(gamma) || !al16(beta) || !al16(Y) || !al16(mean) || !al16(rstd)) return TP_ERR_ALIGN;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  return gemm_status(
      tpb::launch_ln_fwd(X, gamma, beta, Y, mean, rstd, T, h, eps, static_cast<cudaStream_t>(stream), 0, err));
}

int tp_layernorm_bwd(int dtype, int64_t T, int64_t h, const void* X, const void* gamma, const float* mean,
                     const float* rstd, const void* dY, const void* dR, void* dX, void* dgamma, void* dbeta, void* ws,
                     size_t ws_bytes, void* stream) {
  TP_TRACE;
  if (dtype != TP_BF16) return TP_ERR_DTYPE;
  if (!tpb::ln_shape_ok(T, h)) return TP_ERR_SHAPE;
  if (!X || !gamma || !mean || !rstd || !dY || !dX || !dgamma || !dbeta) return TP_ERR_NULL;
  if (!al16(X) || !al16(gamma) || !al16(mean) || !al16(rstd) || !al16(dY) || !al16(dR) || !al16(dX) ||
      !al16(dgamma) || !al16(dbeta))
    return TP_ERR_ALIGN;
  if (!ws || ws_bytes < tp_layernorm_workspace_bytes(dtype, T, h)) return TP_ERR_WORKSPACE;
  if (!al256(ws)) return TP_ERR_ALIGN;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  return gemm_status(tpb::launch_ln_bwd(X, gamma, mean, rstd, dY, dR, dX, dgamma, dbeta, static_cast<float*>(ws), T,
                                        h, static_cast<cudaStream_t>(stream), 0, err));
}

size_t tp_layer_save_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N) {
  if (layer_check(dtype, B, S, h, H, d, f, N) != TP_OK) return 0;
  return layer_save(B, S, h, H, d, f).total;
}

size_t tp_layer_workspace_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N) {
  if (layer_check(dtype, B, S, h, H, d, f, N) != TP_OK) return 0;
  return layer_ws(B, S, h, H, d, f).total;
}

}  // extern "C"

namespace {
// The pre-norm layer's forward and backward kernel sequences; ``sp`` selects
// sequence-sharded X, Z, dZ, dX (and the saved LN outputs and H1, which stay in
// the same row order).
int layer_fwd_impl(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N, int causal, float eps,
                   const void* X, const void* ln1_g, const void* ln1_b, const void* Wqkv, const void* Wo,
                   const void* ln2_g, const void* ln2_b, const void* W1s, const void* W2s, void* save,
                   size_t save_bytes, void* Z, void* stream, Sp sp) {
  const int sc = layer_check(dtype, B, S, h, H, d, f, N);
  if (sc != TP_OK) return sc;
  if (!(eps >= kEpsMin)) return TP_ERR_SHAPE;
  if (!X || !ln1_g || !ln1_b || !Wqkv || !Wo || !ln2_g || !ln2_b || !W1s || !W2s || !save || !Z) return TP_ERR_NULL;
  if (!al16(X) || !al16(ln1_g) || !al16(ln1_b) || !al16(Wqkv) || !al16(Wo) || !al16(ln2_g) || !al16(ln2_b) ||
      !al16(W1s) || !al16(W2s) || !al16(Z))
    return TP_ERR_ALIGN;
  const LayerSave L = layer_save(B, S, h, H, d, f);
  if (save_bytes < L.total) return TP_ERR_WORKSPACE;
  if (!al256(save)) return TP_ERR_ALIGN;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* sv = static_cast<char*>(save);
  const int64_t T = B * S;
  float* mean1 = reinterpret_cast<float*>(sv + L.mean1);
  float* rstd1 = reinterpret_cast<float*>(sv + L.rstd1);
  float* mean2 = reinterpret_cast<float*>(sv + L.mean2);
  float* rstd2 = reinterpret_cast<float*>(sv + L.rstd2);
  // fp16 copies of the weights whose other operand is an fp16 activation
  int rc = tpb::launch_bf16_to_f16(Wqkv, sv + L.wqkv16, static_cast<long long>(h) * 3 * H * d, st);
  if (!rc) rc = tpb::launch_bf16_to_f16(Wo, sv + L.wo16, static_cast<long long>(H) * d * h, st);
  if (!rc) rc = tpb::launch_bf16_to_f16(W1s, sv + L.w1_16, static_cast<long long>(h) * f, st);
  if (rc) return gemm_status(rc);
  // LN1(X) in fp16 (row by row, so in whatever row order X is stored)
  rc = tpb::launch_ln_fwd(X, ln1_g, ln1_b, sv + L.ln1, mean1, rstd1, T, h, eps, st, tpb::kLnYF16, err);
  if (rc) return gemm_status(rc);
  // H1 = X + Attn(LN1(X)): the residual is added in the output projection's epilogue
  rc = attn_fwd_seq(B, S, h, H, H, d, N, causal, sv + L.ln1, Wqkv, Wo, sv + L.qkv, sv + L.o,
                    reinterpret_cast<float*>(sv + L.lse), sv + L.h1, X, err, st, sp, sv + L.wo16, false,
                    sv + L.wqkv16);
  if (rc) return rc;
  // LN2(H1) in fp16
  rc = tpb::launch_ln_fwd(sv + L.h1, ln2_g, ln2_b, sv + L.ln2, mean2, rstd2, T, h, eps, st, tpb::kLnYF16, err);
  if (rc) return gemm_status(rc);
  // Z = H1 + MLP(LN2(H1)): the residual is added in the second GEMM's epilogue
  return mlp_fwd_seq(T, h, f, N, sv + L.ln2, W1s, W2s, sv + L.y, sv + L.a, Z, sv + L.h1, err, st, sp, sv + L.w1_16);
}

int layer_bwd_impl(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N, int causal,
                   const void* X, const void* ln1_g, const void* Wqkv, const void* Wo, const void* ln2_g,
                   const void* W1s, const void* W2s, const void* save, size_t save_bytes, const void* dZ, void* dX,
                   void* dln1_g, void* dln1_b, void* dWqkv, void* dWo, void* dln2_g, void* dln2_b, void* dW1s,
                   void* dW2s, void* ws, size_t ws_bytes, void* stream, Sp sp) {
  const int sc = layer_check(dtype, B, S, h, H, d, f, N);
  if (sc != TP_OK) return sc;
  if (!X || !ln1_g || !Wqkv || !Wo || !ln2_g || !W1s || !W2s || !save || !dZ || !dX || !dln1_g || !dln1_b ||
      !dWqkv || !dWo || !dln2_g || !dln2_b || !dW1s || !dW2s)
    return TP_ERR_NULL;
  if (!al16(X) || !al16(ln1_g) || !al16(Wqkv) || !al16(Wo) || !al16(ln2_g) || !al16(W1s) || !al16(W2s) ||
      !al16(dZ) || !al16(dX) || !al16(dln1_g) || !al16(dln1_b) || !al16(dWqkv) || !al16(dWo) || !al16(dln2_g) ||
      !al16(dln2_b) || !al16(dW1s) || !al16(dW2s))
    return TP_ERR_ALIGN;
  const LayerSave L = layer_save(B, S, h, H, d, f);
  const LayerWs W = layer_ws(B, S, h, H, d, f);
  if (save_bytes < L.total || !ws || ws_bytes < W.total) return TP_ERR_WORKSPACE;
  if (!al256(save) || !al256(ws)) return TP_ERR_ALIGN;
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  const char* sv = static_cast<const char*>(save);
  char* wb = static_cast<char*>(ws);
  const int64_t T = B * S;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* dLN = wb + W.dln;
  void* dH1 = wb + W.dh1;
  float* part = reinterpret_cast<float*>(wb + W.part);
  // MLP block backward on LN2(H1): dLN2 -> dLN (fp16; dY in the block scratch)
  int rc = mlp_bwd_seq(T, h, f, N, sv + L.ln2, W1s, W2s, sv + L.y, sv + L.a, dZ, dLN, dW1s, dW2s, wb + W.blk, err, st,
                       sp, sv + L.w1_16);
  if (rc) return rc;
  // dH1 = dZ + LN2'(dLN2)   (the residual passes dZ through); fp16
  rc = tpb::launch_ln_bwd(sv + L.h1, ln2_g, reinterpret_cast<const float*>(sv + L.mean2),
                          reinterpret_cast<const float*>(sv + L.rstd2), dLN, dZ, dH1, dln2_g, dln2_b, part, T, h, st,
                          tpb::kLnDyF16 | tpb::kLnDxF16, err);
  if (rc) return gemm_status(rc);
  // attention block backward on LN1(X) with upstream dH1: dLN1 -> dLN (fp16)
  rc = attn_bwd_seq(B, S, h, H, H, d, N, causal, sv + L.ln1, Wqkv, Wo, sv + L.qkv, sv + L.o,
                    reinterpret_cast<const float*>(sv + L.lse), dH1, dLN, dWqkv, dWo, wb + W.blk, attn_ws(B, S, H, H, d),
                    err, st, sp, sv + L.wo16, sv + L.wqkv16);
  if (rc) return rc;
  // dX = dH1 + LN1'(dLN1)
  rc = tpb::launch_ln_bwd(X, ln1_g, reinterpret_cast<const float*>(sv + L.mean1),
                          reinterpret_cast<const float*>(sv + L.rstd1), dLN, dH1, dX, dln1_g, dln1_b, part, T, h, st,
                          tpb::kLnDyF16 | tpb::kLnDrF16, err);
  return gemm_status(rc);
}

// The sequence split of the layer: N shards of S/N tokens per sequence, each a
// multiple of 128 so that no tile of a GEMM spans two shards.
int sp_of(int64_t S, int N, Sp* sp) {
  if (N < 1 || S % N || (S / N) % 128) return TP_ERR_SHAPE;
  sp->S = static_cast<int>(S);
  sp->L = static_cast<int>(S / N);
  return TP_OK;
}
}  // namespace

extern "C" {

int tp_layer_fwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N, int causal, float eps,
                 const void* X, const void* ln1_g, const void* ln1_b, const void* Wqkv, const void* Wo,
                 const void* ln2_g, const void* ln2_b, const void* W1s, const void* W2s, void* save,
                 size_t save_bytes, void* Z, void* stream) {
  TP_TRACE;
  return layer_fwd_impl(dtype, B, S, h, H, d, f, N, causal, eps, X, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s,
                        save, save_bytes, Z, stream, Sp());
}

int tp_layer_bwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N, int causal,
                 const void* X, const void* ln1_g, const void* Wqkv, const void* Wo, const void* ln2_g,
                 const void* W1s, const void* W2s, const void* save, size_t save_bytes, const void* dZ, void* dX,
                 void* dln1_g, void* dln1_b, void* dWqkv, void* dWo, void* dln2_g, void* dln2_b, void* dW1s,
                 void* dW2s, void* ws, size_t ws_bytes, void* stream) {
  TP_TRACE;
  return layer_bwd_impl(dtype, B, S, h, H, d, f, N, causal, X, ln1_g, Wqkv, Wo, ln2_g, W1s, W2s, save, save_bytes,
                        dZ, dX, dln1_g, dln1_b, dWqkv, dWo, dln2_g, dln2_b, dW1s, dW2s, ws, ws_bytes, stream, Sp());
}

int tp_sp_layer_fwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N, int causal,
                    float eps, const void* X, const void* ln1_g, const void* ln1_b, const void* Wqkv, const void* Wo,
                    const void* ln2_g, const void* ln2_b, const void* W1s, const void* W2s, void* save,
                    size_t save_bytes, void* Z, void* stream) {
  TP_TRACE;
  Sp sp;
  const int sc = layer_check(dtype, B, S, h, H, d, f, N);
  if (sc != TP_OK) return sc;
  if (sp_of(S, N, &sp) != TP_OK) return TP_ERR_SHAPE;
  return layer_fwd_impl(dtype, B, S, h, H, d, f, N, causal, eps, X, ln1_g, ln1_b, Wqkv, Wo, ln2_g, ln2_b, W1s, W2s,
                        save, save_bytes, Z, stream, sp);
}

int tp_sp_layer_bwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N, int causal,
                    const void* X, const void* ln1_g, const void* Wqkv, const void* Wo, const void* ln2_g,
                    const void* W1s, const void* W2s, const void* save, size_t save_bytes, const void* dZ, void* dX,
                    void* dln1_g, void* dln1_b, void* dWqkv, void* dWo, void* dln2_g, void* dln2_b, void* dW1s,
                    void* dW2s, void* ws, size_t ws_bytes, void* stream) {
  TP_TRACE;
  Sp sp;
  const int sc = layer_check(dtype, B, S, h, H, d, f, N);
  if (sc != TP_OK) return sc;
  if (sp_of(S, N, &sp) != TP_OK) return TP_ERR_SHAPE;
  return layer_bwd_impl(dtype, B, S, h, H, d, f, N, causal, X, ln1_g, Wqkv, Wo, ln2_g, W1s, W2s, save, save_bytes,
                        dZ, dX, dln1_g, dln1_b, dWqkv, dWo, dln2_g, dln2_b, dW1s, dW2s, ws, ws_bytes, stream, sp);
}

}  // extern "C"

// ------------------------------------------------------------ kernel timing
extern "C" {

int tp_set_gemm_tiling(int mode) {
  return tpb::set_gemm_tiling_mode(mode) ? TP_OK : TP_ERR_SHAPE;
}

int tp_set_launch_overlap(int on) {
  if (on != 0 && on != 1) return TP_ERR_SHAPE;
  tpb::set_launch_overlap(on != 0);
  return TP_OK;
}

int tp_timing_enable(int on) {
  tpb::timing_enable(on != 0);
  return TP_OK;
}

int tp_timing_kinds(void) { return tpb::kNumKernelKinds; }

const char* tp_timing_name(int kind) { return tpb::kernel_kind_name(kind); }

int tp_timing_read(int kind, int64_t* launches, double* total_ms) {
  if (kind < 0 || kind >= tpb::kNumKernelKinds) return TP_ERR_SHAPE;
  long long n = 0;
  double t = 0.0;
  if (!tpb::timing_read(kind, &n, &t)) return TP_ERR_CUDA;
  if (launches) *launches = n;
  if (total_ms) *total_ms = t;
  return TP_OK;
}

}  // extern "C"

// ------------------------------------------------- MLP forward without allocation
// A fixed scratch array in device memory for callers that may not allocate: the
// activation A of tp_mlp_fwd_noalloc lives here instead of in a caller's
// workspace.  Every GPU that loads the library holds these bytes until exit.
static __device__ __align__(256) unsigned char g_tp_noalloc_scratch[TP_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDev];  // device address of the array, per device (set up on first use)

// The array's name is only a host-side stand-in in host code; its device address
// comes from the runtime, once per device, with that device current.
int noalloc_scratch(void** out) {
  const int d = current_device();
  if (d < 0) return TP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tp_noalloc_scratch) != cudaSuccess || !p) return TP_ERR_CUDA;
    g_noalloc_ptr[d] = p;
  }
  *out = g_noalloc_ptr[d];
  return TP_OK;
}
}  // namespace

extern "C" {

int tp_mlp_fwd_noalloc(int dtype, int64_t T, int64_t h, int64_t f, int N, const void* X, const void* W1s,
                       const void* W2s, void* Z, void* stream) {
  TP_TRACE;
  const int sc = mlp_shape_check(dtype, T, h, f, N);
  if (sc != TP_OK) return sc;
  if (!X || !W1s || !W2s || !Z) return TP_ERR_NULL;
  if (!al16(X) || !al16(W1s) || !al16(W2s) || !al16(Z)) return TP_ERR_ALIGN;
  if (mlp_act_bytes(dtype, T, f) > static_cast<size_t>(TP_NOALLOC_SCRATCH_BYTES))
    return TP_ERR_WORKSPACE;  // the activation does not fit the fixed scratch array
  unsigned* err = nullptr;
  const int dc = check_device(&err);
  if (dc != TP_OK) return dc;
  void* Abuf = nullptr;
  const int ss = noalloc_scratch(&Abuf);
  if (ss != TP_OK) return ss;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t fN = f / N;
  if (dtype == TP_F32) {
    tpb::SimtArgs a1{};
    a1.A = static_cast<const float*>(X);
    a1.B = static_cast<const float*>(W1s);
    a1.C = static_cast<float*>(Abuf);
    a1.M = static_cast<int>(T);
    a1.N = static_cast<int>(fN);
    a1.K = static_cast<int>(h);
    a1.G = N;
    a1.S = 1;
    a1.b_sg = h * fN;
    a1.c_sg = T * fN;
    a1.lda = h;
    a1.ldb = fN;
    a1.ldc = fN;
    a1.gelu = 1;
    int rc = tpb::launch_gemm_f32(a1, st, tpb::kKMlpF32Fc1);
    if (rc) return gemm_status(rc);
    tpb::SimtArgs a2{};
    a2.A = static_cast<const float*>(Abuf);
    a2.B = static_cast<const float*>(W2s);
    a2.C = static_cast<float*>(Z);
    a2.M = static_cast<int>(T);
    a2.N = static_cast<int>(h);
    a2.K = static_cast<int>(fN);
    a2.G = 1;
    a2.S = N;
    a2.a_ss = T * fN;
    a2.b_ss = fN * h;
    a2.lda = fN;
    a2.ldb = h;
    a2.ldc = h;
    return gemm_status(tpb::launch_gemm_f32(a2, st, tpb::kKMlpF32Fc2));
  }
  const tpb::GemmOperand opX{X, h, T, 1, false, 0, 0};
  const tpb::GemmOperand opW1{W1s, fN, h, N, true, 1, 0};
  int rc = tpb::launch_gemm_bf16(tpb::kEpiGelu, opX, opW1, Abuf, nullptr, false, T, fN, N, 1, h, err, kWaitTimeoutNs,
                                 st, tpb::kKMlpFc1);
  if (rc) return gemm_status(rc);
  const tpb::GemmOperand opA{Abuf, fN, T, N, false, 0, 1};
  const tpb::GemmOperand opW2{W2s, h, fN, N, true, 0, 1};
  rc = tpb::launch_gemm_bf16(tpb::kEpiStore, opA, opW2, Z, nullptr, false, T, h, 1, N, fN, err, kWaitTimeoutNs, st,
                             tpb::kKMlpFc2);
  return gemm_status(rc);
}

}  // extern "C"
