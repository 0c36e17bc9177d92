/*
 * libtpblock — the Megatron tensor-parallel transformer block on one GB300 (sm_103a).
 *
 * The block is the pair of matrix splits the pages describe: a column-split GEMM
 * whose shards apply the element-wise activation on their own, followed by a
 * row-split ("outer-product-sum") GEMM whose per-shard partial products are added
 * (damodev 3D并行 §1.1 and §1.2.1; io.zouht.com 张量并行 §2.1 and §2.2.1; wangyu.me
 * 张量并行 §两种切分方式 and §多层感知机（MLP）中的张量并行).  The N shards here are
 * logical partitions on ONE GPU: where the pages place an all-reduce, this library
 * adds the N partial sums on the device, inside one fp32 accumulator, in the fixed
 * order shard 0, 1, ..., N-1.  There is no inter-GPU communication.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Y = X W with W stored [in x out], row-major and dense (wangyu.me 张量并行
 *    §两种切分方式: X is B x M, W is M x N).  T = tokens (= B*S), h = hidden size,
 *    f = FFN size, H = heads, d = head dim, N = shard count.
 *  - Every tensor pointer is a DEVICE pointer owned by the caller, 16-byte aligned
 *    (TP_ERR_ALIGN otherwise).  The library never allocates device memory that the
 *    caller sees; scratch space is the caller's workspace ``ws`` (256-byte
 *    aligned, at least the size the matching *_workspace_bytes call returns).
 *  - Weights are passed shard-major, exactly as the pages split them:
 *      column split  W1s [N][h][f/N]     block i = columns i*f/N..(i+1)*f/N-1 of W1
 *      row split     W2s [N][f/N][h]     block i = rows of W2 (same bytes as W2)
 *      attention     Wqkv [N][h][3][H/N][d]  shard i = the Q, K and V columns of
 *                    heads i*H/N..(i+1)*H/N-1 (column split by head)
 *                    Wo [N][(H/N)*d][h]  row split by head (same bytes as Wo)
 *  - N must divide f (MLP) and H (attention); a shard count that does not divide
 *    the head count is an error (io.zouht.com 张量并行 §2.2.1, 32 heads on 5 GPUs).
 *  - Row lengths that TMA moves must be multiples of 8 elements (16 bytes):
 *    h, f/N, (H/N)*d, and d must be a multiple of 64 with d <= 128 for attention.
 *  - ``stream`` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *    asynchronous: the return code reports validation and launch errors only.
 *    Errors detected on the device (a bounded wait that ran out) are latched in a
 *    device error word and surface through tp_sync_status().
 *  - dtype: TP_BF16 (bf16 storage, fp32 accumulation) everywhere; TP_F32 (fp32
 *    FFMA, no TF32) is accepted by tp_mlp_fwd (and tp_mlp_fwd_noalloc) only.
 */
#ifndef TPBLOCK_H
#define TPBLOCK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TP_API __attribute__((visibility("default")))
#else
#define TP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TP_OK = 0,
  TP_ERR_NULL = 1,      /* a required pointer is NULL */
  TP_ERR_SHAPE = 2,     /* a size < 1, N does not divide f or H, a row length not a multiple of 8 */
  TP_ERR_DTYPE = 3,     /* dtype not supported by this call */
  TP_ERR_WORKSPACE = 4, /* ws is NULL or smaller than the *_workspace_bytes figure */
  TP_ERR_CUDA = 5,      /* a CUDA runtime/driver call failed (launch, tensor-map encode, sync) */
  TP_ERR_TIMEOUT = 6,   /* a kernel's bounded wait ran out (reported by tp_sync_status) */
  TP_ERR_ALIGN = 7,     /* a pointer is not 16-byte aligned (ws: 256-byte) */
  TP_ERR_DEVICE = 8,    /* the current device is not a compute capability 10.3 (sm_103) GPU */
  TP_ERR_BOUNDS = 9     /* a debug build's device-side bounds or alignment check failed
                           (reported by tp_sync_status; release builds never raise it) */
} tp_status;

typedef enum { TP_F32 = 0, TP_BF16 = 1 } tp_dtype;

/* Library version, (major << 16) | minor. */
TP_API int tp_version(void);

/* Static string for a tp_status value ("unknown status" for anything else). */
TP_API const char* tp_status_string(int status);

/* TP_OK if the current CUDA device is sm_103 and the kernels can run on it,
 * TP_ERR_DEVICE if not, TP_ERR_CUDA if no device can be queried. */
TP_API int tp_device_check(void);

/* Waits for ``stream``, then reads and clears the device error word.
 * Returns TP_ERR_TIMEOUT if any kernel since the last call gave up on a bounded
 * wait, TP_ERR_BOUNDS if (in a library built with -DTPBLOCK_DEBUG) a kernel found
 * an index outside its tensor or a TMA coordinate off its 16-byte boundary and
 * skipped that access, TP_ERR_CUDA if the synchronisation itself failed, TP_OK
 * otherwise. */
TP_API int tp_sync_status(void* stream);

/* ---------------------------------------------------------------- MLP block */

/* Bytes of scratch for tp_mlp_fwd and tp_mlp_bwd: one [N][T][f/N] activation-sized
 * buffer (A in the forward when A_save is NULL, dY in the backward), rounded up to
 * 256 bytes, plus, for bf16 shapes whose row-parallel GEMMs (Z, dX) have too few
 * tiles to fill the GPU (at most 76 tiles of 128 x 256, at least 32 K blocks of
 * 64), room for their split-K partial sums: 2 x T x h fp32.  The activation-sized
 * part is required; with the rest present those GEMMs run their K loop (the
 * shards) in two halves on twice the SMs and a second kernel adds the two fp32
 * partials in that fixed order (deterministic; a different rounding order than the
 * unsplit sum).  0 for invalid sizes. */
TP_API size_t tp_mlp_workspace_bytes(int dtype, int64_t T, int64_t h, int64_t f, int N);

/* MLP block forward, Z = sum_i GeLU(X W1_i) W2_i.
 * (damodev 3D并行 §1.2.1: column split of the first GEMM, element-wise Act per
 *  shard, row split of the second GEMM, one all-reduce; io.zouht.com 张量并行
 *  §2.2.1 前馈网络: Gelu(X W_1) split by columns, the second layer by rows.)
 *   X      [T][h]                 input (read)
 *   W1s    [N][h][f/N]            column blocks of W1 (read)
 *   W2s    [N][f/N][h]            row blocks of W2 (read)
 *   Y_save [N][T][f/N] or NULL    pre-activation Y_i = X W1_i (written if not NULL;
 *                                 tp_mlp_bwd needs it)
 *   A_save [N][T][f/N] or NULL    A_i = GeLU_tanh(Y_i) (written; if NULL it lives in ws)
 *   Z      [T][h]                 output, the shard partial sums added on the device
 *                                 in order i = 0..N-1 in one fp32 accumulator
 * GeLU_tanh(x) = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), evaluated in fp32.
 * TP_F32: every tensor fp32, FFMA accumulation; when the output tiles would leave
 * most SMs idle (few tokens) each tile's K loop (shard 0..N-1, then K within a
 * shard) is split into up to 8 contiguous ranges whose fp32 partial sums are added
 * in range order, so the order stays fixed for a shape.  TP_BF16: bf16 tensors,
 * fp32 accumulation, outputs rounded to bf16 once. */
TP_API int tp_mlp_fwd(int dtype, int64_t T, int64_t h, int64_t f, int N,
               const void* X, const void* W1s, const void* W2s,
               void* Y_save, void* A_save, void* Z,
               void* ws, size_t ws_bytes, void* stream);

/* MLP block backward for an upstream gradient dZ (bf16 only).
 * (wangyu.me 张量并行 §通信模式: for the row split dL/dY_i = dL/dY and
 *  dW_i = X_i^T dY; for the column split dW_i = X^T dY_i and dX = sum_i dY_i W_i^T,
 *  the all-reduce of io.zouht.com 张量并行 §2.3 f in the backward pass.)
 *   dY_i  = (dZ W2_i^T) * GeLU'(Y_i)   kept in ws [N][T][f/N]
 *   dW2_i = A_i^T dZ      -> dW2s [N][f/N][h]
 *   dW1_i = X^T dY_i      -> dW1s [N][h][f/N]
 *   dX    = sum_i dY_i W1_i^T  -> dX [T][h], shard sum on the device, order 0..N-1
 * Y_save and A_save are the tensors tp_mlp_fwd wrote for the same X, W1s. */
TP_API int tp_mlp_bwd(int dtype, int64_t T, int64_t h, int64_t f, int N,
               const void* X, const void* W1s, const void* W2s,
               const void* Y_save, const void* A_save, const void* dZ,
               void* dX, void* dW1s, void* dW2s,
               void* ws, size_t ws_bytes, void* stream);

/* Size of the fixed device array tp_mlp_fwd_noalloc keeps its scratch in (32 MiB). */
#define TP_NOALLOC_SCRATCH_BYTES (32u << 20)

/* MLP block forward for callers that cannot allocate device memory.
 * The method on the pages has no counterpart to this call; it exists for the
 * software around it.  Some callers cannot call cudaMalloc at the point where
 * they run the block: a plug-in inside a host framework that owns every device
 * allocation and plans memory ahead of time, or a runtime with a fixed memory
 * budget that forbids allocation once serving has started (cudaMalloc can also
 * synchronise the device, which such callers must avoid).  This call computes
 * the same Z as tp_mlp_fwd with Y_save = A_save = NULL, but keeps the activation
 * A in a fixed array of TP_NOALLOC_SCRATCH_BYTES in the library's own device
 * memory instead of a caller's workspace; the caller still passes X, W1s, W2s
 * and Z.  It calls neither cudaMalloc nor cudaFree nor any allocating routine.
 *  - Limit: T * f * sizeof(element) <= TP_NOALLOC_SCRATCH_BYTES, else
 *    TP_ERR_WORKSPACE (every other check as in tp_mlp_fwd).
 *  - The first call on a device looks up the array's device address with that
 *    device current; make that first call before any stream capture.
 *  - All calls on a device share the one array.  The array is written before it
 *    is read in every call (nothing in it has to start at zero), but calls whose
 *    kernels overlap on the GPU, such as calls on two streams at once, race on it.
 *  - The device address is kept for the life of the process: do not use the
 *    library on a device after cudaDeviceReset() on it (the same holds for the
 *    device error word every call uses). */
TP_API int tp_mlp_fwd_noalloc(int dtype, int64_t T, int64_t h, int64_t f, int N,
                              const void* X, const void* W1s, const void* W2s, void* Z, void* stream);

/* ------------------------------------------------------ gated MLP block */

/* Bytes of scratch tp_gmlp_fwd (with A_save == NULL) and tp_gmlp_bwd need: one
 * [N][T][2][f/N] buffer (the backward's dG, dU) plus alignment.  0 for invalid
 * sizes or a dtype other than TP_BF16. */
TP_API size_t tp_gmlp_workspace_bytes(int dtype, int64_t T, int64_t h, int64_t f, int N);

/* Gated (SwiGLU) MLP block forward (bf16), Z = sum_i (silu(X Wg_i) * (X Wu_i)) Wd_i.
 * (wangyu.me 张量并行 §多层感知机（MLP）中的张量并行: the Qwen3 MLP, gate and up
 *  projections fused by concatenating their columns so that one product gives
 *  both; both split by columns, the down projection by rows, one all-reduce.)
 *   X       [T][h]              input (read)
 *   Wgus    [N][h][2][f/N]      shard i = [Wg_i | Wu_i]: columns i*f/N..(i+1)*f/N-1
 *                               of W_gate, then the same columns of W_up (read)
 *   Wds     [N][f/N][h]         row blocks of W_down (read)
 *   GU_save [N][T][2][f/N] or NULL  G_i = X Wg_i and U_i = X Wu_i (written if not
 *                               NULL; tp_gmlp_bwd needs it)
 *   A_save  [N][T][f/N] or NULL A_i = silu(G_i) * U_i (written; if NULL it lives in ws)
 *   Z       [T][h]              output, shard partial sums added on the device in
 *                               order i = 0..N-1 in one fp32 accumulator
 * silu(x) = x / (1 + e^-x) in fp32 on the fp32 accumulators; f is the width of
 * each of the gate and up projections.  TP_ERR_DTYPE for TP_F32. */
TP_API int tp_gmlp_fwd(int dtype, int64_t T, int64_t h, int64_t f, int N,
                       const void* X, const void* Wgus, const void* Wds,
                       void* GU_save, void* A_save, void* Z,
                       void* ws, size_t ws_bytes, void* stream);

/* Gated MLP block backward for an upstream gradient dZ (bf16).  The pages give
 * no backward for this block; this is the chain rule through the forward:
 *   dA_i  = dZ Wd_i^T
 *   dG_i  = dA_i * U_i * silu'(G_i),  dU_i = dA_i * silu(G_i)   kept in ws [N][T][2][f/N]
 *   dWd_i = A_i^T dZ                       -> dWds  [N][f/N][h]
 *   [dWg_i | dWu_i] = X^T [dG_i | dU_i]    -> dWgus [N][h][2][f/N]
 *   dX    = sum_i [dG_i | dU_i] [Wg_i | Wu_i]^T -> dX [T][h], shard sum on the
 *           device, order 0..N-1 (the column split's backward all-reduce)
 * silu'(x) = s (1 + x (1 - s)) with s = 1 / (1 + e^-x).  GU_save and A_save are
 * what tp_gmlp_fwd wrote for the same X, Wgus. */
TP_API int tp_gmlp_bwd(int dtype, int64_t T, int64_t h, int64_t f, int N,
                       const void* X, const void* Wgus, const void* Wds,
                       const void* GU_save, const void* A_save, const void* dZ,
                       void* dX, void* dWgus, void* dWds,
                       void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------- attention block */

/* Bytes of scratch tp_attn_fwd (with NULL saves) and tp_attn_bwd need: the
 * forward's QKV, O and LSE (or the backward's dQKV, dO and Dsum in the same
 * regions), plus the backward's dS tiles, B x H x ceil(S/128)^2 x 32 KB (fp16
 * 128 x 128 tiles of dS, which the dQ kernel multiplies by K). */
TP_API size_t tp_attn_workspace_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int N);

/* Self-attention block forward (bf16), heads split over N shards.
 * (damodev 3D并行 §1.2.2; io.zouht.com 张量并行 §2.2.1 多头注意力机制: Q/K/V split
 *  by columns so each shard owns whole heads, W_O split by rows, one all-reduce;
 *  wangyu.me 张量并行 §注意力机制中的张量并行.)
 *   QKV_i = X Wqkv_i                       -> QKV_save [N][T][3][H/N][d] (or ws): planes
 *                                             Q, K, V, stored as fp16 (11 significant
 *                                             bits, so that the scores Q K^T, which the
 *                                             softmax exponentiates, carry about 2^-11
 *                                             relative error instead of bf16's 2^-8,
 *                                             and P V is an fp16 product; entries
 *                                             above 65504 overflow)
 *   O_j   = softmax(mask(Q_j K_j^T / sqrt(d))) V_j, per batch and head j; the
 *           probabilities enter P V as fp16
 *                                          -> O_save [N][T][(H/N)*d] (or ws), bf16
 *   LSE   = log sum_k exp(Q_j K_j^T/sqrt(d)) per query -> LSE_save [B][H][S] fp32 (or ws)
 *   Z     = sum_i O_i Wo_i                 -> Z [T][h], shard sum on the device
 * X is [B*S][h] (token t = b*S + s).  causal != 0 masks keys after the query. */
TP_API int tp_attn_fwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int N, int causal,
                const void* X, const void* Wqkv, const void* Wo,
                void* QKV_save, void* O_save, float* LSE_save, void* Z,
                void* ws, size_t ws_bytes, void* stream);

/* Self-attention block backward (bf16) for an upstream gradient dZ.
 * The pages give no attention backward; this is the chain rule through the
 * forward's definition:
 *   dO_i  = dZ Wo_i^T,  dWo_i = O_i^T dZ
 *   per head: D = rowsum(dO * O), P = exp(S/sqrt(d) - LSE), dV = P^T dO,
 *             dP = dO V^T, dS = P * (dP - D), dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d)
 *   dWqkv_i = X^T dQKV_i,  dX = sum_i dQKV_i Wqkv_i^T (shard sum on the device)
 *   (dQKV [N][T][3][H/N][d], all bf16, lives in ws, and so does dO, stored as
 *   fp16: every product of the core is fp16; P is recomputed from the saved fp16
 *   Q, K and LSE)
 * QKV_save, O_save, LSE_save are what tp_attn_fwd wrote for the same inputs. */
TP_API int tp_attn_bwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int N, int causal,
                const void* X, const void* Wqkv, const void* Wo,
                const void* QKV_save, const void* O_save, const float* LSE_save,
                const void* dZ, void* dX, void* dWqkv, void* dWo,
                void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------- grouped-query attention block */

/* The attention block with H query heads sharing Hkv key/value heads
 * (grouped-query attention, named on wangyu.me 张量并行 §注意力机制中的张量并行
 * next to multi-head attention; the page gives no formula).  Reading: query head
 * j uses key/value head j / (H/Hkv) (consecutive query heads form a group); the
 * head split puts query heads i*H/N .. (i+1)*H/N-1 and key/value heads
 * i*Hkv/N .. (i+1)*Hkv/N-1 on shard i, so N must divide Hkv (every group stays on
 * one shard; TP_ERR_SHAPE otherwise) and Hkv must divide H.  Hkv = H is exactly
 * tp_attn_fwd / tp_attn_bwd (the same bytes in every layout).
 *   Wqkv     [N][h][(H/N + 2 Hkv/N) d]   shard i: its query heads, then its key
 *                                        heads, then its value heads, d columns each
 *   Wo       [N][(H/N) d][h]             as tp_attn_fwd
 *   QKV_save [N][T][(H/N + 2 Hkv/N) d]   Q, K, V (fp16) as tp_attn_fwd
 *   O_save, LSE_save, Z, dX, dWo         as tp_attn_fwd / tp_attn_bwd
 *   dWqkv    Wqkv's layout; a key/value head's gradient sums its group's query heads */
TP_API size_t tp_gqa_workspace_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int Hkv, int d, int N);
TP_API int tp_gqa_fwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int Hkv, int d, int N, int causal,
                      const void* X, const void* Wqkv, const void* Wo,
                      void* QKV_save, void* O_save, float* LSE_save, void* Z,
                      void* ws, size_t ws_bytes, void* stream);
TP_API int tp_gqa_bwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int Hkv, int d, int N, int causal,
                      const void* X, const void* Wqkv, const void* Wo,
                      const void* QKV_save, const void* O_save, const float* LSE_save,
                      const void* dZ, void* dX, void* dWqkv, void* dWo,
                      void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------ attention block then MLP block (layer) */

/* Bytes of the ``save`` buffer tp_attn_mlp_fwd fills and tp_attn_mlp_bwd reads, and
 * of tp_attn_mlp_bwd's scratch.  0 for invalid sizes (the attention rules and the
 * MLP rules above apply, with T = B*S). */
TP_API size_t tp_attn_mlp_save_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N);
TP_API size_t tp_attn_mlp_workspace_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f,
                                          int N);

/* Transformer layer forward (bf16 inputs, weights and output): the attention
 * block, then the MLP block on its output, Z = MLP(Attn(X)).  The pages put the
 * two tensor-parallel blocks one after the other and keep LayerNorm, dropout and
 * the residuals outside them (io.zouht.com 张量并行 §2.2.2; damodev 3D并行 §1.2.1
 * and §1.2.2); this call is the two blocks alone.  Attn and MLP compute what
 * tp_attn_fwd and tp_mlp_fwd compute, with one difference in storage: the
 * attention output H, the MLP's input, is kept in fp16 instead of bf16, and so is
 * O.  The MLP's GeLU' is steep where its pre-activations cross zero, so an error
 * in H reaches the backward's dY amplified; fp16's 11 significant bits keep it an
 * eighth of bf16's.  The products with an fp16 operand (O Wo, H W1) take fp16
 * copies of Wo and W1s that this call makes in ``save`` (exact for weights of
 * magnitude 2^-17 .. 65504; smaller ones round to a multiple of 2^-24).
 * ``save`` (256-byte aligned, tp_attn_mlp_save_bytes) receives QKV, O, LSE, the
 * fp16 weight copies, H, Y and A; its layout is private to the library. */
TP_API int tp_attn_mlp_fwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N,
                           int causal, const void* X, const void* Wqkv, const void* Wo,
                           const void* W1s, const void* W2s, void* save, size_t save_bytes,
                           void* Z, void* stream);

/* The layer's backward for an upstream dZ: the MLP block's backward on H (dY and
 * dH kept in fp16), then the attention block's backward with upstream dH.  Every
 * gradient is written: dX [T][h], dWqkv, dWo, dW1s, dW2s in the forward's layouts
 * (bf16).  ``save`` is what tp_attn_mlp_fwd wrote for the same inputs; ws:
 * tp_attn_mlp_workspace_bytes. */
TP_API int tp_attn_mlp_bwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N,
                           int causal, const void* X, const void* Wqkv, const void* Wo,
                           const void* W1s, const void* W2s, const void* save, size_t save_bytes,
                           const void* dZ, void* dX, void* dWqkv, void* dWo, void* dW1s, void* dW2s,
                           void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------ LayerNorm and residuals */

/* The pages keep LayerNorm, dropout and the residual connections outside the
 * tensor-parallel blocks, replicated on every shard (io.zouht.com 张量并行 §2.2.2;
 * sunjinbo.space 并行方式 §SP).  LayerNorm of one hidden state h of d_model values
 * (io.zouht.com 张量并行 §2.2.2, LayerNorm):
 *   mu = mean_i h_i,  sigma^2 = mean_i (h_i - mu)^2,
 *   h_hat = (h - mu) / sqrt(sigma^2 + eps),  h' = gamma * h_hat + beta.
 * Rows are bf16 [T][h] with h a multiple of 8 and h <= 16384; gamma, beta bf16 [h];
 * statistics fp32, computed on the device in fp32. */

/* Scratch of tp_layernorm_bwd (fp32 partial column sums).  0 for invalid sizes. */
TP_API size_t tp_layernorm_workspace_bytes(int dtype, int64_t T, int64_t h);

/* Y = LayerNorm(X) per row; mean [T] and rstd [T] = 1 / sqrt(sigma^2 + eps) are
 * written for the backward.  eps >= 0 (TP_ERR_SHAPE otherwise). */
TP_API int tp_layernorm_fwd(int dtype, int64_t T, int64_t h, float eps,
                            const void* X, const void* gamma, const void* beta,
                            void* Y, float* mean, float* rstd, void* stream);

/* Backward of Y = LayerNorm(X) for an upstream dY, plus an optional residual
 * gradient dR [T][h] (NULL = none).  The pages give no backward; by the chain
 * rule, with g = dY * gamma and x_hat = (X - mean) * rstd per row:
 *   dX = rstd (g - mean(g) - x_hat mean(g x_hat)) + dR
 *   dgamma = sum over rows of dY * x_hat,  dbeta = sum over rows of dY   (bf16 [h])
 * The column sums are finished from per-CTA fp32 partials in a fixed order (the
 * result does not vary run to run).  mean, rstd: what tp_layernorm_fwd wrote. */
TP_API int tp_layernorm_bwd(int dtype, int64_t T, int64_t h,
                            const void* X, const void* gamma, const float* mean, const float* rstd,
                            const void* dY, const void* dR, void* dX, void* dgamma, void* dbeta,
                            void* ws, size_t ws_bytes, void* stream);

/* Bytes of the ``save`` buffer tp_layer_fwd fills and tp_layer_bwd reads, and of
 * tp_layer_bwd's scratch.  0 for invalid sizes (the attention and MLP rules
 * above, plus the LayerNorm rules, apply). */
TP_API size_t tp_layer_save_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N);
TP_API size_t tp_layer_workspace_bytes(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N);

/* Pre-norm transformer layer forward (bf16): the two tensor-parallel blocks with
 * LayerNorm and a residual connection around each, dropout off.  The pages do not
 * fix the order; the pre-norm placement is the reading taken:
 *   H1 = X + Attn(LN1(X))      (the residual is added in the output projection's
 *                               epilogue, after the shard sum)
 *   Z  = H1 + MLP(LN2(H1))     (likewise in the second MLP GEMM's epilogue)
 * Attn and MLP compute what tp_attn_fwd and tp_mlp_fwd compute.  Inside the layer
 * the LayerNorm outputs LN1(X) and LN2(H1), the attention output O and, in the
 * backward, dY, the LayerNorm input gradients, dH1 and dQKV are stored in fp16
 * (11 significant bits) instead of bf16: LN1(X) feeds the scores the softmax
 * exponentiates and LN2(H1) the MLP whose GeLU' amplifies errors, and with bf16
 * there the layer's gradients missed a 5e-3 relative error bound at h = 8192.
 * The products with an fp16 operand take fp16 copies of Wqkv, Wo and W1s that this
 * call makes in ``save`` (exact for weights of magnitude 2^-17 .. 65504; smaller
 * ones round to a multiple of 2^-24).  ``save`` (256-byte aligned,
 * tp_layer_save_bytes) receives LN1(X), H1 (bf16), LN2(H1), their row statistics,
 * the blocks' saved tensors and the weight copies; its layout is private to the
 * library. */
TP_API int tp_layer_fwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N,
                        int causal, float eps,
                        const void* X, const void* ln1_g, const void* ln1_b, const void* Wqkv, const void* Wo,
                        const void* ln2_g, const void* ln2_b, const void* W1s, const void* W2s,
                        void* save, size_t save_bytes, void* Z, void* stream);

/* Pre-norm layer backward for an upstream dZ: the MLP block's backward on LN2(H1),
 * dH1 = dZ + LN2'(.), the attention block's backward with upstream dH1, then
 * dX = dH1 + LN1'(.).  Every gradient is written: dX [T][h], dln1_g, dln1_b,
 * dln2_g, dln2_b [h], dWqkv, dWo, dW1s, dW2s in the forward's layouts.  ``save``
 * is what tp_layer_fwd wrote for the same inputs; ws: tp_layer_workspace_bytes. */
TP_API int tp_layer_bwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N, int causal,
                        const void* X, const void* ln1_g, const void* Wqkv, const void* Wo,
                        const void* ln2_g, const void* W1s, const void* W2s,
                        const void* save, size_t save_bytes, const void* dZ,
                        void* dX, void* dln1_g, void* dln1_b, void* dWqkv, void* dWo,
                        void* dln2_g, void* dln2_b, void* dW1s, void* dW2s,
                        void* ws, size_t ws_bytes, void* stream);

/* The same pre-norm layer in the tensor + sequence parallel form (io.zouht.com
 * 张量并行 §2.2.2 与序列并行结合 and §2.3): outside the blocks, X, Z, dZ, dX (and the
 * saved LayerNorm outputs and H1) are split along the sequence into N shards,
 *   X, Z, dZ, dX   [N][B][S/N][h]   shard c holds positions c*S/N .. (c+1)*S/N-1
 *                                   of every sequence
 * LayerNorm and the residual adds work shard by shard.  Where the pages place an
 * all-gather before a block (g) the column-parallel GEMM's TMA copies read the
 * rows of every shard in sequence order; where they place a reduce-scatter after
 * it (g*) the row-parallel GEMM sums the tensor shards in its accumulator and its
 * stores put each row in its sequence shard.  No extra pass over memory is made.
 * Requires S/N to be a multiple of 128 (no GEMM tile spans two shards; else
 * TP_ERR_SHAPE); everything else as tp_layer_fwd / tp_layer_bwd, whose save
 * buffer and workspace sizes apply. */
TP_API int tp_sp_layer_fwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N,
                           int causal, float eps,
                           const void* X, const void* ln1_g, const void* ln1_b, const void* Wqkv, const void* Wo,
                           const void* ln2_g, const void* ln2_b, const void* W1s, const void* W2s,
                           void* save, size_t save_bytes, void* Z, void* stream);
TP_API int tp_sp_layer_bwd(int dtype, int64_t B, int64_t S, int64_t h, int H, int d, int64_t f, int N, int causal,
                           const void* X, const void* ln1_g, const void* Wqkv, const void* Wo,
                           const void* ln2_g, const void* W1s, const void* W2s,
                           const void* save, size_t save_bytes, const void* dZ,
                           void* dX, void* dln1_g, void* dln1_b, void* dWqkv, void* dWo,
                           void* dln2_g, void* dln2_b, void* dW1s, void* dW2s,
                           void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------ diagnostics */

/* Launches one block whose single thread waits on a shared-memory barrier that
 * nothing ever signals, with the same bounded wait the GEMM and attention kernels
 * use, limited to ``timeout_ns``.  The wait runs out, the kernel latches
 * TP_ERR_TIMEOUT in the device error word and returns; the context stays usable.
 * Used to test the timeout path (tp_sync_status must then report TP_ERR_TIMEOUT). */
TP_API int tp_debug_timeout_probe(int64_t timeout_ns, void* stream);

/* ------------------------------------------------------------ GEMM tiling */

/* Tiling of every GEMM the library launches (process-wide; for tests and
 * measurement): 0 = automatic (default: a CTA pair per 256 x 256 tile through
 * tcgen05 cta_group::2 unless the output has at most 128 rows, then one CTA per
 * 128 x 256 tile), 1 = always one CTA per tile, 2 = always CTA pairs.  Every
 * tiling computes the same products; TP_ERR_SHAPE for another value (the setting
 * is then unchanged).  Each CTA loads only its own tiles: no TMA load is
 * multicast across a cluster. */
TP_API int tp_set_gemm_tiling(int mode);

/* ------------------------------------------------------- launch overlap */

/* Programmatic dependent launch (process-wide; for tests and measurement).
 * 1 (default): every kernel is launched with programmatic stream serialisation
 * (cudaLaunchAttributeProgrammaticStreamSerialization).  Its CTAs may become
 * resident while the previous kernel in the stream finishes; each runs only its
 * prologue (barrier set-up, tensor-map prefetch, TMEM allocation) and then waits,
 * in the PTX griddepcontrol.wait instruction, until that kernel has completed and its
 * writes are visible, before it reads or writes global memory.  That hides the
 * launch latency and the prologue between the dependent kernels of a call.
 * 0: ordinary stream order.  The results are bit-identical either way.
 * TP_ERR_SHAPE for a value other than 0 or 1 (the setting is then unchanged). */
TP_API int tp_set_launch_overlap(int on);

/* ---------------------------------------------------------- kernel timing */

/* Every kernel the library launches is counted per kind.  With timing on, a
 * pair of CUDA events is also recorded on the launch stream around each launch.
 * tp_timing_enable() clears the counts and the recorded times. */
TP_API int tp_timing_enable(int on);

/* Number of kernel kinds (indices 0 .. n-1 for the calls below). */
TP_API int tp_timing_kinds(void);

/* Static name of kernel kind ``kind`` (NULL if out of range). */
TP_API const char* tp_timing_name(int kind);

/* Launch count since the last tp_timing_enable() and, if timing was on, the sum
 * of the launches' event-measured durations in milliseconds (waits for the
 * events).  TP_ERR_SHAPE for a bad index, TP_ERR_CUDA if an event query fails. */
TP_API int tp_timing_read(int kind, int64_t* launches, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* TPBLOCK_H */
