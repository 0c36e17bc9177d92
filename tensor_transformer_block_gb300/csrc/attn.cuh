// Per-head fused causal attention on tcgen05 (forward and backward cores).
//
// Tensors are in the shard-major layouts of the boundary.  H query heads share
// Hkv key/value heads (grouped-query attention; Hkv = H is multi-head attention):
// query head j uses key/value head j / (H/Hkv).  Per shard, hN = H/N query and
// hkvN = Hkv/N key/value heads (io.zouht.com 张量并行 §2.2.1: each shard owns
// whole heads; with GQA it owns whole groups):
//   QKV  [N][B][S][W] with W = (hN + 2 hkvN) d: Q (hN heads), K and V (hkvN each),
//        all fp16
//   dQKV [N][B][S][W]: dQ, dK, dV (bf16, or fp16 with dqkv_f16)
//   O    [N][B][S][hN][d]  bf16, or fp16 with o_f16
//   dO   [N][B][S][hN][d]  fp16
//   LSE  [B][H][S] fp32          natural-log sum of exp of the scaled scores
// Global query head j lives in shard i = j / hN as local head jj = j % hN.
//
// Q and K are kept in fp16 (11 significant bits instead of bf16's 8): the softmax
// exponentiates scores whose range reaches tens of units, where bf16 Q and K would
// move the largest weights by several percent; fp16 puts the scores within ~2^-11
// relative and the products Q K^T still run as single tensor-core MMAs (fp16 x
// fp16, fp32 accumulation).  V, the probabilities P, dO and dS are fp16 too, so
// that every product of the core is an fp16 MMA and the attention output carries
// an eighth of bf16's rounding error.  Entries beyond +-65504 would overflow.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace tpb {

struct AttnDims {
  int B, S, H, hN, N, d, causal;
  int Hkv, hkvN;  // key/value heads in total and per shard (= H, hN without grouping)
  int o_f16 = 0;     // O stored as fp16 (else bf16)
  int dqkv_f16 = 0;  // dQ, dK, dV stored as fp16 (else bf16)
  // column offsets (elements) of local head jj (query) or kv (key/value) in QKV
  __host__ __device__ int qkv_width() const { return (hN + 2 * hkvN) * d; }
  __host__ __device__ int col_q(int jj) const { return jj * d; }
  __host__ __device__ int col_k(int kv) const { return (hN + kv) * d; }
  __host__ __device__ int col_v(int kv) const { return (hN + hkvN + kv) * d; }
  __host__ __device__ int dqkv_width() const { return (hN + 2 * hkvN) * d; }
  __host__ __device__ int group() const { return hN / hkvN; }
};

// Order in which the CTAs of an attention core are launched.  A CTA covers one
// (batch, head) unit and one block of it; with a causal mask the blocks carry
// unequal work, ranked r = 0 (most) .. blocks-1 (least).  The hardware gives CTAs
// to SMs in linear index order as SMs free up, so the units are taken in groups of
// `group`, and inside a group every unit's rank-0 block comes first, then every
// unit's rank-1 block, and so on (longest first within the group): the light
// blocks of one group run beside the heavy blocks of the next.  The group left
// over (units % group) goes first, so that the launch ends on the light blocks of
// a full group.  A group of about two waves of CTAs keeps the makespan within a
// few percent of the average load while the key/value tiles in use stay those of
// a few dozen heads.
struct WorkOrder {
  int units, blocks, group;
  __host__ __device__ void decode(int idx, int& unit, int& rank) const {
    const int first = units % group;  // size of the leading partial group (0: none)
    int base = 0, gsize = first, within = idx;
    if (idx >= first * blocks) {
      const int i = idx - first * blocks;
      const int grp = i / (group * blocks);
      within = i - grp * group * blocks;
      gsize = group;
      base = first + grp * group;
    }
    rank = within / gsize;
    unit = base + (within - rank * gsize);
  }
  __host__ __device__ int ctas() const { return units * blocks; }
};
inline WorkOrder make_work_order(int units, int blocks, int sms) {
  int group = (2 * sms + blocks - 1) / blocks;
  if (group > units) group = units;
  if (group < 1) group = 1;
  return WorkOrder{units, blocks, group};
}

// dS tiles written by the dK/dV kernel and read by the dQ kernel: for every
// (batch, query head, query block qb, key block kb) the core visits, 128 keys x 128
// queries of fp16 dS^T (key rows, query columns contiguous: 32 KB).  A head's tiles
// are ordered by query block, then key block: qb (qb + 1) / 2 + kb with the causal
// mask (kb <= qb), qb * nb + kb without it.
__host__ __device__ inline long long ds_tiles_per_head(const AttnDims& a) {
  const long long nb = (a.S + 127) / 128;
  return a.causal ? nb * (nb + 1) / 2 : nb * nb;
}
__host__ __device__ inline long long ds_tiles(const AttnDims& a) {
  return static_cast<long long>(a.B) * a.H * ds_tiles_per_head(a);
}
__host__ __device__ inline long long ds_tile_index(const AttnDims& a, int b, int j, int qb, int kb) {
  const long long nb = (a.S + 127) / 128;
  const long long within = a.causal ? static_cast<long long>(qb) * (qb + 1) / 2 + kb : qb * nb + kb;
  return (static_cast<long long>(b) * a.H + j) * ds_tiles_per_head(a) + within;
}

// Number of d-wide planes per (token, local head) in QKV without grouping.
constexpr int kQkvPlanes = 3;

// Forward: O and LSE from QKV (returns 0, 1 bad arguments, 2 CUDA failure).
int launch_attn_fwd(const AttnDims& a, const void* qkv, void* o, float* lse, unsigned* err,
                    unsigned long long timeout_ns, cudaStream_t st);

// Backward cores.  Dsum[b][j][s] = sum_e dO * O over the head dim; dqkv gets dQ,
// dK, dV (a key/value head's gradient summed over the query heads of its group).
// ``dsbuf``: scratch of ds_tiles(a) x 32 KB (16-byte aligned) for the dS tiles.
int launch_attn_bwd(const AttnDims& a, const void* qkv, const void* o, const void* dout, const float* lse,
                    float* dsum, void* dsbuf, void* dqkv, unsigned* err, unsigned long long timeout_ns,
                    cudaStream_t st);

}  // namespace tpb
