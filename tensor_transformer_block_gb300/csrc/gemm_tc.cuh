// Persistent, warp-specialised tcgen05 GEMM for the tensor-parallel block.
//
// One launch computes, for g = 0..G-1,
//     C[g] (M x N) = sum_{s=0}^{S-1} A(g, s) (M x Ks) * B(g, s) (Ks x N)
// with bf16 operands, an fp32 accumulator in TMEM and a fused epilogue.
//   * G > 1, S = 1 is the column-parallel GEMM: one output block per shard
//     (Y_i = X W1_i; damodev 3D并行 §1.2.1 列切分).
//   * G = 1, S = N is the row-parallel GEMM: the K loop walks shard 0's K tiles,
//     then shard 1's, ..., all into ONE accumulator, so the shard partial sums
//     (the pages' all-reduce, damodev 3D并行 §1.1 外积和切分) are added in TMEM in
//     a fixed order and never written out.
// Every operand is addressed through a 3-D TMA map whose outer coordinate is the
// shard index z = g*zg + s*zs, so shard-major layouts need no repacking, and
// K-ragged shards read zeros past their end.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tpb {

enum GemmEpi : int {
  kEpiStore = 0,  // C = bf16(acc)
  kEpiGelu = 1,   // C = bf16(GeLU_tanh(acc)); optionally Yout = bf16(acc)
  kEpiDGelu = 2,  // C = bf16(acc * GeLU_tanh'(Yin)), Yin read through a TMA map
  kEpiSplit = 3,  // C = fp16(acc) for columns < split_cols (a multiple of 64), bf16(acc) after
  // Gated (SwiGLU) MLP.  B is a two-part operand [G][K][2][N] (gate columns, then
  // up columns); one tile computes 128 output columns n: the MMA's 256 accumulator
  // columns hold gate(n) in 0..127 and up(n) in 128..255.
  kEpiSwiGLU = 4,   // C = bf16(silu(gate) * up); optionally Yaux [G][M][2][N] = bf16(gate), bf16(up)
  kEpiDSwiGLU = 5,  // Yaux [G][M][2][N] holds G, U; C [G][M][2][N] gets
                    // C(.,0,.) = bf16(acc * U * silu'(G)), C(.,1,.) = bf16(acc * silu(G))
  kEpiResidual = 6,  // C = bf16(acc + R), R = Yaux [G][M][ldc] (a residual connection)
  // split-K: the fp32 accumulator of one K-split written to partial[split][G][M][N];
  // a second kernel adds the splits in order 0, 1, ... and applies kEpiStore or
  // kEpiResidual (chosen by the launcher, never passed in)
  kEpiPartial = 7,
};

struct GemmShape {
  int M, N;        // output rows / cols per group
  int G;           // independent output groups
  int S;           // segments added into one output
  int kb_per_seg;  // 64-wide K blocks per segment
  int tiles_m, tiles_n;
  int a_zg, a_zs, b_zg, b_zs;  // outer TMA coordinate = g*zg + s*zs
  int store_y;                 // kEpiGelu: also write the pre-activation
  int split_cols;              // kEpiStore / kEpiSplit: columns < split_cols are stored as fp16
  int ab_f16;                  // A and B are fp16 (else bf16); one MMA's operands share a type
  int ksplit;                  // K-splits per output tile (1: none); tile index = split * tiles + tile
  int kps;                     // 64-wide K blocks per split
  int c_f16;                   // kEpiDGelu, kEpiResidual: the output C is fp16 (else bf16)
  // token remaps (0 = off): the operand's row coordinate t (A, B: d1; C, Yaux: M)
  // is a token b*S + s stored at [s / L][b][s % L] (sequence-sharded layout)
  int a_spS, a_spL, b_spS, b_spL, c_spS, c_spL;
  int g_mode;  // tile order across groups (gemm_tc.cu decode_tile)
  // an MN-major operand whose rows are whole 64-element chunks is read through a map
  // with the chunk as an outer dimension ({64, K, chunks, ...}), so one copy per
  // stage brings all of its columns (the producer's issue time per copy is ~100 cycles)
  int a_chunked, b_chunked;
  unsigned* err;
  unsigned long long timeout_ns;
};

// One operand as the host describes it: a row-major [d2][d1][d0] bf16 tensor
// (d0 contiguous).  K-major: d0 runs along K, d1 along M (or N).  MN-major: d0
// runs along M (or N), d1 along K.
struct GemmOperand {
  const void* ptr;
  int64_t d0, d1, d2;
  bool mn_major;
  int zg, zs;
  int parts = 1;  // 2: the tensor is [d2][d1][2][d0] (kEpiSwiGLU's B: gate, up)
  // Sequence-sharded rows (d2 must be 1): row t = b*sp_S + s of the logical
  // [d1][d0] tensor is stored at [s / sp_L][b][s % sp_L][d0] (sp_S = 0: plain).
  int sp_S = 0, sp_L = 0;
};

// Host launcher (gemm_tc.cu).  C and Yaux are [G][M][ldc] bf16 tensors of which
// columns 0..N-1 are computed (ldc = 0 means ldc = N); for the gated epilogues
// the two-part tensors are [G][M][2][N] and ldc must be 0.
struct GemmExtra {
  int64_t ldc = 0;
  int64_t split_cols = 0;  // kEpiSplit (a multiple of 64)
  bool c_f16 = false;      // the whole output C in fp16 (kEpiStore, kEpiDGelu, kEpiResidual)
  bool ab_f16 = false;     // A and B hold fp16 values (both; tcgen05 kind::f16 takes one type)
  // scratch for split-K partial sums (kEpiStore / kEpiResidual): when it holds
  // gemm_splitk_bytes() and the launch has too few tiles to fill the GPU, the K loop
  // is split in two and the partials added by a second kernel in fixed order
  void* part_ws = nullptr;
  size_t part_ws_bytes = 0;
  int c_sp_S = 0, c_sp_L = 0;  // sequence-sharded rows of C and Yaux (kEpiStore, kEpiResidual)
};
int launch_gemm_bf16(int epi, const GemmOperand& A, const GemmOperand& B, void* C, const void* Yaux,
                     bool store_y, int64_t M, int64_t N, int G, int S, int64_t Ks, unsigned* err,
                     unsigned long long timeout_ns, cudaStream_t stream, int kind,
                     const GemmExtra& extra = GemmExtra());

// Bytes of split-K partials a launch of this shape may use (0: it never splits):
// launches with at most 76 single-CTA tiles of 128 x 256 and at least 32 K blocks.
size_t gemm_splitk_bytes(int64_t M, int64_t N, int G, int S, int64_t Ks);

// 0: choose per launch (CTA pairs unless M <= 128),
// 1: always one CTA per 128 x 256 tile, 2: always a CTA pair per 256 x 256 tile.
// Returns false (and keeps the mode) for another value.
bool set_gemm_tiling_mode(int mode);

}  // namespace tpb
