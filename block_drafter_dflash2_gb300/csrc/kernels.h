// Internal launchers shared by the C-ABI layer (api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tc_gemm_args.h"

namespace df {

// tcgen05 GEMM + top-K/lse partials (bf16). grid = n_rc * parts.
// g128 / g16: 128- and 16-row box maps of the gate matrix (any valid maps when
// args.gate_cols == 0; g128 is used only when gate_cols >= 128); vocab: the ranked columns;
// gate_out [M, gate_cols] fp32 receives the gate columns.
cudaError_t launch_lmhead_topk_bf16(const CUtensorMap& a, const CUtensorMap& a_tail, const CUtensorMap& b128,
                                    const CUtensorMap& b16, const CUtensorMap& g128, const CUtensorMap& g16,
                                    const TcGemmArgs& args, int vocab, float* part_val, int32_t* part_id,
                                    float* part_ms, float* gate_out, cudaStream_t s);

// tcgen05 GEMM + conv-layer epilogue (bf16): y = mix(x) with taps = x * W^T.
cudaError_t launch_conv_layer_bf16(const CUtensorMap& a, const CUtensorMap& a_tail, const CUtensorMap& b128,
                                   const CUtensorMap& b16,
                                   const TcGemmArgs& args, const void* x, void* y, int T, int raw,
                                   cudaStream_t s);

// All conv layers in one cooperative launch (bf16, hidden % 256 == 0): row blocks x group
// blocks of CTAs, mma.sync taps; conv_chain_plan picks the kernel variant and the grid for the
// device's SM count (false if no variant fits). Zeroes the row blocks' barrier counters first.
struct ConvChainPlan {
  int variant;       // kernel instantiation
  int row_blocks;    // blocks of 16 or 64 rows
  int group_blocks;  // CTAs per row block, each owning a range of channel groups
  int wtaps;         // the most projection rows one CTA owns
  size_t smem;       // dynamic shared memory per CTA
};
bool conv_chain_plan(int M, int H, int sms, ConvChainPlan* out);
cudaError_t launch_conv_chain(const ConvChainPlan& pl, const void* x, const void* conv_w, void* buf0, void* buf1,
                              void* z, int M, int H, int T, int NL, int raw, unsigned* bar_counts, int32_t* err,
                              cudaStream_t s);

// All conv layers in one cooperative launch for larger row counts (bf16, hidden % 64 == 0):
// CTAs = row tiles (128 rows) x tap tiles x K-slices; tcgen05 partial taps per K-slice, summed
// after a grid barrier and fused with the mix. conv_splitk_plan sizes the grid for the SM count
// (false if the row tiles do not fit); part_bytes of workspace hold the partial taps.
struct ConvSplitPlan {
  int RT, NT, KS;      // row tiles, tap tiles, K-slices
  int Nt;              // projection rows per tap tile
  int a_tail_rows;     // TMA box rows of the last row tile
  int Mp;              // rows of a partial-tap plane (M rounded up to 4)
  int grid;            // RT * NT * KS CTAs
  size_t smem;         // dynamic shared memory per CTA
  size_t part_bytes;   // workspace for the partial taps, [2][KS][H/8][Mp] fp32
  int gc;              // channel groups per mix chunk
  int br;              // rows of the partial-tap and row boxes (128, or a single tile's rows)
  int xb, nxs;         // channels of a mix row box (br rows), row boxes per chunk
  uint32_t pbox_bytes, xbox_bytes;  // a chunk's partial-tap box; one row box
  int x_early;         // row boxes in their own region, loaded as each layer starts
  uint32_t xoff;       // byte offset of the row boxes from the operand ring
  uint32_t aboff;      // byte offset of the row above the tile ([gc][16] bf16) from the ring
};
bool conv_splitk_plan(int M, int H, int NL, int sms, ConvSplitPlan* out);
// maps: 0-5 the x operand (128-row box, tail box) of x, buf0, buf1 (128-B swizzle, 64 columns);
// 6 all layers' weights [NL * H/8, H] (Nt-row box); 7 the partial taps [2 KS][H/8][Mp] fp32
// with a (br, Nt, 1) box, 8 the same with a (br, 2 gc, KS) box; 9-11 the mix row boxes
// (xb columns, br rows, no swizzle) of x, buf0, buf1. Zeroes the barrier counters first.
cudaError_t launch_conv_splitk(const ConvSplitPlan& pl, const CUtensorMap* maps, const void* x, void* buf0,
                               void* buf1, void* z, int M, int H, int T, int NL, int raw, unsigned* bar_counts,
                               int32_t* err, cudaStream_t s);

// fp32 instantiations (small sizes).
cudaError_t launch_conv_layer_f32(const float* x, const float* w, float* y, int M, int H, int T, int raw,
                                  cudaStream_t s);
cudaError_t launch_lmhead_topk_f32(const float* z, const float* w, const float* gate_w, const TcGemmArgs& args,
                                   float* part_val, int32_t* part_id, float* part_ms, float* gate_out,
                                   cudaStream_t s);

// Merge of the per-partition top-16 lists and (max, sum) pairs -> top-K, log-probs, lse.
cudaError_t launch_topk_merge(const float* part_val, const int32_t* part_id, const float* part_ms, int parts,
                              int M, int K, int32_t* cand_ids, float* cand_lp, float* lse, cudaStream_t s);

// Merge of the partials fused with the transition tiles and the walk, one CTA per sequence
// (the whole-tail call); cand_ids / cand_lp / lse may be null. Needs select_walk_smem(parts)
// bytes of shared memory (at most 227 KB).
size_t select_walk_smem(int parts);
// T slots per sequence at rows first .. first+T-1 of the sequence's rows_per_seq LM-head rows
// (per-slot outputs); gate: [B*rows_per_seq, R] fp32 context gate of every row, or nullptr.
// walk_flags: kWalkFlagGreedy (the greedy walk; with uniforms, per-step draws along it) |
// kWalkFlagScoreLogits (the Viterbi / greedy score on raw logits: plus the slots' lse).
constexpr int kWalkFlagGreedy = 1;
constexpr int kWalkFlagScoreLogits = 2;
cudaError_t launch_select_walk(bool bf16, const float* part_val, const int32_t* part_id, const float* part_ms,
                               int parts, int M, const int32_t* anchor, const void* U, const void* V,
                               const float* gate, int B, int T, int rows_per_seq, int first, int K, int R,
                               int vocab, int walk_flags, const float* uniforms, float inv_temp, int32_t* cand_ids,
                               float* cand_lp, float* lse, int32_t* path_ids, int32_t* path_idx, float* score,
                               int32_t* err, cudaStream_t s);

// Transition tiles + Viterbi / greedy walk, one CTA per sequence. uniforms [B, T] (nullptr: no
// sampling) and inv_temp: draw a path at temperature 1 / inv_temp instead. Slot t's candidates
// (and gate row, and lse_rows entry) are row first + t of the sequence's cand_rows rows; outputs
// are per slot. lse_rows (nullable) is read only with kWalkFlagScoreLogits.
cudaError_t launch_transition_walk(bool bf16, const int32_t* anchor, const int32_t* cand_ids,
                                   const float* cand_lp, const void* U, const void* V, const float* gate,
                                   const float* lse_rows, int B, int T, int cand_rows, int first, int K, int R,
                                   int vocab, int walk_flags,
                                   const float* uniforms, float inv_temp, int32_t* path_ids, int32_t* path_idx,
                                   float* score, int32_t* err, cudaStream_t s);

}  // namespace df
