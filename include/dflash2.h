/*
 * dflash2.h — C ABI of the DFlash2 draft tail on one NVIDIA GB300 (sm_103a).
 *
 * The draft tail runs once per verify step of the DFlash2 parallel drafter:
 *   1. a grouped dynamic depthwise convolution inside each block, so a proposal
 *      position sees the positions before it without another backbone pass
 *      ("vLLM adds DFlash2 ...", section "2つの追加要素" (the two additions);
 *      shapes from "RTX 4090 ... DFlash2 vs MTP", section 4, dflash_config:
 *      conv_group_size 16, conv_kernel_size 2);
 *   2. the LM-head contraction, keeping each slot's top-K tokens and its
 *      log-sum-exp (selector_top_k 16, same dflash_config; "DFlash 2: keeping
 *      drafts parallel", section "正しいトークンはすでにそこにあります", Table 1);
 *   3. pairwise transition scores between adjacent slots' candidates through two
 *      rank-R token embeddings, and the best path from the verified anchor
 *      ("DFlash 2: keeping drafts parallel", section "軽量パスセレクター"
 *      (lightweight path selector); selector_rank 256).
 *
 * Conventions for every call:
 *  - All tensor arguments are caller-owned DEVICE pointers to contiguous,
 *    row-major memory. bf16 tensors hold IEEE bfloat16 bit patterns.
 *  - `hidden`, `lm_head`, `U`, `V`, `conv_w`, rows, and the workspace must be
 *    16-byte aligned (they are read by TMA and 128-bit loads).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Every launch is
 *    asynchronous on it; no call synchronises except dflash2_read_device_error.
 *  - The library allocates no memory. Scratch lives in the caller's workspace
 *    `ws` of `ws_bytes` bytes (query dflash2_workspace_size). Zero the
 *    workspace once before its first use (it carries the device error word).
 *    Calls that share a workspace must not overlap in time.
 *  - Argument errors are detected on the host and returned before any launch.
 *    A launch failure returns DFLASH2_ERR_CUDA. Data errors found on the device
 *    (a token id outside [0, vocab), an internal wait that ran out of time) set
 *    bits in the workspace's error word; the kernel clamps and carries on, and
 *    dflash2_read_device_error reports and clears them.
 *  - Supported shapes: hidden % 64 == 0, conv_group_size == 16 (channels per
 *    group), conv_kernel_size == 2, 1 <= top_k <= 16, top_k <= vocab,
 *    rank % 16 == 0 and rank <= 1024, 1 <= block <= 32, batch >= 1,
 *    0 <= conv_layers <= 16. dtype FP32 is a small-size instantiation
 *    (batch*block <= 64, hidden <= 4096).
 */
#ifndef DFLASH2_H
#define DFLASH2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DFLASH2_OK = 0,
  DFLASH2_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, misaligned pointer */
  DFLASH2_ERR_UNSUPPORTED = 2,      /* a shape outside the supported set above */
  DFLASH2_ERR_WORKSPACE_TOO_SMALL = 3,
  DFLASH2_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
  DFLASH2_ERR_DEVICE = 5            /* the device error word is non-zero */
} dflash2_status_t;

typedef enum { DFLASH2_BF16 = 0, DFLASH2_FP32 = 1 } dflash2_dtype_t;

/* shape.flags bits */
enum {
  DFLASH2_CONV_TAPS_SOFTMAX = 0,      /* default: each group's 2 taps are softmax-normalised */
  DFLASH2_CONV_TAPS_RAW = 1u << 0,    /* taps used as projected, unnormalised */
  DFLASH2_WALK_VITERBI = 0,           /* default: exact best path (Viterbi) */
  DFLASH2_WALK_GREEDY = 1u << 1,      /* the pages' greedy walk: best successor at each step */
  DFLASH2_FIRST_SLOT_1 = 1u << 2,     /* row 0 of each block is the anchor's own position */
  DFLASH2_SCORE_LOGITS = 1u << 3      /* whole-tail calls: report the walk's score on raw logits */
};

/* Slots. By default all `block` rows of a sequence are slots and the anchor is the token
 * before slot 0. With DFLASH2_FIRST_SLOT_1 (block >= 2), row 0 of each block is the anchor's
 * own position (the block is 1 + the speculative tokens: "RTX 4090 ... DFlash2 vs MTP",
 * section 4): its hidden row goes through the conv with the others, so the slots see it, and
 * the slots are rows 1..block-1, walked from the anchor token. S = block - 1 slots then, and
 * every per-slot argument of the walk calls (cand_ids, cand_lp, lse, gate, uniforms,
 * path_ids, path_idx) has S slots per sequence instead of block. dflash2_conv and
 * dflash2_select_topk work on all B*block rows either way; the tail's gate output (when
 * requested) holds every row's gate, [B, block, R]. */

/* Device error word bits (dflash2_read_device_error). */
enum {
  DFLASH2_DEVERR_ANCHOR_RANGE = 1 << 0,    /* an anchor id was outside [0, vocab); clamped */
  DFLASH2_DEVERR_CANDIDATE_RANGE = 1 << 1, /* a candidate id was outside [0, vocab); clamped */
  DFLASH2_DEVERR_WAIT_TIMEOUT = 1 << 2     /* an internal pipeline wait ran out of time */
};

typedef struct {
  int32_t batch;            /* B: sequences */
  int32_t block;            /* T: slots per sequence (block_size) */
  int32_t hidden;           /* H: hidden width (5120 on the pages) */
  int32_t vocab;            /* V: vocabulary (248,320 on the pages) */
  int32_t top_k;            /* K: candidates kept per slot (16) */
  int32_t rank;             /* R: selector embedding width (256) */
  int32_t conv_group_size;  /* channels per conv group (16) */
  int32_t conv_kernel_size; /* conv taps (2) */
  int32_t conv_layers;      /* NL: conv layers chained (5) */
  int32_t dtype;            /* dflash2_dtype_t of hidden, lm_head, U, V, conv_w */
  uint32_t flags;           /* DFLASH2_CONV_TAPS_* | DFLASH2_WALK_* | DFLASH2_FIRST_SLOT_1 |
                               DFLASH2_SCORE_LOGITS */
} dflash2_shape_t;

/* Bytes of workspace that every call below needs for `shape` on the current
 * device (one size covers all of them). Returns 0 for an invalid shape. */
size_t dflash2_workspace_size(const dflash2_shape_t* shape);

/* Grouped dynamic depthwise convolution, all conv_layers chained.
 *   x      [B, T, H]              input rows (dtype)
 *   conv_w [NL, 2H/16, H]          per layer, projection row 2g+j gives group g's
 *                                  tap j; tap 0 weights position t-1, tap 1 position t
 *   y      [B, T, H]              output (dtype); may not alias x
 * Per layer, position t and group g: p_j = x[t] . conv_w[l][2g+j];
 * (a, b) = softmax(p_0, p_1) (or (p_0, p_1) with DFLASH2_CONV_TAPS_RAW);
 * y[t, c] = a * x[t-1, c] + b * x[t, c] for the 16 channels c of group g, with
 * x[-1] = 0 inside each sequence's block; each layer's output is rounded to
 * dtype (bf16: round to nearest even) before the next layer. fp32 accumulation. */
dflash2_status_t dflash2_conv(const dflash2_shape_t* shape, const void* x, const void* conv_w,
                              void* y, void* ws, size_t ws_bytes, void* stream);

/* LM-head contraction with per-row top-K and log-sum-exp; the [M, V] logits are
 * never written to memory.
 *   rows     [M, H] (M = B*T)      input rows (dtype)
 *   lm_head  [V, H]                 (dtype)
 *   cand_ids [M, K] int32           top-K token ids, logit descending, ties to the lower id
 *   cand_lp  [M, K] fp32            log-softmax of those tokens: logit - lse (fp32)
 *   lse      [M]    fp32            log sum_v exp(logit[v]); may be NULL
 * Logits are fp32 dot products of the dtype inputs (fp32 accumulation). */
dflash2_status_t dflash2_select_topk(const dflash2_shape_t* shape, const void* rows, const void* lm_head,
                                     int32_t* cand_ids, float* cand_lp, float* lse,
                                     void* ws, size_t ws_bytes, void* stream);

/* Context gate (optional; "DFlash 2: keeping drafts parallel", section "軽量パスセレクター"
 * (lightweight path selector): S_t(a, b) = U_t(b) + <A(a) (.) H(h_t), B(b)>, where the context
 * gate H(h_t) decides which part of the embedding match counts). The pages give no formula for
 * H; here it is a linear map of the slot's hidden row h_t (the row the LM head reads):
 *   gate[m, r] = sum_h rows[m, h] * gate_w[r, h],   gate_w [R, H] (bf16), gate [M, R] fp32,
 * and the gated transition is tau_t(i, j) = sum_r U[prev_i, r] * gate[slot t, r] * V[cur_j, r]
 * (the gate of the current slot t; for t = 0 the anchor is the previous token).
 * The gate is contracted in the LM-head pass itself (its R rows are appended to the head's
 * columns), so it costs no extra pass over the rows. gate_w has the call's dtype. In the walk,
 * V[cur_j, r] * gate[r] is formed in fp32 and split into two bf16 parts (hi = bf16 of the
 * product, lo = bf16 of the remainder; together within about 2^-17 of the fp32 product), and
 * both are contracted with U with fp32 accumulation (fp32 embeddings keep the product in fp32).
 *
 * dflash2_select_topk_gated: dflash2_select_topk plus gate [M, R] fp32 out (gate_w non-NULL;
 * gate_w NULL is dflash2_select_topk, gate ignored). */
dflash2_status_t dflash2_select_topk_gated(const dflash2_shape_t* shape, const void* rows, const void* lm_head,
                                           const void* gate_w, int32_t* cand_ids, float* cand_lp, float* lse,
                                           float* gate, void* ws, size_t ws_bytes, void* stream);

/* dflash2_select_topk without a workspace argument and without any allocation, for callers
 * that cannot obtain device memory at the point of the call: a plugin inside a serving
 * engine that has already reserved the whole GPU for its own pools and exposes no
 * allocator, code that runs while a CUDA graph is being captured (where cudaMalloc is not
 * allowed), or a latency-critical loop that must not risk the implicit device
 * synchronisation an allocation can cause. No counterpart in the DFlash2 pages: it is the
 * same selection as dflash2_select_topk (same kernels, same results), with its scratch in a
 * fixed 4 MiB device array inside the library instead of the caller's workspace.
 *  - Every GPU that loads the library holds those 4 MiB until the process exits.
 *  - The first call on each device looks up the array's device address (with that device
 *    current); make that first call before any stream capture that includes this call.
 *  - Shapes whose partials need more than 4 MiB (parts * rows * 136 bytes + 256, where
 *    parts is about the SM count divided by ceil(rows / 128)) return
 *    DFLASH2_ERR_WORKSPACE_TOO_SMALL before any launch.
 *  - All calls share the array: calls that may overlap on the GPU (different streams, or
 *    different host threads) race with each other and must be serialised by the caller.
 *  - Each call clears the array's error word first; device-side errors of this call are
 *    not reported (there is no workspace to read them from). */
dflash2_status_t dflash2_select_topk_noalloc(const dflash2_shape_t* shape, const void* rows, const void* lm_head,
                                             int32_t* cand_ids, float* cand_lp, float* lse, void* stream);

/* The two stages of dflash2_select_topk, callable on their own (e.g. to time the
 * contraction, or to merge partials that the caller gathered from several vocab shards).
 * dflash2_lmhead_partials runs the LM-head contraction with its fused epilogue and leaves,
 * in the workspace, one partial per (row, column partition): that partition's top-16
 * (logit desc, id asc) and its (max logit, sum of exp(logit - max)).
 * dflash2_merge_partials turns the workspace's partials into cand_ids, cand_lp and lse
 * exactly as dflash2_select_topk does. Both take the same shape and workspace. */
dflash2_status_t dflash2_lmhead_partials(const dflash2_shape_t* shape, const void* rows, const void* lm_head,
                                         void* ws, size_t ws_bytes, void* stream);
dflash2_status_t dflash2_merge_partials(const dflash2_shape_t* shape, int32_t* cand_ids, float* cand_lp,
                                        float* lse, void* ws, size_t ws_bytes, void* stream);

/* Transition scores and the walk from the anchor.
 *   anchor   [B] int32              verified token preceding slot 0 of each sequence
 *   cand_ids [B, T, K] int32, cand_lp [B, T, K] fp32   (as from dflash2_select_topk)
 *   U, V     [V, R] (dtype)         U embeds the previous token, V the current one
 *   path_ids [B, T] int32           chosen token per slot
 *   path_idx [B, T] int32           chosen candidate index per slot
 *   score    [B] fp32               path score
 * tau_0(j) = <U[anchor], V[c_{0,j}]>, tau_t(i, j) = <U[c_{t-1,i}], V[c_{t,j}]>;
 * Viterbi (default): delta_0(j) = lp_0(j) + tau_0(j),
 * delta_t(j) = lp_t(j) + max_i (delta_{t-1}(i) + tau_t(i, j)), fp32, every
 * argmax taking the lowest index; score = max_j delta_{T-1}(j).
 * Greedy (DFLASH2_WALK_GREEDY): j_t = argmax_j (lp_t(j) + tau_t(j_{t-1}, j)),
 * score accumulated along the path in the same order as the Viterbi recursion.
 * DFLASH2_SCORE_LOGITS is accepted only by the whole-tail calls (the walk calls here, which take
 * log-probabilities, return DFLASH2_ERR_UNSUPPORTED with it). */
dflash2_status_t dflash2_viterbi(const dflash2_shape_t* shape, const int32_t* anchor,
                                 const int32_t* cand_ids, const float* cand_lp,
                                 const void* U, const void* V,
                                 int32_t* path_ids, int32_t* path_idx, float* score,
                                 void* ws, size_t ws_bytes, void* stream);

/* dflash2_viterbi with the context gate: gate [B, T, R] fp32 (16-byte aligned) is each slot's
 * gate row as above; NULL is dflash2_viterbi. */
dflash2_status_t dflash2_viterbi_gated(const dflash2_shape_t* shape, const int32_t* anchor,
                                       const int32_t* cand_ids, const float* cand_lp,
                                       const void* U, const void* V, const float* gate,
                                       int32_t* path_ids, int32_t* path_idx, float* score,
                                       void* ws, size_t ws_bytes, void* stream);

/* A path sampled at temperature T > 0 instead of the best one ("DFlash 2: keeping drafts
 * parallel", section "軽量パスセレクター": the walk can also sample from the same scores).
 * Two forms, by the shape's walk flag.
 * Default (Viterbi flag): the whole path is drawn from the path distribution,
 * P(path) = exp(score(path) / T) / Z over the K^T paths, score(path) as for dflash2_viterbi
 * (with the context gate when gate is non-NULL, as in dflash2_viterbi_gated). Forward filtering
 * in fp32, alpha_0(j) = (lp_0(j) + tau_0(j)) / T, alpha_t(j) = lp_t(j) / T +
 * logsumexp_i (alpha_{t-1}(i) + tau_t(i, j) / T); then backward draws: j_{T-1} ~ softmax(alpha_{T-1}),
 * j_{t-1} ~ softmax_i (alpha_{t-1}(i) + tau_t(i, j_t) / T), each the smallest candidate index
 * whose cumulative probability exceeds uniforms[b, t] (slot t's draw, in [0, 1)).
 * DFLASH2_WALK_GREEDY: the pages' walk with each step's arg-max replaced by a draw from the same
 * step scores: j_0 ~ softmax_j ((lp_0(j) + tau_0(j)) / T), j_t ~ softmax_j ((lp_t(j) +
 * tau_t(j_{t-1}, j)) / T), each the smallest index whose cumulative probability exceeds
 * uniforms[b, t]; score receives sum_t log p_t(j_t), the log-probability of the drawn path.
 *   temperature > 0 (finite); uniforms [B, T] fp32 device: the caller's random numbers
 *   (the library draws none, so a result is reproducible from its inputs)
 *   score [B] fp32 receives log P(path) of the drawn path.
 * uniforms NULL: the Viterbi / greedy walk (temperature ignored). */
dflash2_status_t dflash2_sample_walk(const dflash2_shape_t* shape, const int32_t* anchor,
                                     const int32_t* cand_ids, const float* cand_lp,
                                     const void* U, const void* V, const float* gate,
                                     float temperature, const float* uniforms,
                                     int32_t* path_ids, int32_t* path_idx, float* score,
                                     void* ws, size_t ws_bytes, void* stream);

/* The whole tail in one call: conv -> LM head top-K + lse -> transitions + walk.
 *   hidden [B, T, H], lm_head [V, H], U/V [V, R], conv_w [NL, 2H/16, H], anchor [B]
 *   path_ids, path_idx [B, T] int32; score [B] fp32
 *   cand_ids [B, T, K], cand_lp [B, T, K], lse [B, T]: optional copies of the
 *   intermediate candidates (NULL to skip).
 * With DFLASH2_SCORE_LOGITS the Viterbi / greedy score is reported on the head's raw logits
 * (the pages' per-slot score is the drafter's own logit, "DFlash 2: keeping drafts parallel",
 * section "軽量パスセレクター"): sum_t logit_t(j_t) + transitions = the log-softmax score plus
 * sum_t lse_t, summed in fp32. The path is the same under either score (per-slot constants do
 * not move an arg-max); a sampled walk's score stays log P(path). */
dflash2_status_t dflash2_draft_tail(const dflash2_shape_t* shape, const void* hidden, const void* lm_head,
                                    const void* U, const void* V, const void* conv_w,
                                    const int32_t* anchor, int32_t* path_ids, int32_t* path_idx,
                                    float* score, int32_t* cand_ids, float* cand_lp, float* lse,
                                    void* ws, size_t ws_bytes, void* stream);

/* dflash2_draft_tail with the context gate: gate_w [R, H] (bf16) as above; the gate rows are
 * formed in the LM-head pass from the conv output and applied in the walk. gate [B, T, R] fp32
 * receives them (NULL: kept in the workspace only). gate_w NULL is dflash2_draft_tail. */
dflash2_status_t dflash2_draft_tail_gated(const dflash2_shape_t* shape, const void* hidden, const void* lm_head,
                                          const void* U, const void* V, const void* conv_w, const void* gate_w,
                                          const int32_t* anchor, int32_t* path_ids, int32_t* path_idx,
                                          float* score, int32_t* cand_ids, float* cand_lp, float* lse,
                                          float* gate, void* ws, size_t ws_bytes, void* stream);

/* dflash2_draft_tail_gated with the walk sampling at temperature T > 0 from the caller's
 * uniforms [B, T] (as dflash2_sample_walk; score receives log P(path)); gate_w may be NULL
 * (no context gate); uniforms NULL is dflash2_draft_tail_gated. */
dflash2_status_t dflash2_draft_tail_sampled(const dflash2_shape_t* shape, const void* hidden, const void* lm_head,
                                            const void* U, const void* V, const void* conv_w, const void* gate_w,
                                            const int32_t* anchor, float temperature, const float* uniforms,
                                            int32_t* path_ids, int32_t* path_idx, float* score,
                                            int32_t* cand_ids, float* cand_lp, float* lse, float* gate,
                                            void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, returns the workspace's device error word in *code_out
 * (a DFLASH2_DEVERR_* bit set; 0 = none) and clears it. Returns DFLASH2_OK, or
 * DFLASH2_ERR_CUDA if the copy failed. */
dflash2_status_t dflash2_read_device_error(void* ws, void* stream, int32_t* code_out);

/* Static description of a status code. */
const char* dflash2_status_string(dflash2_status_t status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t dflash2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_H */
