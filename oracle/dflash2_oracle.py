"""CPU oracle for the DFlash2 draft tail — TEST INFRASTRUCTURE, not part of the product.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
module. It shares no code with the CUDA library: it reads inputs produced by the
``synth`` generator and computes every step directly from its definition, in
float64 unless stated otherwise.

Sources (page title, section):
  [P1] "vLLM adds DFlash2 ..." (ai-jitan-hub news), section "2つの追加要素": the two
       additions — a grouped dynamic depthwise convolution inside each block so a
       proposal position sees the positions before it, and a candidate selector that
       keeps the head's top-K per slot, scores adjacent transitions and walks the best
       path from the verified anchor. Section "追加した仕組みのコストも測っている":
       5 layers, hidden 5120, vocab 248,320, block 8, K=16.
  [P3] "RTX 4090 ... DFlash2 vs MTP" (qiita), section 4: dflash_config
       block_size 8, conv_group_size 16, conv_kernel_size 2, selector_rank 256,
       selector_top_k 16; block_size = 1 + num_speculative_tokens.
  [P4] "DFlash 2: keeping drafts parallel" (hackernews.jp), section
       "軽量パスセレクター" (lightweight path selector): pairwise score
       S_t(a,b) = U_t(b) + <A(a) (.) H(h_t), B(b)> over adjacent candidates, 256-dim
       token embeddings, the walk from the last verified token; section
       "正しいトークンはすでにそこにあります" (Table 1): top-16 candidates per position.

Readings where the pages are silent (each is a fixed choice, stated where used):
  R1 taps: each group's two taps come from a linear projection of the position's
     hidden state and are normalised by a softmax over the two ('softmax' mode);
     'raw' mode uses the projected values unnormalised.
  R2 conv_group_size = channels per group; channel c belongs to group c // 16.
  R3 projection row 2g+0 weights x[t-1], row 2g+1 weights x[t]; no bias.
  R4 layers are chained directly, with no residual, norm or activation between them
     and no norm before the LM head.
  R5 causal within the block, x[-1] = 0, sequences independent.
  R6 all `block` rows are slots; the anchor is the predecessor of slot 0. The other reading
     (first_slot = 1): row 0 of each block is the anchor's own position (the block is 1 +
     the speculative tokens [P3]); its hidden row goes through the conv with the others, so the
     slots see it, and the candidates and the walk cover rows 1..block-1, starting from the
     anchor token.
  R7 per-slot score = log-softmax of the head's logits (this library's contract); the
     pages' raw-logit score gives the same path (per-slot constants cancel).
  R8 the context gate H(h_t) is taken as all-ones by default; with the gate on, H is a
     linear map of the slot's hidden row with no nonlinearity (the pages give none):
     g_t[r] = sum_h z_t[h] * gate_w[r, h], z_t = the slot's conv output (the row the LM
     head reads), gate_w [R, H]. The selector's +2.0M parameters of Table 2 fit one such
     [hidden x 256] map per embedding (3 x 2560 x 256 at the 4B target's hidden 2560).
  R9 the walk is a Viterbi (exact best path); the pages' greedy walk is kept as
     ``greedy_walk``; at temperature T > 0 a path is sampled from the same scores, either
     as a whole (``sample_walk``: P(path) proportional to exp(score / T), forward filtering
     and backward sampling) or step by step along the greedy walk (``greedy_sample_walk``:
     each step drawn from the softmax of that step's scores), with the caller's uniform draws.
  R10 top-K order: logit descending, ties to the lower token id; Viterbi ties go
      to the lower candidate index.
  R12 storage: layer outputs are rounded to the input dtype (bf16 RNE or fp32);
      logits, log-softmax, transitions and path scores are fp32 values.
Decisions that turn floats into integers (the top-K order, every Viterbi and greedy
argmax) are taken in fp32, the precision the CUDA path takes them in: logits are formed
in float64 and rounded once to fp32 before sorting; the Viterbi recursion adds and
compares fp32 values in the order the recursion is written; each greedy step compares
the fp32 sums lp_t(j) + tau_t(j_{t-1}, j). Scores of a chosen path are float64 sums.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

# ---------------------------------------------------------------------------
# storage conversions
# ---------------------------------------------------------------------------


def widen(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) or float32 -> float64, exactly."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def round_bf16(y: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, round to nearest even, taken from the double.

    Written with integer operations on the float64 bit pattern: keep the top 8
    significant bits, round on the 45 dropped bits. Only normal bf16 results occur
    for this path's values; subnormal results are rounded through the exact scaled
    integer.
    """
    y = np.ascontiguousarray(y, dtype=np.float64)
    bits = y.view(np.uint64)
    sign = ((bits >> np.uint64(63)) << np.uint64(15)).astype(np.uint16)
    expo = ((bits >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64)
    mant = (bits & np.uint64((1 << 52) - 1)) | np.uint64(1 << 52)
    q = (mant >> np.uint64(45)).astype(np.int64)
    rem = (mant & np.uint64((1 << 45) - 1)).astype(np.int64)
    half = 1 << 44
    up = (rem > half) | ((rem == half) & ((q & 1) == 1))
    q = q + up
    e = expo - 1023
    carry = q == 256
    q = np.where(carry, 128, q)
    e = np.where(carry, e + 1, e)
    out = (sign.astype(np.int64) | ((e + 127) << 7) | (q & 0x7F)).astype(np.int64)
    # zeros and values below the bf16 normal range
    small = (expo == 0) | (e < -126)
    if np.any(small):
        sub = np.rint(np.abs(y[small]) * 2.0 ** 133).astype(np.int64)  # rint: ties to even
        out[small] = sign[small].astype(np.int64) | sub
    overflow = e > 127
    out = np.where(overflow, sign.astype(np.int64) | 0x7F80, out)
    return out.astype(np.uint16)


def store(y: np.ndarray, dtype: str) -> np.ndarray:
    """Round a float64 layer output to the storage dtype (reading R12)."""
    if dtype == "bf16":
        return round_bf16(y)
    return y.astype(np.float32)


# ---------------------------------------------------------------------------
# (1) grouped dynamic depthwise convolution, kernel size 2  [P1 "2つの追加要素"; P3 §4]
# ---------------------------------------------------------------------------


def conv_layer(x: np.ndarray, w: np.ndarray, group_size: int, taps: str = "softmax") -> np.ndarray:
    """One conv layer on float64 data.

    x: [B, T, H] float64 (one block per sequence), w: [P, H] float64 with P = 2H/group_size.
    For every position t and group g: p = x[t] . w[2g + j] for j = 0, 1 (R3); the taps are
    softmax(p0, p1) (R1); channel c of group g = c // group_size (R2) gets
    y[t, c] = a * x[t-1, c] + b * x[t, c] with x[-1] = 0 (R5). Returns float64 [B, T, H].
    """
    B, T, H = x.shape
    G = H // group_size
    p = x @ w.T  # [B, T, 2G]
    p0 = p[..., 0::2]
    p1 = p[..., 1::2]
    if taps == "softmax":
        mx = np.maximum(p0, p1)
        e0 = np.exp(p0 - mx)
        e1 = np.exp(p1 - mx)
        a = e0 / (e0 + e1)
        b = e1 / (e0 + e1)
    elif taps == "raw":
        a, b = p0, p1
    else:
        raise ValueError(taps)
    a_c = np.repeat(a, group_size, axis=-1)  # [B, T, H]: channel c -> group c // group_size
    b_c = np.repeat(b, group_size, axis=-1)
    x_prev = np.zeros_like(x)
    x_prev[:, 1:, :] = x[:, :-1, :]
    assert a_c.shape[-1] == G * group_size == H
    return a_c * x_prev + b_c * x


def conv_chain(hidden: np.ndarray, conv_w: np.ndarray, dtype: str, group_size: int = 16,
               taps: str = "softmax") -> np.ndarray:
    """All conv layers in order (R4), each output rounded to storage (R12).

    hidden: [B, T, H] storage dtype; conv_w: [NL, P, H] storage dtype. Returns z in
    storage dtype, [B, T, H]. With zero layers z = hidden.
    """
    x = np.asarray(hidden)
    for layer in range(conv_w.shape[0]):
        y = conv_layer(widen(x), widen(conv_w[layer]), group_size, taps)
        x = store(y, dtype)
    return x


# ---------------------------------------------------------------------------
# (2) LM head logits, log-sum-exp, top-K  [P1 "追加した仕組み..."; P3 §4; P4 Table 1]
# ---------------------------------------------------------------------------


def logits(z_rows: np.ndarray, lm_head: np.ndarray, chunk: int = 4096) -> np.ndarray:
    """fp32 logits [M, V]: l[m, v] = sum_h z[m, h] * W[v, h], float64 accumulation,
    rounded once to fp32. The product is taken chunk by chunk over the vocabulary
    only to bound memory; every entry is one float64 dot product."""
    z = widen(z_rows)  # [M, H]
    Vv = lm_head.shape[0]
    out = np.empty((z.shape[0], Vv), dtype=np.float32)
    for v0 in range(0, Vv, chunk):
        w = widen(lm_head[v0:v0 + chunk])  # [c, H]
        out[:, v0:v0 + chunk] = (z @ w.T).astype(np.float32)
    return out


def logsumexp_rows(l32: np.ndarray) -> np.ndarray:
    """lse[m] = max + log(sum_v exp(l - max)) over the fp32 logits, in float64."""
    l = l32.astype(np.float64)
    mx = l.max(axis=1)
    return mx + np.log(np.exp(l - mx[:, None]).sum(axis=1))


def topk_rows(l32: np.ndarray, k: int):
    """Full sort of each row by (logit descending, id ascending); first k (R10)."""
    order = np.argsort(-l32, axis=1, kind="stable")  # stable: equal logits keep id order
    ids = order[:, :k].astype(np.int32)
    vals = np.take_along_axis(l32, order[:, :k], axis=1)
    nxt = np.take_along_axis(l32, order[:, k:k + 1], axis=1)[:, 0] if l32.shape[1] > k else \
        np.full(l32.shape[0], -np.inf, dtype=np.float32)
    return ids, vals, nxt


def cand_logprob(vals32: np.ndarray, lse: np.ndarray) -> np.ndarray:
    """log-softmax of the kept candidates: fp32(l) - fp32(lse), subtracted in fp32 (R7)."""
    return (vals32.astype(np.float32) - lse.astype(np.float32)[..., None]).astype(np.float32)


# ---------------------------------------------------------------------------
# (3) transitions and the walk  [P4 "軽量パスセレクター"]
# ---------------------------------------------------------------------------


def context_gate(z_rows: np.ndarray, gate_w: np.ndarray) -> np.ndarray:
    """The context gate H(h_t) of every slot row (R8): g[m, r] = sum_h z[m, h] * gate_w[r, h],
    float64 dot products of the stored inputs, rounded once to fp32. z_rows [M, H], gate_w [R, H]."""
    return (widen(z_rows) @ widen(gate_w).T).astype(np.float32)


def transitions(anchor: np.ndarray, cand_ids: np.ndarray, U: np.ndarray, V: np.ndarray,
                gate: np.ndarray | None = None) -> np.ndarray:
    """tau [B, T, K, K] fp32. tau[b, 0, i, j] = <U[anchor_b] (.) g_{b,0}, V[c_{b,0,j}]> for every i
    (slot 0's predecessor is the anchor, R6); tau[b, t, i, j] = <U[c_{b,t-1,i}] (.) g_{b,t}, V[c_{b,t,j}]>,
    the pages' <A(a) (.) H(h_t), B(b)> with U = A (previous token) and V = B (current token);
    g_{b,t} = gate[b, t] [R], the gate of the current slot t, or all-ones when gate is None (R8).
    float64 sums of the triple products, rounded once to fp32."""
    B, T, K = cand_ids.shape
    Uw = widen(U)
    Vw = widen(V)
    tau = np.empty((B, T, K, K), dtype=np.float32)
    for b in range(B):
        prev = np.repeat(np.asarray([anchor[b]]), K)
        for t in range(T):
            cur = cand_ids[b, t]
            a = Uw[prev]
            if gate is not None:
                a = a * np.asarray(gate[b, t], dtype=np.float64)[None, :]
            tau[b, t] = (a @ Vw[cur].T).astype(np.float32)
            prev = cur
    return tau


def viterbi(cand_lp: np.ndarray, tau: np.ndarray):
    """Best path per sequence (R9, R10), fp32 arithmetic.

    delta_0(j) = lp_0(j) + tau_0(0, j);
    delta_t(j) = lp_t(j) + max_i [delta_{t-1}(i) + tau_t(i, j)], backpointer = lowest i at the max;
    final state = lowest j at max delta_{T-1}; path read back through the backpointers.
    Returns (path_idx [B,T] int32, score [B] float32).
    """
    B, T, K = cand_lp.shape
    lp = cand_lp.astype(np.float32)
    tau = tau.astype(np.float32)
    path = np.zeros((B, T), dtype=np.int32)
    score = np.zeros(B, dtype=np.float32)
    for b in range(B):
        delta = (lp[b, 0] + tau[b, 0, 0]).astype(np.float32)
        back = np.zeros((T, K), dtype=np.int64)
        for t in range(1, T):
            s = (delta[:, None] + tau[b, t]).astype(np.float32)  # [i, j]
            bp = np.argmax(s, axis=0)  # first index at the max
            back[t] = bp
            delta = (lp[b, t] + s[bp, np.arange(K)]).astype(np.float32)
        j = int(np.argmax(delta))
        score[b] = delta[j]
        for t in range(T - 1, -1, -1):
            path[b, t] = j
            j = int(back[t, j])
    return path, score


def path_score(cand_lp: np.ndarray, tau: np.ndarray, path_idx: np.ndarray) -> np.ndarray:
    """Score of given paths in float64: sum_t lp_t(j_t) + tau_t(j_{t-1}, j_t)."""
    B, T, _ = cand_lp.shape
    out = np.zeros(B, dtype=np.float64)
    for b in range(B):
        s = float(cand_lp[b, 0, path_idx[b, 0]]) + float(tau[b, 0, 0, path_idx[b, 0]])
        for t in range(1, T):
            s += float(cand_lp[b, t, path_idx[b, t]]) + float(tau[b, t, path_idx[b, t - 1], path_idx[b, t]])
        out[b] = s
    return out


def viterbi_two_best(cand_lp: np.ndarray, tau: np.ndarray):
    """Exact best and second-best path scores per sequence (list Viterbi, float64).

    Each state keeps its two best partial scores over distinct paths. Returns
    (best [B], second [B]); margin = best - second (second = -inf when K^T == 1)."""
    B, T, K = cand_lp.shape
    lp = cand_lp.astype(np.float64)
    tt = tau.astype(np.float64)
    best = np.zeros(B)
    second = np.zeros(B)
    for b in range(B):
        top = np.full((K, 2), -np.inf)
        top[:, 0] = lp[b, 0] + tt[b, 0, 0]
        for t in range(1, T):
            new = np.full((K, 2), -np.inf)
            for j in range(K):
                cands = np.concatenate([top[:, 0] + tt[b, t, :, j], top[:, 1] + tt[b, t, :, j]])
                cands = np.sort(cands)[::-1]
                new[j, 0] = lp[b, t, j] + cands[0]
                new[j, 1] = lp[b, t, j] + cands[1]
            top = new
        allv = np.sort(top.reshape(-1))[::-1]
        best[b], second[b] = allv[0], allv[1]
    return best, second


def greedy_walk(cand_lp: np.ndarray, tau: np.ndarray):
    """The pages' walk (R9): from the anchor, take the best successor at each step.

    j_0 = argmax_j lp_0(j) + tau_0(0, j); j_t = argmax_j lp_t(j) + tau_t(j_{t-1}, j), lowest j on
    ties. Each step's candidate scores are fp32 sums, the precision the arg-max is taken in (R12);
    the returned score is the path's score in float64 (``path_score``).
    Returns (path_idx [B,T] int32, score [B] float64)."""
    B, T, K = cand_lp.shape
    lp = cand_lp.astype(np.float32)
    tt = tau.astype(np.float32)
    path = np.zeros((B, T), dtype=np.int32)
    for b in range(B):
        j = 0  # slot 0's predecessor is the anchor: every row of tau_0 is the same
        for t in range(T):
            v = (lp[b, t] + tt[b, t, j]).astype(np.float32)
            j = int(np.argmax(v))
            path[b, t] = j
    return path, path_score(cand_lp, tau, path)


def _inverse_cdf(p: np.ndarray, u: float):
    """Smallest index whose cumulative probability exceeds u (candidates in index order), and the
    distance from u to the nearest interior cumulative boundary (inf for a single candidate)."""
    c = np.cumsum(p)
    k = min(int(np.searchsorted(c, u, side="right")), len(p) - 1)
    near = float(np.min(np.abs(c[:-1] - u))) if len(p) > 1 else np.inf
    return k, near


def greedy_sample_walk(cand_lp: np.ndarray, tau: np.ndarray, temperature: float, u: np.ndarray):
    """The pages' sampling along the walk (R9, [P4] "各ステップで最良の後続を貪欲にたどり、同じスコア
    からサンプリング"): the greedy walk with each step's arg-max replaced by a draw from the same
    step scores at temperature T > 0, in float64:
      j_0 ~ softmax_j ((lp_0(j) + tau_0(0, j)) / T),  j_t ~ softmax_j ((lp_t(j) + tau_t(j_{t-1}, j)) / T),
    each by inverse CDF on u[b, t] (slot t's draw; the smallest index whose cumulative probability
    exceeds it).
    Returns (path_idx [B,T] int32, logprob [B] float64 = sum_t log p_t(j_t), cdf_margin [B] float64 =
    the smallest distance between a draw and a cumulative-probability boundary along the path)."""
    B, T, K = cand_lp.shape
    lp = cand_lp.astype(np.float64)
    tt = tau.astype(np.float64)
    inv_t = 1.0 / float(temperature)
    path = np.zeros((B, T), dtype=np.int32)
    logp = np.zeros(B)
    margin = np.full(B, np.inf)
    for b in range(B):
        j = 0
        for t in range(T):
            s = (lp[b, t] + tt[b, t, j]) * inv_t
            p = np.exp(s - s.max())
            p = p / p.sum()
            j, near = _inverse_cdf(p, float(u[b, t]))
            path[b, t] = j
            logp[b] += np.log(p[j])
            margin[b] = min(margin[b], near)
    return path, logp, margin


def sample_walk(cand_lp: np.ndarray, tau: np.ndarray, temperature: float, u: np.ndarray):
    """A path drawn from the same scores at temperature T > 0 (the pages' sampling mode,
    [P4] "同じスコアからサンプリング"): P(path) = exp(score(path) / T) / Z over the K^T paths of
    the candidate lattice, score(path) = sum_t lp_t(j_t) + tau_t(j_{t-1}, j_t) as in ``viterbi``.

    Forward filtering, then backward sampling, in float64:
      alpha_0(j) = (lp_0(j) + tau_0(0, j)) / T,
      alpha_t(j) = lp_t(j) / T + logsumexp_i (alpha_{t-1}(i) + tau_t(i, j) / T);
      j_{T-1} ~ softmax_j alpha_{T-1}(j);  j_{t-1} ~ softmax_i (alpha_{t-1}(i) + tau_t(i, j_t) / T).
    Each draw takes u[b, t] in [0, 1) (slot t's draw) and picks the smallest index whose cumulative
    probability exceeds it (inverse CDF, candidates in index order).
    Returns (path_idx [B,T] int32, logprob [B] float64 = log P(path), cdf_margin [B] float64 = the
    smallest distance between a draw and a cumulative-probability boundary along the path)."""
    B, T, K = cand_lp.shape
    lp = cand_lp.astype(np.float64)
    tt = tau.astype(np.float64)
    inv_t = 1.0 / float(temperature)
    path = np.zeros((B, T), dtype=np.int32)
    logp = np.zeros(B)
    margin = np.full(B, np.inf)

    def lse(v):
        m = np.max(v)
        return m + np.log(np.sum(np.exp(v - m))) if np.isfinite(m) else m

    def draw(logw, uu):
        p = np.exp(logw - lse(logw))
        k, near = _inverse_cdf(p, uu)
        return k, float(np.log(p[k])), near

    for b in range(B):
        alpha = np.zeros((T, K))
        alpha[0] = (lp[b, 0] + tt[b, 0, 0]) * inv_t
        for t in range(1, T):
            for j in range(K):
                alpha[t, j] = lp[b, t, j] * inv_t + lse(alpha[t - 1] + tt[b, t, :, j] * inv_t)
        j, lpj, near = draw(alpha[T - 1], float(u[b, T - 1]))
        path[b, T - 1] = j
        logp[b] += lpj
        margin[b] = min(margin[b], near)
        for t in range(T - 1, 0, -1):
            i, lpi, near = draw(alpha[t - 1] + tt[b, t, :, j] * inv_t, float(u[b, t - 1]))
            path[b, t - 1] = i
            logp[b] += lpi
            margin[b] = min(margin[b], near)
            j = i
    return path, logp, margin


def log_partition(cand_lp: np.ndarray, tau: np.ndarray, temperature: float) -> np.ndarray:
    """log Z per sequence at temperature T: log sum over the K^T paths of exp(score(path) / T),
    by the forward recursion of ``sample_walk`` in float64 (logsumexp of the last alpha)."""
    B, T, K = cand_lp.shape
    lp = cand_lp.astype(np.float64)
    tt = tau.astype(np.float64)
    out = np.zeros(B)
    for b in range(B):
        a = (lp[b, 0] + tt[b, 0, 0]) / temperature
        for t in range(1, T):
            a = lp[b, t] / temperature + np.logaddexp.reduce(a[:, None] + tt[b, t] / temperature, axis=0)
        out[b] = np.logaddexp.reduce(a)
    return out


def brute_force_best(cand_lp: np.ndarray, tau: np.ndarray):
    """Enumerate all K^T paths of each sequence (tiny K, T only); float64 scores.
    Returns (path_idx [B,T] of the maximum, score [B]); the first path in
    lexicographic order wins exact ties."""
    B, T, K = cand_lp.shape
    assert K ** T <= 2_000_000
    path = np.zeros((B, T), dtype=np.int32)
    best = np.full(B, -np.inf)
    for b in range(B):
        for combo in itertools.product(range(K), repeat=T):
            c = np.asarray(combo)[None, :]
            s = path_score(cand_lp[b:b + 1], tau[b:b + 1], c)[0]
            if s > best[b]:
                best[b] = s
                path[b] = combo
    return path, best


# ---------------------------------------------------------------------------
# the whole tail
# ---------------------------------------------------------------------------


def draft_tail(inp: dict, shape, seqs=None, row_block: int = 256) -> dict:
    """Run the whole tail for the listed sequences (all by default).

    inp: dict from synth.make_inputs; shape: synth.Shape. Returns per-sequence outputs:
    z [b,T,H], cand_ids/cand_lp [b,T,K], lse [b,T] (float64 and fp32), the K-th and
    (K+1)-th logits and max logit per row, tau, path_idx/path_ids/score, the list-Viterbi
    best/second scores.
    """
    B = shape.batch
    seqs = list(range(B)) if seqs is None else list(seqs)
    hidden = np.asarray(inp["hidden"])[seqs]
    z = conv_chain(hidden, inp["conv_w"], shape.dtype, shape.group_size, shape.taps)
    return select_from_z(z, inp, shape, seqs, row_block)


def select_from_z(z: np.ndarray, inp: dict, shape, seqs, row_block: int = 256) -> dict:
    """The tail after the conv, on given conv outputs z [b, T, H] of the listed sequences:
    logits, lse, top-K, transitions from those sequences' anchors, Viterbi and margins.
    With shape.first_slot = 1 (R6) the slots are rows 1..T-1 and every per-slot output has
    T-1 slots."""
    H, K = shape.hidden, shape.top_k
    first = int(getattr(shape, "first_slot", 0))
    T = shape.block - first
    seqs = list(seqs)
    anchor = np.asarray(inp["anchor"])[seqs]
    nb = len(seqs)
    rows = np.asarray(z)[:, first:, :].reshape(nb * T, H)
    M = rows.shape[0]
    ids = np.empty((M, K), dtype=np.int32)
    vals = np.empty((M, K), dtype=np.float32)
    nxt = np.empty(M, dtype=np.float32)
    lmax = np.empty(M, dtype=np.float32)
    lse = np.empty(M, dtype=np.float64)
    for r0 in range(0, M, row_block):
        l32 = logits(rows[r0:r0 + row_block], inp["lm_head"])
        lse[r0:r0 + row_block] = logsumexp_rows(l32)
        i_, v_, n_ = topk_rows(l32, K)
        ids[r0:r0 + row_block], vals[r0:r0 + row_block], nxt[r0:r0 + row_block] = i_, v_, n_
        lmax[r0:r0 + row_block] = l32.max(axis=1)
    lp = cand_logprob(vals, lse).reshape(nb, T, K)
    cids = ids.reshape(nb, T, K)
    gate = context_gate(rows, inp["gate_w"]).reshape(nb, T, -1) if getattr(shape, "gate", False) else None
    tau = transitions(anchor, cids, inp["U"], inp["V"], gate)
    path_idx, score = viterbi(lp, tau)
    path_ids = np.take_along_axis(cids, path_idx[..., None].astype(np.int64), axis=2)[..., 0]
    best, second = viterbi_two_best(lp, tau)
    return dict(z=np.asarray(z), cand_ids=cids, cand_lp=lp, cand_logit=vals.reshape(nb, T, K),
                next_logit=nxt.reshape(nb, T), max_logit=lmax.reshape(nb, T),
                lse=lse.reshape(nb, T), lse32=lse.astype(np.float32).reshape(nb, T),
                tau=tau, gate=gate, path_idx=path_idx, path_ids=path_ids.astype(np.int32), score=score,
                best=best, second=second, seqs=np.asarray(seqs))
