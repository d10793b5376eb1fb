"""Parity harness: runs the CUDA library through its C ABI and compares it with the oracle.

Tolerances (from the draft-tail contract): token ids and paths bit-exact except at
near-ties; lse, candidate log-probs and path scores within 2e-3 absolute; conv outputs
within 1e-2 relative.

Each step is compared with the oracle on that step's own input, so that a legitimate
difference upstream is not counted against a later step: the conv output z against the
oracle's conv; the LM-head selection against the oracle run on the GPU's own z (a bf16 ulp
of difference in z moves a logit by ~1e-3, more than the near-tie band); the walk exactly on
the GPU's own candidates. Agreement with the oracle end to end (the GPU's results against the
oracle run on its own conv output) is asserted as well, under the same near-tie rules.

With the context gate, the gate rows are compared with the oracle's H(h_t) of the GPU's own
conv output within 1e-3 absolute (they are O(1)), and the walk is checked on the GPU's own
candidates and gate rows.

Near-tie rules used here:
  * top-K: the GPU's k-th candidate may differ from the oracle's k-th only if the two
    tokens' oracle logits lie within 1e-3 * |max logit| of each other (at the K/K+1
    boundary this is the set-membership tie; inside the list, an order swap);
  * paths: the walk is checked exactly on the GPU's own candidates (the oracle Viterbi
    re-run on them), and against the full oracle path when the sequence had no top-K
    near-tie; either comparison may differ only when the oracle's best/second-best margin
    is below 1e-2.
"""
from __future__ import annotations

import numpy as np
import torch

import block_drafter_dflash2_gb300 as df2
from oracle import core as O

LSE_TOL = 2e-3
LP_TOL = 2e-3
SCORE_TOL = 2e-3
CONV_RTOL = 1e-2
TIE_REL = 1e-3
MARGIN = 1e-2
GATE_TOL = 1e-3


def shape_of(sh, greedy=False) -> df2.Shape:
    return df2.Shape.make(sh.batch, sh.block, sh.hidden, sh.vocab, sh.top_k, sh.rank, sh.layers,
                          dtype=sh.dtype, raw_taps=(sh.taps == "raw"), greedy=greedy,
                          first_slot=getattr(sh, "first_slot", 0))


def dev(a: np.ndarray) -> torch.Tensor:
    """Upload a numpy array (bf16 bit patterns travel as int16) to cuda:0."""
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")


def host(t: torch.Tensor, like=None) -> np.ndarray:
    a = t.cpu().numpy()
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    return a


def workspace(shape: df2.Shape) -> torch.Tensor:
    n = df2.workspace_size(shape)
    assert n > 0
    return torch.zeros(n, dtype=torch.uint8, device="cuda:0")


def upload_inputs(inp: dict) -> dict:
    return {k: dev(v) for k, v in inp.items()
            if v is not None and k in ("hidden", "lm_head", "U", "V", "conv_w", "anchor", "gate_w")}


def run_tail(shape: df2.Shape, d: dict, ws=None, stream=None, gated=False) -> dict:
    """The whole tail through dflash2_draft_tail, or dflash2_draft_tail_gated (gate rows out).
    Per-slot outputs have S = block - first slots (first = 1 with DFLASH2_FIRST_SLOT_1); the gate
    rows cover every row."""
    B, T, K = shape.batch, shape.block, shape.top_k
    S = T - (1 if shape.flags & df2.FIRST_SLOT_1 else 0)
    o = {
        "path_ids": torch.empty((B, S), dtype=torch.int32, device="cuda:0"),
        "path_idx": torch.empty((B, S), dtype=torch.int32, device="cuda:0"),
        "score": torch.empty((B,), dtype=torch.float32, device="cuda:0"),
        "cand_ids": torch.empty((B, S, K), dtype=torch.int32, device="cuda:0"),
        "cand_lp": torch.empty((B, S, K), dtype=torch.float32, device="cuda:0"),
        "lse": torch.empty((B, S), dtype=torch.float32, device="cuda:0"),
    }
    ws = workspace(shape) if ws is None else ws
    if gated:
        o["gate"] = torch.empty((B, T, shape.rank), dtype=torch.float32, device="cuda:0")
        df2.draft_tail_gated(shape, d["hidden"], d["lm_head"], d["U"], d["V"], d["conv_w"], d["gate_w"], d["anchor"],
                             o["path_ids"], o["path_idx"], o["score"], ws, cand_ids=o["cand_ids"],
                             cand_lp=o["cand_lp"], lse=o["lse"], gate=o["gate"], stream=stream)
    else:
        df2.draft_tail(shape, d["hidden"], d["lm_head"], d["U"], d["V"], d["conv_w"], d["anchor"], o["path_ids"],
                       o["path_idx"], o["score"], ws, cand_ids=o["cand_ids"], cand_lp=o["cand_lp"], lse=o["lse"],
                       stream=stream)
    torch.cuda.synchronize()
    err = df2.read_device_error(ws)
    out = {k: host(v) for k, v in o.items()}
    out["device_error"] = err
    # the conv output the tail used (the library is deterministic: same kernels, same inputs)
    z = torch.empty_like(d["hidden"])
    df2.conv(shape, d["hidden"], d["conv_w"], z, ws, stream=stream)
    torch.cuda.synchronize()
    out["z"] = host(z)
    out["z_layers"] = run_conv_layers(shape, d["hidden"], d["conv_w"])
    return out


def run_conv_layers(shape: df2.Shape, x: torch.Tensor, conv_w: torch.Tensor) -> list:
    """The conv chain one layer per dflash2_conv call (each call on the previous call's output):
    the per-layer outputs, host arrays. The chain's kernels apply the same per-layer arithmetic
    whatever the layer count, so the last one equals the whole chain's output bit for bit."""
    one = df2.Shape.make(shape.batch, shape.block, shape.hidden, shape.vocab, shape.top_k, shape.rank, 1,
                         dtype=shape.dtype, raw_taps=bool(shape.flags & df2.CONV_TAPS_RAW))
    ws = workspace(one)
    outs = []
    cur = x
    for l in range(conv_w.shape[0]):
        y = torch.empty_like(x)
        df2.conv(one, cur, conv_w[l:l + 1], y, ws)
        outs.append(y)
        cur = y
    torch.cuda.synchronize()
    assert df2.read_device_error(ws) == 0
    return [host(y) for y in outs]


def run_conv(shape: df2.Shape, x: torch.Tensor, conv_w: torch.Tensor) -> np.ndarray:
    y = torch.empty_like(x)
    ws = workspace(shape)
    df2.conv(shape, x, conv_w, y, ws)
    torch.cuda.synchronize()
    assert df2.read_device_error(ws) == 0
    return host(y)


def run_topk(shape: df2.Shape, rows: torch.Tensor, lm_head: torch.Tensor):
    M, K = shape.batch * shape.block, shape.top_k
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda:0")
    lp = torch.empty((M, K), dtype=torch.float32, device="cuda:0")
    lse = torch.empty((M,), dtype=torch.float32, device="cuda:0")
    ws = workspace(shape)
    df2.select_topk(shape, rows, lm_head, ids, lp, lse, ws)
    torch.cuda.synchronize()
    assert df2.read_device_error(ws) == 0
    return host(ids), host(lp), host(lse)


def run_viterbi(shape: df2.Shape, anchor, cand_ids, cand_lp, U, V, gate=None):
    """dflash2_viterbi, or dflash2_viterbi_gated when gate [B,S,R] fp32 is given (S slots:
    block, or block - 1 with DFLASH2_FIRST_SLOT_1)."""
    B = shape.batch
    T = shape.block - (1 if shape.flags & df2.FIRST_SLOT_1 else 0)
    pid = torch.empty((B, T), dtype=torch.int32, device="cuda:0")
    pix = torch.empty((B, T), dtype=torch.int32, device="cuda:0")
    sc = torch.empty((B,), dtype=torch.float32, device="cuda:0")
    ws = workspace(shape)
    if gate is None:
        df2.viterbi(shape, anchor, cand_ids, cand_lp, U, V, pid, pix, sc, ws)
    else:
        df2.viterbi_gated(shape, anchor, cand_ids, cand_lp, U, V, gate, pid, pix, sc, ws)
    torch.cuda.synchronize()
    err = df2.read_device_error(ws)
    return host(pid), host(pix), host(sc), err


# ------------------------------------------------------------------ comparators


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Unit in the last place of bf16 at magnitude v (8 significant bits): 2^(floor(log2 v) - 7)."""
    v = np.maximum(np.abs(v), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(v)) - 7)


def conv_cone_scale(layer_inputs: list) -> np.ndarray:
    """Per output element, the largest magnitude any layer's input takes over the positions the
    element depends on (layer l's y[t] reads x_l[t-1] and x_l[t] of the same channel):
    S_0 = max(|x_0[t]|, |x_0[t-1]|), S_l[t] = max(|x_l[t]|, |x_l[t-1]|, S_{l-1}[t], S_{l-1}[t-1])."""
    S = None
    for x in layer_inputs:
        a = np.abs(O.widen(x))
        ap = np.zeros_like(a)
        ap[:, 1:] = a[:, :-1]
        cur = np.maximum(a, ap)
        if S is not None:
            Sp = np.zeros_like(S)
            Sp[:, 1:] = S[:, :-1]
            cur = np.maximum(cur, np.maximum(S, Sp))
        S = cur
    return S


def check_conv(z_gpu: np.ndarray, z_ref: np.ndarray, x_last=None, one_layer=False, min_exact=0.95,
               max_norm_rel=2e-3, cone=None, layers=1):
    """Conv outputs within 1e-2 relative, per element, |gpu - ref| <= 1e-2 * max(|ref|, rms of the ref
    row), the scale floored as follows.

    One layer (`one_layer`, x_last = that layer's input): every element is bounded by
    2^-7 * max(|x[t-1]|, |x[t]|), two bf16 units of the operands at most (the output rounding plus
    the tap error), and bf16 outputs must be bit-identical in at least `min_exact` of the elements.
    Several layers against the oracle's own chain (`cone` = conv_cone_scale of the oracle's layer
    inputs): two results that are each correctly rounded to bf16 at every layer drift apart: where
    the fp32 and float64 values of a layer fall on either side of a rounding boundary they differ by
    one unit, later layers carry it (convex combinations: not amplified) and every later tap moves
    by ~1e-4, which makes more such straddles. So the floor is (layers + 1) bf16 units of the largest
    magnitude on the element's dependency cone; the whole output must still be within
    `max_norm_rel` in 2-norm and bf16 outputs bit-identical in at least `min_exact` of the elements.
    fp32 outputs take the relative bound alone (floored at 1e-2 of the operands)."""
    bf16 = z_gpu.dtype == np.uint16
    g = O.widen(z_gpu).reshape(-1, z_gpu.shape[-1])
    r = O.widen(z_ref).reshape(-1, z_ref.shape[-1])
    rms = np.sqrt(np.mean(r * r, axis=1, keepdims=True))
    bound = CONV_RTOL * np.maximum(np.abs(r), rms)
    op = None
    if x_last is not None:
        x = O.widen(x_last)
        xp = np.zeros_like(x)
        xp[:, 1:] = x[:, :-1]
        op = np.maximum(np.abs(x), np.abs(xp)).reshape(g.shape)
        bound = np.maximum(bound, CONV_RTOL * op if not bf16 else 0.0)
    if cone is not None and bf16:
        bound = np.maximum(bound, (layers + 1) * bf16_ulp(np.maximum(cone.reshape(g.shape), np.abs(r))))
    bad = np.abs(g - r) > bound
    assert not bad.any(), f"conv: {bad.sum()} of {bad.size} elements outside the bound; " \
                          f"max abs diff {np.abs(g - r).max():.3e}"
    row_err = np.linalg.norm(g - r, axis=1) / np.maximum(np.linalg.norm(r, axis=1), 1e-30)
    exact = float((g == r).mean())
    norm_rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    if bf16:
        assert exact >= min_exact, f"conv: only {exact:.4f} of the elements bit-identical"
    assert norm_rel <= max_norm_rel, f"conv: 2-norm relative error {norm_rel:.3e}"
    rep = {"conv_exact_frac": exact, "conv_max_abs": float(np.abs(g - r).max()),
           "conv_row_rel_max": float(row_err.max()), "conv_norm_rel": norm_rel,
           "conv_bound_used_max": float((np.abs(g - r) / np.maximum(bound, 1e-30)).max())}
    if one_layer:
        over = np.abs(g - r) > 2.0 ** -7 * op + 1e-30
        assert not over.any(), f"conv: {over.sum()} elements beyond 2 operand ulps"
        rep["conv_operand_ulps_max"] = float((np.abs(g - r) / np.maximum(op, 1e-30)).max() * 2 ** 8)
    return rep


def check_conv_layers(hidden, conv_w, dtype, taps, z_layers, z_chain, ref_chain=None):
    """Each GPU layer against the oracle's layer on the GPU's own input of that layer (the one-layer
    bound); the whole chain's output equal bit for bit to the last per-layer output; and, given the
    oracle's own chain output, the chain against it with the multi-layer bound."""
    L = conv_w.shape[0]
    rep = {}
    x = hidden
    worst_exact = 1.0
    for l in range(L):
        ref_l = O.conv_chain(x, conv_w[l:l + 1], dtype, 16, taps)
        r = check_conv(z_layers[l], ref_l, x_last=x, one_layer=True, min_exact=0.99)
        worst_exact = min(worst_exact, r["conv_exact_frac"])
        rep["conv_layer_operand_ulps_max"] = max(rep.get("conv_layer_operand_ulps_max", 0.0),
                                                 r["conv_operand_ulps_max"])
        x = z_layers[l]
    rep["conv_layer_exact_min"] = worst_exact
    if L:
        assert np.array_equal(z_layers[-1], z_chain), "conv: the chain differs from its layer-by-layer composition"
    if ref_chain is not None and L:
        ins = [hidden]
        for l in range(L - 1):
            ins.append(O.conv_chain(ins[-1], conv_w[l:l + 1], dtype, 16, taps))
        # (bit-identical fractions of the chain fall with the block length as straddles cascade:
        # 0.944 measured at block 16 with 5 layers; each layer on its own input stays above 0.99)
        rep.update(check_conv(z_chain, ref_chain, cone=conv_cone_scale(ins), layers=L, min_exact=0.90))
    return rep


def check_topk(ref: dict, g_ids, g_lp, g_lse, z_rows, lm_head, K, lse_allow=None, lp_allow=None):
    """ref: oracle outputs flattened to rows (cand_ids [M,K], cand_logit, max_logit, lse).
    lse_allow / lp_allow [M] (end to end only): what the conv's difference alone moves each row's
    lse and candidate log-probs by, computed by the oracle on both conv outputs; added to the
    tolerances."""
    M = g_ids.shape[0]
    o_ids = ref["cand_ids"].reshape(M, K)
    o_val = ref["cand_logit"].reshape(M, K)
    o_max = ref["max_logit"].reshape(M)
    o_lse = ref["lse"].reshape(M)
    lse_allow = np.zeros(M) if lse_allow is None else np.asarray(lse_allow).reshape(M)
    lp_allow = np.zeros(M) if lp_allow is None else np.asarray(lp_allow).reshape(M)
    lse_err = np.abs(g_lse.reshape(M).astype(np.float64) - o_lse)
    over = lse_err - lse_allow
    assert over.max() <= LSE_TOL, f"lse error {lse_err[np.argmax(over)]:.3e} (allowance {lse_allow[np.argmax(over)]:.3e})"
    tie_rows = []
    lp_err = 0.0
    for m in range(M):
        band = TIE_REL * abs(float(o_max[m]))
        if np.array_equal(g_ids[m], o_ids[m]):
            lg = o_val[m]
        else:
            assert len(set(g_ids[m].tolist())) == K, f"row {m}: repeated ids {g_ids[m]}"
            assert np.all((g_ids[m] >= 0) & (g_ids[m] < lm_head.shape[0])), f"row {m}: id out of range"
            lg = O.logits(z_rows[m:m + 1], lm_head[g_ids[m]])[0]
            gap = np.abs(lg.astype(np.float64) - o_val[m].astype(np.float64))
            assert gap.max() <= band, f"row {m}: ids {g_ids[m]} vs {o_ids[m]}, logit gap {gap.max():.3e} > {band:.3e}"
            tie_rows.append(m)
        e = np.abs(g_lp[m].astype(np.float64) - (lg.astype(np.float64) - o_lse[m])).max()
        assert e <= LP_TOL + lp_allow[m], f"row {m}: cand_lp error {e:.3e} (allowance {lp_allow[m]:.3e})"
        lp_err = max(lp_err, e)
    return {"near_tie_rows": tie_rows, "lse_max_err": float(lse_err.max()), "lp_max_err": float(lp_err),
            "lse_allow_max": float(lse_allow.max()), "lp_allow_max": float(lp_allow.max())}


def check_walk(shape, anchor, U, V, g_ids, g_lp, g_path_idx, g_path_ids, g_score, ref=None, tie_rows=(),
               greedy=False, gate=None):
    """Exact check of the walk on the GPU's own candidates (and gate rows [B,T,R], when gated),
    and (when given) against the full oracle."""
    B, T, K = shape.batch, shape.block, shape.top_k
    g_ids = g_ids.reshape(B, T, K)
    g_lp = g_lp.reshape(B, T, K)
    tau = O.transitions(anchor, g_ids, U, V, gate)
    stats = {"path_mismatch_small_margin": 0, "path_vs_oracle_mismatch_small_margin": 0}
    if greedy:
        # each step's arg-max in fp32 on both sides; a path may part from the oracle's only at a
        # step whose two choices score within MARGIN of each other (the steps after it then follow
        # a different prefix), and the score is the float64 score of the GPU's own path
        o_path, _ = O.greedy_walk(g_lp, tau)
        g_scores = O.path_score(g_lp, tau, g_path_idx)
        for b in range(B):
            assert np.array_equal(g_path_ids[b], g_ids[b, np.arange(T), g_path_idx[b]]), f"seq {b}: path ids"
            diff = np.nonzero(g_path_idx[b] != o_path[b])[0]
            if len(diff):
                t0 = int(diff[0])
                prev = 0 if t0 == 0 else int(o_path[b, t0 - 1])
                v = (g_lp[b, t0].astype(np.float32) + tau[b, t0, prev].astype(np.float32)).astype(np.float64)
                gap = abs(v[o_path[b, t0]] - v[g_path_idx[b, t0]])
                assert gap < MARGIN, f"seq {b}: greedy step {t0} differs with gap {gap:.3e}"
                stats["path_mismatch_small_margin"] += 1
            assert abs(float(g_score[b]) - g_scores[b]) <= SCORE_TOL, f"seq {b}: score {g_score[b]} vs {g_scores[b]}"
        return stats
    o_path, o_score = O.viterbi(g_lp, tau)
    best, second = O.viterbi_two_best(g_lp, tau)
    for b in range(B):
        assert np.array_equal(g_path_ids[b], g_ids[b, np.arange(T), g_path_idx[b]]), f"seq {b}: path ids inconsistent"
        if not np.array_equal(g_path_idx[b], o_path[b]):
            margin = best[b] - second[b]
            assert margin < MARGIN, f"seq {b}: path {g_path_idx[b]} vs {o_path[b]} with margin {margin:.3e}"
            stats["path_mismatch_small_margin"] += 1
            assert abs(float(g_score[b]) - float(o_score[b])) <= margin + SCORE_TOL
        else:
            assert abs(float(g_score[b]) - float(o_score[b])) <= SCORE_TOL, f"seq {b}: score {g_score[b]} vs {o_score[b]}"
    if ref is not None:
        seq_tie = {m // T for m in tie_rows}
        for b in range(B):
            if b in seq_tie:
                continue
            if not np.array_equal(g_path_idx[b], ref["path_idx"][b]):
                margin = ref["best"][b] - ref["second"][b]
                assert margin < MARGIN, f"seq {b}: path vs full oracle differs with margin {margin:.3e}"
                stats["path_vs_oracle_mismatch_small_margin"] += 1
            else:
                assert np.array_equal(g_path_ids[b], ref["path_ids"][b])
                assert abs(float(g_score[b]) - float(ref["score"][b])) <= SCORE_TOL
    return stats


def check_gate(g_gpu: np.ndarray, g_ref: np.ndarray) -> dict:
    """Gate rows within GATE_TOL absolute (they are O(1) sums of H bf16 products; fp32 sums in
    the MMA order against the oracle's float64 sums rounded once)."""
    err = np.abs(g_gpu.astype(np.float64) - g_ref.astype(np.float64))
    assert err.max() <= GATE_TOL, f"gate: max abs error {err.max():.3e} > {GATE_TOL}"
    return {"gate_max_abs_err": float(err.max())}


def check_tail(shape, inp: dict, ref: dict, g: dict, seqs=None) -> dict:
    """Compare a draft_tail result with the oracle on the listed sequences (see the module
    docstring); ref is the oracle's end-to-end result for those sequences.

    Asserted step by step, each step on its own input: the conv output; the selection on the
    GPU's own conv output; the walk exactly on the GPU's own candidates (and gate rows). Asserted
    end to end, against the oracle's own conv output, with the same near-tie rules: every row's
    top-K ids (a differing id only inside the tie band of the oracle's logits), lse and candidate
    log-probs within 2e-3, and every path (a differing path only where the oracle's best/second
    margin is below 1e-2 or the sequence holds an end-to-end near-tie row), with its score within
    2e-3 where the paths agree."""
    B, K, H = shape.batch, shape.top_k, shape.hidden
    first = int(getattr(shape, "first_slot", 0))
    T = shape.block - first  # slots per sequence
    seqs = list(range(B)) if seqs is None else list(seqs)
    assert g["device_error"] == 0, f"device error word {g['device_error']}"
    sel = np.asarray(seqs)
    # 1. conv (every row): each layer on the GPU's own layer input, and the chain end to end
    hid = np.asarray(inp["hidden"])[sel]
    rep = check_conv_layers(hid, inp["conv_w"], shape.dtype, shape.taps, [z[sel] for z in g["z_layers"]],
                            g["z"][sel], ref_chain=ref["z"])
    # 2. selection, on the GPU's own conv output (the slot rows)
    ref_g = O.select_from_z(g["z"][sel], inp, shape, seqs)
    z_rows = ref_g["z"][:, first:, :].reshape(-1, H)
    rows = (sel[:, None] * T + np.arange(T)[None, :]).reshape(-1)
    g_ids = g["cand_ids"].reshape(B * T, K)[rows]
    g_lp = g["cand_lp"].reshape(B * T, K)[rows]
    g_lse = g["lse"].reshape(B * T)[rows]
    rep.update(check_topk(ref_g, g_ids, g_lp, g_lse, z_rows, inp["lm_head"], K))
    g_gate = None
    if getattr(shape, "gate", False):
        # the gate rows: H(h_t) of the GPU's own conv output (fp32 sums of bf16 products)
        g_gate = g["gate"][sel][:, first:]
        rep.update(check_gate(g_gate.reshape(-1, g_gate.shape[-1]), ref_g["gate"].reshape(-1, g_gate.shape[-1])))

    class _S:  # the subset as a shape
        batch, block, top_k = len(seqs), T, K
    # 3. walk: exact on the GPU's candidates, and against the oracle's path from the same z
    rep.update(check_walk(_S, np.asarray(inp["anchor"])[sel], inp["U"], inp["V"], g_ids, g_lp,
                          g["path_idx"][sel], g["path_ids"][sel], g["score"][sel], ref=ref_g,
                          tie_rows=rep["near_tie_rows"], greedy=bool(getattr(shape, "greedy", False)),
                          gate=g_gate))
    # 4. end to end, against the oracle's own conv output. The continuous values may also differ by
    # what the conv's difference alone explains: the oracle's values on the GPU's conv output minus
    # those on its own (zero where the two conv outputs agree)
    z_ref_rows = np.asarray(ref["z"])[:, first:, :].reshape(-1, H)
    lse_allow = np.abs(ref_g["lse"].reshape(-1) - ref["lse"].reshape(-1))
    lp_allow = np.zeros(len(rows))
    for m in range(len(rows)):
        if not np.array_equal(O.widen(z_rows[m]), O.widen(z_ref_rows[m])):
            l_g = O.logits(z_rows[m:m + 1], inp["lm_head"][g_ids[m]])[0].astype(np.float64)
            l_r = O.logits(z_ref_rows[m:m + 1], inp["lm_head"][g_ids[m]])[0].astype(np.float64)
            lp_allow[m] = np.abs((l_g - ref_g["lse"].reshape(-1)[m]) - (l_r - ref["lse"].reshape(-1)[m])).max()
    e2e = check_topk(ref, g_ids, g_lp, g_lse, z_ref_rows, inp["lm_head"], K, lse_allow=lse_allow, lp_allow=lp_allow)
    seq_tie = {m // T for m in e2e["near_tie_rows"]}
    paths_same = 0
    e2e_small_margin = 0
    for i in range(len(seqs)):
        same = np.array_equal(g["path_idx"][sel[i]], ref["path_idx"][i])
        paths_same += int(same)
        if i in seq_tie:
            continue  # a near tie in the candidate lists: the lists themselves may differ
        if same:
            assert np.array_equal(g["path_ids"][sel[i]], ref["path_ids"][i])
            allow = abs(float(ref_g["score"][i]) - float(ref["score"][i])) \
                if np.array_equal(ref_g["path_idx"][i], ref["path_idx"][i]) else 0.0
            assert abs(float(g["score"][sel[i]]) - float(ref["score"][i])) <= SCORE_TOL + allow, \
                f"seq {seqs[i]}: end-to-end score {g['score'][sel[i]]} vs {ref['score'][i]} (allowance {allow:.3e})"
        else:
            margin = ref["best"][i] - ref["second"][i]
            assert margin < MARGIN, f"seq {seqs[i]}: end-to-end path differs with margin {margin:.3e}"
            e2e_small_margin += 1
    rep["e2e_near_tie_rows"] = len(e2e["near_tie_rows"])
    rep["e2e_lse_max_err"] = e2e["lse_max_err"]
    rep["e2e_lp_max_err"] = e2e["lp_max_err"]
    rep["e2e_lse_conv_allowance_max"] = e2e["lse_allow_max"]
    rep["e2e_lp_conv_allowance_max"] = e2e["lp_allow_max"]
    rep["e2e_rows_same_ids"] = float(np.mean([np.array_equal(a, b) for a, b in
                                              zip(g_ids, ref["cand_ids"].reshape(-1, K))]))
    rep["e2e_paths_same"] = paths_same / len(seqs)
    rep["e2e_paths_small_margin"] = e2e_small_margin
    return rep
