"""Parity harness: runs the CUDA library through its C ABI and compares it with the oracle.

Tolerances (from the draft-tail contract): token ids and paths bit-exact except at
near-ties; lse, candidate log-probs and path scores within 2e-3 absolute; conv outputs
within 1e-2 relative.

Each step is compared with the oracle on that step's own input, so that a legitimate
difference upstream is not counted against a later step: the conv output z against the
oracle's conv; the LM-head selection against the oracle run on the GPU's own z (a bf16 ulp
of difference in z moves a logit by ~1e-3, more than the near-tie band); the walk exactly on
the GPU's own candidates. Agreement with the oracle end to end is reported as well.

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
    return out


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


def check_conv(z_gpu: np.ndarray, z_ref: np.ndarray, x_in=None):
    """Conv outputs within 1e-2 relative, read per output row: ||gpu - ref||_2 <= 1e-2 ||ref||_2.
    A per-element ratio is not used because a * x[t-1] + b * x[t] can cancel to near zero while
    its rounding error stays at the operands' scale. When the layer input `x_in` is given (one
    layer), every element is also bounded by 2^-7 * max(|x[t]|, |x[t-1]|): two bf16 units in the
    last place of the operands, i.e. the output rounding plus the tap error."""
    g = O.widen(z_gpu).reshape(-1, z_gpu.shape[-1])
    r = O.widen(z_ref).reshape(-1, z_ref.shape[-1])
    row_err = np.linalg.norm(g - r, axis=1) / np.maximum(np.linalg.norm(r, axis=1), 1e-30)
    assert row_err.max() <= CONV_RTOL, f"conv: row relative error {row_err.max():.3e} > {CONV_RTOL}"
    rep = {"conv_exact_frac": float((g == r).mean()), "conv_max_abs": float(np.abs(g - r).max()),
           "conv_row_rel_max": float(row_err.max())}
    if x_in is not None:
        x = O.widen(x_in)
        xp = np.zeros_like(x)
        xp[:, 1:] = x[:, :-1]
        scale = np.maximum(np.abs(x), np.abs(xp)).reshape(g.shape)
        over = np.abs(g - r) > 2.0 ** -7 * scale + 1e-30
        assert not over.any(), f"conv: {over.sum()} elements beyond 2 operand ulps"
        rep["conv_operand_ulps_max"] = float((np.abs(g - r) / np.maximum(scale, 1e-30)).max() * 2 ** 8)
    return rep


def check_topk(ref: dict, g_ids, g_lp, g_lse, z_rows, lm_head, K):
    """ref: oracle outputs flattened to rows (cand_ids [M,K], cand_logit, max_logit, lse)."""
    M = g_ids.shape[0]
    o_ids = ref["cand_ids"].reshape(M, K)
    o_val = ref["cand_logit"].reshape(M, K)
    o_max = ref["max_logit"].reshape(M)
    o_lse = ref["lse"].reshape(M)
    lse_err = np.abs(g_lse.reshape(M).astype(np.float64) - o_lse)
    assert lse_err.max() <= LSE_TOL, f"lse error {lse_err.max():.3e}"
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
        lp_err = max(lp_err, e)
    assert lp_err <= LP_TOL, f"cand_lp error {lp_err:.3e}"
    return {"near_tie_rows": tie_rows, "lse_max_err": float(lse_err.max()), "lp_max_err": float(lp_err)}


def check_walk(shape, anchor, U, V, g_ids, g_lp, g_path_idx, g_path_ids, g_score, ref=None, tie_rows=(),
               greedy=False, gate=None):
    """Exact check of the walk on the GPU's own candidates (and gate rows [B,T,R], when gated),
    and (when given) against the full oracle."""
    B, T, K = shape.batch, shape.block, shape.top_k
    g_ids = g_ids.reshape(B, T, K)
    g_lp = g_lp.reshape(B, T, K)
    tau = O.transitions(anchor, g_ids, U, V, gate)
    if greedy:
        o_path, o_score = O.greedy_walk(g_lp, tau)
        best = second = None
    else:
        o_path, o_score = O.viterbi(g_lp, tau)
        best, second = O.viterbi_two_best(g_lp, tau)
    stats = {"path_mismatch_small_margin": 0, "path_vs_oracle_mismatch_small_margin": 0}
    for b in range(B):
        assert np.array_equal(g_path_ids[b], g_ids[b, np.arange(T), g_path_idx[b]]), f"seq {b}: path ids inconsistent"
        if not np.array_equal(g_path_idx[b], o_path[b]):
            margin = (best[b] - second[b]) if best is not None else 0.0
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
    """Compare a draft_tail result with the oracle on the listed sequences, step by step (see
    the module docstring); ref is the oracle's end-to-end result for those sequences."""
    B, K, H = shape.batch, shape.top_k, shape.hidden
    first = int(getattr(shape, "first_slot", 0))
    T = shape.block - first  # slots per sequence
    seqs = list(range(B)) if seqs is None else list(seqs)
    assert g["device_error"] == 0, f"device error word {g['device_error']}"
    sel = np.asarray(seqs)
    # 1. conv (every row)
    rep = check_conv(g["z"][sel], ref["z"])
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
    # end to end against the oracle's own conv: reported, not asserted
    e2e_ids = ref["cand_ids"].reshape(-1, K)
    rep["e2e_rows_same_ids"] = float(np.mean([np.array_equal(a, b) for a, b in zip(g_ids, e2e_ids)]))
    rep["e2e_rows_same_set"] = float(np.mean([set(a.tolist()) == set(b.tolist()) for a, b in zip(g_ids, e2e_ids)]))
    rep["e2e_paths_same"] = float(np.mean([np.array_equal(a, b) for a, b in zip(g["path_ids"][sel], ref["path_ids"])]))
    rep["e2e_lse_max_err"] = float(np.abs(g_lse.astype(np.float64) - ref["lse"].reshape(-1)).max())
    return rep
