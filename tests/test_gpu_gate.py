"""GPU parity of the context gate H(h_t) (the pages' S_t(a, b) = U_t(b) + <A(a) (.) H(h_t), B(b)>,
"DFlash 2: keeping drafts parallel", section "軽量パスセレクター") against the CPU oracle:
the gate rows formed in the LM-head pass, the gated transitions and walk, and the whole gated
tail. Each call goes through the C ABI."""
import numpy as np
import pytest
import torch

import synth
from oracle import core as O
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import block_drafter_dflash2_gb300 as df2
    assert torch.cuda.is_available()
    df2.load()


def _recipe(base=2, **kw):
    return synth.scaled_recipe(synth.recipe(base), **kw)


GATED_CASES = {
    # several vocab tiles per CTA, vocab not a multiple of 16 (gate columns start at 70,016)
    "b3_t8_h512_v70005": dict(batch=3, block=8, hidden=512, vocab=70_005, layers=2),
    # two row chunks of 128 (160 rows, the second ragged), each loading the gate columns
    "b20_t8_h256_v20003": dict(batch=20, block=8, hidden=256, vocab=20_003, layers=1),
    # vocab smaller than the partitions: some partitions hold only gate columns; K < 16, block 1
    "b4_t1_h128_v100_k4": dict(batch=4, block=1, hidden=128, vocab=100, top_k=4, rank=32, layers=3),
    # rank 272: the walk stages the embeddings in two chunks and gates each
    "b2_t5_h64_v999_r272_nl0": dict(batch=2, block=5, hidden=64, vocab=999, rank=272, layers=0),
    # the page's hidden size and rank at 8 rows (the fused select + walk with early gathers)
    "b1_t8_h5120_v30011": dict(batch=1, block=8, hidden=5120, vocab=30_011, layers=5),
}


@pytest.mark.parametrize("name", sorted(GATED_CASES))
def test_draft_tail_gated_small(name):
    rc = _recipe(**GATED_CASES[name])
    sh = rc.shape
    sh.gate = True
    inp = synth.make_inputs(rc)
    ref = O.draft_tail(inp, sh)
    g = P.run_tail(P.shape_of(sh), P.upload_inputs(inp), gated=True)
    rep = P.check_tail(sh, inp, ref, g)
    print(name, {k: v for k, v in rep.items() if k != "near_tie_rows"}, "ties", len(rep["near_tie_rows"]))


def test_draft_tail_gated_greedy():
    rc = _recipe(batch=4, block=8, hidden=256, vocab=9_001, layers=2)
    sh = rc.shape
    sh.gate = True
    sh.greedy = True
    inp = synth.make_inputs(rc)
    g = P.run_tail(P.shape_of(sh, greedy=True), P.upload_inputs(inp), gated=True)
    assert g["device_error"] == 0
    # the greedy walk on the GPU's own candidates and gate rows
    tau = O.transitions(inp["anchor"], g["cand_ids"], inp["U"], inp["V"], g["gate"])
    gp, gs = O.greedy_walk(g["cand_lp"], tau)
    assert np.array_equal(g["path_idx"], gp)
    assert np.allclose(g["score"], gs, atol=P.SCORE_TOL)
    P.check_walk(sh, inp["anchor"], inp["U"], inp["V"], g["cand_ids"], g["cand_lp"], g["path_idx"],
                 g["path_ids"], g["score"], greedy=True, gate=g["gate"])


@pytest.mark.parametrize("M,V,H,R", [(8, 31_040, 5120, 256), (200, 12_345, 256, 64), (1, 777, 64, 16)])
def test_select_topk_gated_gate_rows_and_unchanged_ranking(M, V, H, R):
    import block_drafter_dflash2_gb300 as df2
    rc = _recipe(batch=M, block=1, hidden=H, vocab=V, rank=R, layers=0)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    rows = inp["hidden"].reshape(M, H)
    shape = P.shape_of(sh)
    d_rows, d_w, d_g = P.dev(rows), P.dev(inp["lm_head"]), P.dev(inp["gate_w"])
    ids = torch.empty((M, sh.top_k), dtype=torch.int32, device="cuda:0")
    lp = torch.empty((M, sh.top_k), dtype=torch.float32, device="cuda:0")
    lse = torch.empty((M,), dtype=torch.float32, device="cuda:0")
    gate = torch.full((M, R), float("nan"), dtype=torch.float32, device="cuda:0")
    ws = P.workspace(shape)
    df2.select_topk_gated(shape, d_rows, d_w, d_g, ids, lp, lse, gate, ws)
    torch.cuda.synchronize()
    assert df2.read_device_error(ws) == 0
    rep = P.check_gate(P.host(gate), O.context_gate(rows, inp["gate_w"]))
    # the gate columns do not disturb the ranking: same ids as the ungated call
    ids0, lp0, lse0 = P.run_topk(shape, d_rows, d_w)
    assert np.array_equal(P.host(ids), ids0)
    assert np.allclose(P.host(lp), lp0, atol=1e-5)
    assert np.allclose(P.host(lse), lse0, atol=1e-5)
    print(M, V, H, R, rep)


@pytest.mark.parametrize("T,K,R,dtype", [(8, 16, 256, "bf16"), (1, 16, 256, "bf16"), (16, 4, 64, "bf16"),
                                         (3, 16, 384, "bf16"), (4, 4, 32, "f32")])
def test_viterbi_gated_step(T, K, R, dtype):
    rng = np.random.default_rng(T * 1000 + K * 10 + R)
    B, Vv = 6, 3000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0, dtype=dtype)
    kind = "bf16" if dtype == "bf16" else "f32"
    U = synth.normal(7, 3, (Vv, R), 0.1, kind)
    V = synth.normal(7, 4, (Vv, R), 0.1, kind)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    lp = (-np.sort(np.abs(rng.standard_normal((B, T, K))), axis=2) * 2).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    gate = rng.standard_normal((B, T, R)).astype(np.float32)
    pid, pix, sc, err = P.run_viterbi(P.shape_of(sh), P.dev(anchor), P.dev(cand), P.dev(lp), P.dev(U), P.dev(V),
                                      gate=P.dev(gate))
    assert err == 0
    P.check_walk(sh, anchor, U, V, cand, lp, pix, pid, sc, gate=gate)


def test_viterbi_gate_of_ones_is_ungated_bitwise():
    # bf16(v * 1) = v: the all-ones gate reproduces the ungated walk exactly
    rng = np.random.default_rng(11)
    B, T, K, R, Vv = 5, 8, 16, 256, 2000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(8, 3, (Vv, R), 0.2)
    V = synth.normal(8, 4, (Vv, R), 0.2)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    lp = (-np.sort(np.abs(rng.standard_normal((B, T, K))), axis=2)).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    args = (P.dev(anchor), P.dev(cand), P.dev(lp), P.dev(U), P.dev(V))
    p0 = P.run_viterbi(P.shape_of(sh), *args)
    p1 = P.run_viterbi(P.shape_of(sh), *args, gate=P.dev(np.ones((B, T, R), np.float32)))
    for a, b in zip(p0[:3], p1[:3]):
        assert np.array_equal(a, b)


def test_tiny_fp32_workload_gated():
    # dtype fp32: the gate partition of the SIMT LM-head kernel, the fp32 gated tiles
    rc = synth.recipe(1)
    sh = rc.shape
    sh.gate = True
    inp = synth.make_inputs(rc)
    ref = O.draft_tail(inp, sh)
    g = P.run_tail(P.shape_of(sh), P.upload_inputs(inp), gated=True)
    rep = P.check_tail(sh, inp, ref, g)
    assert rep["gate_max_abs_err"] < 1e-4
    # the walk is the brute-force best path over the GPU's candidates and gate rows (4^4 paths)
    tau = O.transitions(inp["anchor"], g["cand_ids"], inp["U"], inp["V"], g["gate"])
    bp, _ = O.brute_force_best(g["cand_lp"], tau)
    assert np.array_equal(bp, g["path_idx"])
