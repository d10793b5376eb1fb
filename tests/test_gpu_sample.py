"""GPU parity of the path sampled at temperature T > 0 (the walk "samples from the same
scores", "DFlash 2: keeping drafts parallel", section "軽量パスセレクター") against the CPU
oracle: the same draws on the same uniforms, the log-probability of the drawn path, the
sampler's distribution over many draws, and the whole tail in sampling mode. Each call goes
through the C ABI."""
import itertools

import numpy as np
import pytest
import torch

import synth
from oracle import core as O
from tests import parity as P

pytestmark = pytest.mark.gpu

LOGP_TOL = 2e-3   # log P(path): fp32 forward filtering against float64 (gated or not)
CDF_BAND = 1e-4   # a draw this close to a cumulative-probability boundary may fall either side


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import block_drafter_dflash2_gb300 as df2
    assert torch.cuda.is_available()
    df2.load()


def greedy_step_logp(lp, tau, temp, path):
    """log P of given paths under per-step sampling along the greedy walk, written out in float64:
    sum_t log softmax_j ((lp_t(j) + tau_t(j_{t-1}, j)) / T)(j_t), slot 0's predecessor the anchor."""
    B, T, K = lp.shape
    out = np.zeros(B)
    for b in range(B):
        prev = 0
        for t in range(T):
            s = (lp[b, t].astype(np.float64) + tau[b, t, prev].astype(np.float64)) / temp
            out[b] += s[path[b, t]] - np.logaddexp.reduce(s)
            prev = int(path[b, t])
    return out


def check_greedy_sample(cand, lp, tau, temp, u, g_pix, g_pid, g_logp, logp_tol=LOGP_TOL):
    """Per-step draws along the greedy walk: exact except where the oracle's draw lies within
    CDF_BAND of a boundary; the GPU's log P matches the exact value for the path it drew."""
    B, T, K = lp.shape
    o_pix, _, margin = O.greedy_sample_walk(lp, tau, temp, u)
    exact = greedy_step_logp(lp, tau, temp, g_pix)
    near = 0
    for b in range(B):
        assert np.array_equal(g_pid[b], cand[b, np.arange(T), g_pix[b]])
        if margin[b] > CDF_BAND:
            assert np.array_equal(g_pix[b], o_pix[b]), f"seq {b}: drew {g_pix[b]} vs {o_pix[b]}"
        elif not np.array_equal(g_pix[b], o_pix[b]):
            near += 1
        assert abs(float(g_logp[b]) - exact[b]) <= logp_tol, f"seq {b}: log P {g_logp[b]} vs {exact[b]}"
    return near


def _run_sample(shape, anchor, cand, lp, U, V, temp, u, gate=None):
    import block_drafter_dflash2_gb300 as df2
    B, T = shape.batch, shape.block
    pid = torch.empty((B, T), dtype=torch.int32, device="cuda:0")
    pix = torch.empty((B, T), dtype=torch.int32, device="cuda:0")
    sc = torch.empty((B,), dtype=torch.float32, device="cuda:0")
    ws = P.workspace(shape)
    df2.sample_walk(shape, P.dev(anchor), P.dev(cand), P.dev(lp), P.dev(U), P.dev(V), temp, P.dev(u), pid, pix, sc,
                    ws, gate=None if gate is None else P.dev(gate))
    torch.cuda.synchronize()
    assert df2.read_device_error(ws) == 0
    return P.host(pid), P.host(pix), P.host(sc)


def check_sample(cand, lp, tau, temp, u, g_pix, g_pid, g_logp, logp_tol=LOGP_TOL):
    """Exact draws except where the oracle's draw lies within CDF_BAND of a boundary; the
    GPU's log P(path) matches the oracle's for the path the GPU drew."""
    B, T, K = lp.shape
    o_pix, o_logp, margin = O.sample_walk(lp, tau, temp, u)
    logz = O.log_partition(lp, tau, temp)
    near = 0
    for b in range(B):
        assert np.array_equal(g_pid[b], cand[b, np.arange(T), g_pix[b]])
        if margin[b] > CDF_BAND:
            assert np.array_equal(g_pix[b], o_pix[b]), f"seq {b}: drew {g_pix[b]} vs {o_pix[b]}"
        elif not np.array_equal(g_pix[b], o_pix[b]):
            near += 1
        exact = O.path_score(lp[b:b + 1], tau[b:b + 1], g_pix[b:b + 1])[0] / temp - logz[b]
        assert abs(float(g_logp[b]) - exact) <= logp_tol, f"seq {b}: log P {g_logp[b]} vs {exact}"
    return near


@pytest.mark.parametrize("T,K,R,temp", [(8, 16, 256, 1.0), (8, 16, 256, 0.3), (1, 16, 64, 2.0),
                                        (16, 4, 64, 1.0), (3, 16, 384, 0.7)])
def test_sample_walk_step(T, K, R, temp):
    rng = np.random.default_rng(T * 100 + K + R)
    B, Vv = 64, 3000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(9, 3, (Vv, R), 0.3)
    V = synth.normal(9, 4, (Vv, R), 0.3)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    lp = (-np.sort(np.abs(rng.standard_normal((B, T, K))), axis=2) * 1.5).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    u = rng.random((B, T)).astype(np.float32)
    pid, pix, sc = _run_sample(P.shape_of(sh), anchor, cand, lp, U, V, temp, u)
    tau = O.transitions(anchor, cand, U, V)
    near = check_sample(cand, lp, tau, temp, u.astype(np.float64), pix, pid, sc)
    print(T, K, R, temp, "draws at a boundary", near)


def test_sample_walk_gated():
    rng = np.random.default_rng(21)
    B, T, K, R, Vv = 32, 8, 16, 256, 2000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(10, 3, (Vv, R), 0.2)
    V = synth.normal(10, 4, (Vv, R), 0.2)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    lp = (-np.sort(np.abs(rng.standard_normal((B, T, K))), axis=2)).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    gate = rng.standard_normal((B, T, R)).astype(np.float32)
    u = rng.random((B, T)).astype(np.float32)
    pid, pix, sc = _run_sample(P.shape_of(sh), anchor, cand, lp, U, V, 1.0, u, gate=gate)
    tau = O.transitions(anchor, cand, U, V, gate)
    check_sample(cand, lp, tau, 1.0, u.astype(np.float64), pix, pid, sc, logp_tol=LOGP_TOL)


def test_sampler_distribution_over_many_draws():
    # one 3 x 3 x 2 lattice repeated over 6000 sequences with independent uniforms: the drawn
    # paths' frequencies match exp(score / T) / Z
    rng = np.random.default_rng(33)
    B, T, K, R, Vv = 6000, 2, 3, 16, 50
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(11, 3, (Vv, R), 0.5)
    V = synth.normal(11, 4, (Vv, R), 0.5)
    cand = np.broadcast_to(rng.integers(0, Vv, size=(1, T, K)), (B, T, K)).astype(np.int32).copy()
    lp = np.broadcast_to(-np.sort(np.abs(rng.standard_normal((1, T, K))), axis=2), (B, T, K)).astype(np.float32).copy()
    anchor = np.full(B, 7, np.int32)
    u = rng.random((B, T)).astype(np.float32)
    temp = 0.8
    pid, pix, sc = _run_sample(P.shape_of(sh), anchor, cand, lp, U, V, temp, u)
    tau = O.transitions(anchor[:1], cand[:1], U, V)
    paths = list(itertools.product(range(K), repeat=T))
    scores = np.array([O.path_score(lp[:1], tau, np.asarray(c)[None])[0] / temp for c in paths])
    prob = np.exp(scores - np.logaddexp.reduce(scores))
    freq = np.array([np.mean(np.all(pix == np.asarray(c)[None], axis=1)) for c in paths])
    # 6000 draws: 4.5 standard errors of the largest cell
    assert np.all(np.abs(freq - prob) <= 4.5 * np.sqrt(prob * (1 - prob) / B) + 1e-3), (freq, prob)


def test_low_temperature_sample_is_the_viterbi_path():
    rng = np.random.default_rng(44)
    B, T, K, R, Vv = 16, 8, 16, 64, 2000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(12, 3, (Vv, R), 0.3)
    V = synth.normal(12, 4, (Vv, R), 0.3)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    lp = (-np.sort(np.abs(rng.standard_normal((B, T, K))), axis=2) * 3).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    u = (rng.random((B, T)) * 0.9 + 0.05).astype(np.float32)
    pid, pix, sc = _run_sample(P.shape_of(sh), anchor, cand, lp, U, V, 1e-3, u)
    vid, vix, vsc, err = P.run_viterbi(P.shape_of(sh), P.dev(anchor), P.dev(cand), P.dev(lp), P.dev(U), P.dev(V))
    tau = O.transitions(anchor, cand, U, V)
    best, second = O.viterbi_two_best(lp, tau)
    for b in range(B):
        if best[b] - second[b] > 0.05:  # a clear best path: all the mass at T = 1e-3
            assert np.array_equal(pix[b], vix[b])


@pytest.mark.parametrize("gated,greedy", [(False, False), (True, False), (False, True), (True, True)])
def test_draft_tail_sampled_small(gated, greedy):
    import block_drafter_dflash2_gb300 as df2
    rc = synth.scaled_recipe(synth.recipe(2), batch=6, block=8, hidden=512, vocab=30_011, layers=2)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    B, T, K, R = sh.batch, sh.block, sh.top_k, sh.rank
    d = P.upload_inputs(inp)
    shape = P.shape_of(sh, greedy=greedy)
    u = np.random.default_rng(55).random((B, T)).astype(np.float32)
    o = {k: torch.empty(v, dtype=dt, device="cuda:0") for k, v, dt in
         [("pid", (B, T), torch.int32), ("pix", (B, T), torch.int32), ("sc", (B,), torch.float32),
          ("ids", (B, T, K), torch.int32), ("lp", (B, T, K), torch.float32), ("gate", (B, T, R), torch.float32)]}
    ws = P.workspace(shape)
    df2.draft_tail_sampled(shape, d["hidden"], d["lm_head"], d["U"], d["V"], d["conv_w"], d["anchor"], 0.9,
                           P.dev(u), o["pid"], o["pix"], o["sc"], ws, gate_w=d["gate_w"] if gated else None,
                           cand_ids=o["ids"], cand_lp=o["lp"], gate=o["gate"] if gated else None)
    torch.cuda.synchronize()
    assert df2.read_device_error(ws) == 0
    cand, lp = P.host(o["ids"]), P.host(o["lp"])
    gate = P.host(o["gate"]) if gated else None
    tau = O.transitions(inp["anchor"], cand, inp["U"], inp["V"], gate)
    check = check_greedy_sample if greedy else check_sample
    check(cand, lp, tau, 0.9, u.astype(np.float64), P.host(o["pix"]), P.host(o["pid"]), P.host(o["sc"]))


# ---------------------------------------------------------------- per-step draws along the greedy walk


@pytest.mark.parametrize("T,K,R,temp", [(8, 16, 256, 1.0), (8, 16, 256, 0.3), (1, 16, 64, 2.0),
                                        (16, 4, 64, 1.0), (3, 16, 384, 0.7)])
def test_greedy_sample_walk_step(T, K, R, temp):
    rng = np.random.default_rng(T * 100 + K + R + 1)
    B, Vv = 64, 3000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(19, 3, (Vv, R), 0.3)
    V = synth.normal(19, 4, (Vv, R), 0.3)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    lp = (-np.sort(np.abs(rng.standard_normal((B, T, K))), axis=2) * 1.5).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    u = rng.random((B, T)).astype(np.float32)
    pid, pix, sc = _run_sample(P.shape_of(sh, greedy=True), anchor, cand, lp, U, V, temp, u)
    tau = O.transitions(anchor, cand, U, V)
    near = check_greedy_sample(cand, lp, tau, temp, u.astype(np.float64), pix, pid, sc)
    print(T, K, R, temp, "draws at a boundary", near)


def test_greedy_sample_walk_gated():
    rng = np.random.default_rng(22)
    B, T, K, R, Vv = 32, 8, 16, 256, 2000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(10, 3, (Vv, R), 0.2)
    V = synth.normal(10, 4, (Vv, R), 0.2)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    lp = (-np.sort(np.abs(rng.standard_normal((B, T, K))), axis=2)).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    gate = rng.standard_normal((B, T, R)).astype(np.float32)
    u = rng.random((B, T)).astype(np.float32)
    pid, pix, sc = _run_sample(P.shape_of(sh, greedy=True), anchor, cand, lp, U, V, 1.0, u, gate=gate)
    tau = O.transitions(anchor, cand, U, V, gate)
    check_greedy_sample(cand, lp, tau, 1.0, u.astype(np.float64), pix, pid, sc)


def test_greedy_sampler_distribution_over_many_draws():
    # one 3-candidate, 2-slot lattice repeated over 6000 sequences with independent uniforms: the
    # drawn paths' frequencies match the product of the step softmaxes
    rng = np.random.default_rng(34)
    B, T, K, R, Vv = 6000, 2, 3, 16, 50
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(13, 3, (Vv, R), 0.5)
    V = synth.normal(13, 4, (Vv, R), 0.5)
    cand = np.broadcast_to(rng.integers(0, Vv, size=(1, T, K)), (B, T, K)).astype(np.int32).copy()
    lp = np.broadcast_to(-np.sort(np.abs(rng.standard_normal((1, T, K))), axis=2), (B, T, K)).astype(np.float32).copy()
    anchor = np.full(B, 9, np.int32)
    u = rng.random((B, T)).astype(np.float32)
    temp = 0.8
    pid, pix, sc = _run_sample(P.shape_of(sh, greedy=True), anchor, cand, lp, U, V, temp, u)
    tau = O.transitions(anchor[:1], cand[:1], U, V)
    paths = list(itertools.product(range(K), repeat=T))
    prob = np.exp(np.array([greedy_step_logp(lp[:1], tau, temp, np.asarray(c)[None])[0] for c in paths]))
    freq = np.array([np.mean(np.all(pix == np.asarray(c)[None], axis=1)) for c in paths])
    assert abs(prob.sum() - 1.0) < 1e-9
    assert np.all(np.abs(freq - prob) <= 4.5 * np.sqrt(prob * (1 - prob) / B) + 1e-3), (freq, prob)


def test_low_temperature_greedy_sample_is_the_greedy_path():
    rng = np.random.default_rng(45)
    B, T, K, R, Vv = 16, 8, 16, 64, 2000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(14, 3, (Vv, R), 0.3)
    V = synth.normal(14, 4, (Vv, R), 0.3)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    lp = (-np.sort(np.abs(rng.standard_normal((B, T, K))), axis=2) * 3).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    u = (rng.random((B, T)) * 0.9 + 0.05).astype(np.float32)
    pid, pix, sc = _run_sample(P.shape_of(sh, greedy=True), anchor, cand, lp, U, V, 1e-3, u)
    tau = O.transitions(anchor, cand, U, V)
    gp, _ = O.greedy_walk(lp, tau)
    for b in range(B):
        # a clear best step everywhere along the greedy path: all the mass at T = 1e-3
        gaps = []
        prev = 0
        for t in range(T):
            v = np.sort(lp[b, t].astype(np.float64) + tau[b, t, prev])[::-1]
            gaps.append(v[0] - v[1])
            prev = gp[b, t]
        if min(gaps) > 0.05:
            assert np.array_equal(pix[b], gp[b])
