"""Pins for the CPU oracle: checks against closed forms, special cases, brute force
and hand-worked values — never against the oracle itself.

Each test names the definition it pins (DFlash2 pages: the conv "inside each block",
the selector's pairwise score and walk from the anchor; see the oracle's header).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import synth
from oracle import core as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_of(values):
    """bf16 bit patterns of values that are exactly representable in bf16."""
    f = np.asarray(values, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


# ---------------------------------------------------------------- storage rounding


def test_round_bf16_known_patterns():
    # 1, halfway cases (ties to even), just above halfway, negative, carry into exponent
    cases = {
        1.0: 0x3F80,
        1.0 + 2.0 ** -8: 0x3F80,              # halfway between 0x3F80 and 0x3F81 -> even
        1.0 + 3 * 2.0 ** -8: 0x3F82,          # halfway between 0x3F81 and 0x3F82 -> even
        1.0 + 2.0 ** -8 + 2.0 ** -40: 0x3F81,  # just above halfway -> up
        -2.5: 0xC020,
        2.0 - 2.0 ** -9: 0x4000,              # rounds up across the binade
        0.0: 0x0000,
        3.0e38: 0x7F62,
    }
    got = O.round_bf16(np.array(list(cases.keys())))
    assert [int(g) for g in got] == list(cases.values())


def test_round_bf16_matches_torch_on_fp32_values():
    # values exact in fp32 round the same way from double and from float (no double rounding)
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200_000) * 3).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.round_bf16(x.astype(np.float64)), ref)


# ---------------------------------------------------------------- conv (kernel size 2)


def _pos_hidden(B, T, H, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.integers(1, 32, size=(B, T, H)) / 4.0  # positive multiples of 1/4: exact in bf16
    return bf16_of(q)


def test_conv_zero_weights_is_pairwise_mean():
    # zero projection -> taps (1/2, 1/2): y[t] = (x[t] + x[t-1]) / 2, y[0] = x[0] / 2
    B, T, H = 2, 5, 32
    rng = np.random.default_rng(1)
    xq = rng.integers(-32, 33, size=(B, T, H)) / 4.0
    x = bf16_of(xq)
    w = np.zeros((1, 2 * H // 16, H), dtype=np.uint16)
    z = O.widen(O.conv_chain(x, w, "bf16", 16))
    exp = np.empty_like(xq)
    exp[:, 0] = xq[:, 0] / 2
    exp[:, 1:] = (xq[:, 1:] + xq[:, :-1]) / 2
    assert np.array_equal(z, exp)


def _tap_weights(H, group_size, mode_per_group, mag=8.0):
    """mode 'shift': tap 0 huge -> y = x[t-1]; mode 'id': tap 1 huge -> y = x[t]."""
    G = H // group_size
    w = np.zeros((2 * G, H), dtype=np.float32)
    for g in range(G):
        s = 1.0 if mode_per_group(g) == "shift" else -1.0
        w[2 * g, :] = s * mag
        w[2 * g + 1, :] = -s * mag
    return bf16_of(w)


@pytest.mark.parametrize("layers", [1, 2, 3, 5])
def test_conv_shift_limit_chains_layers(layers):
    # all taps select x[t-1]: after L layers z[t] = x[t-L] (zero for t < L)
    B, T, H = 2, 8, 64
    x = _pos_hidden(B, T, H)
    w1 = _tap_weights(H, 16, lambda g: "shift")
    w = np.stack([w1] * layers)
    z = O.widen(O.conv_chain(x, w, "bf16", 16))
    xf = O.widen(x)
    exp = np.zeros_like(xf)
    exp[:, layers:] = xf[:, :T - layers]
    assert np.array_equal(z, exp)


def test_conv_identity_limit():
    B, T, H = 1, 4, 64
    x = _pos_hidden(B, T, H, seed=3)
    w = _tap_weights(H, 16, lambda g: "id")[None]
    assert np.array_equal(O.conv_chain(x, w, "bf16", 16), x)


def test_conv_group_mapping_sixteen_channels_per_group():
    # even groups shift, odd groups pass through: channel c follows group c // 16
    B, T, H = 1, 6, 96
    x = _pos_hidden(B, T, H, seed=4)
    w = _tap_weights(H, 16, lambda g: "shift" if g % 2 == 0 else "id")[None]
    z = O.widen(O.conv_chain(x, w, "bf16", 16))
    xf = O.widen(x)
    for c in range(H):
        if (c // 16) % 2 == 0:
            assert np.array_equal(z[0, 0, c], 0.0) and np.array_equal(z[0, 1:, c], xf[0, :-1, c])
        else:
            assert np.array_equal(z[0, :, c], xf[0, :, c])


def test_conv_raw_taps_constant_projection():
    # channel 0 is 1 everywhere; projection rows read only channel 0 -> raw taps (alpha, beta)
    # so y = alpha * x[t-1] + beta * x[t] for every channel
    B, T, H, gs = 1, 5, 32, 16
    rng = np.random.default_rng(5)
    xq = rng.integers(-16, 17, size=(B, T, H)) / 4.0
    xq[..., 0] = 1.0
    alpha, beta = 0.5, 0.25
    w = np.zeros((2 * H // gs, H), dtype=np.float32)
    w[0::2, 0] = alpha
    w[1::2, 0] = beta
    z = O.conv_chain(bf16_of(xq), bf16_of(w)[None], "bf16", gs, taps="raw")
    exp = beta * xq
    exp[:, 1:] += alpha * xq[:, :-1]
    assert np.array_equal(O.widen(z), exp)


def test_conv_causal_and_convex():
    rc = synth.recipe(2)
    sh = synth.Shape(batch=2, block=8, hidden=256, vocab=64, top_k=4, rank=32, layers=3)
    r = synth.Recipe(seed=11, shape=sh, rms_normalise=True, conv_std=0.05)
    inp = synth.make_inputs(r)
    z = O.conv_chain(inp["hidden"], inp["conv_w"], "bf16", 16)
    h2 = inp["hidden"].copy()
    h2[:, 5:] = synth.f64_to_bf16(np.full(h2[:, 5:].shape, 3.0))  # change positions 5..7 only
    z2 = O.conv_chain(h2, inp["conv_w"], "bf16", 16)
    assert np.array_equal(z[:, :5], z2[:, :5])
    assert not np.array_equal(z[:, 5:], z2[:, 5:])
    # one layer: |y[t]| <= max(|x[t]|, |x[t-1]|) elementwise (convex combination)
    z1 = O.widen(O.conv_chain(inp["hidden"], inp["conv_w"][:1], "bf16", 16))
    x = O.widen(inp["hidden"])
    xp = np.zeros_like(x)
    xp[:, 1:] = x[:, :-1]
    assert np.all(np.abs(z1) <= np.maximum(np.abs(x), np.abs(xp)))
    del rc


# ---------------------------------------------------------------- logits, lse, top-K


def test_logits_hand_case_and_orientation():
    z = bf16_of([[1.0, 2.0]])
    W = bf16_of([[3.0, 4.0], [5.0, 6.0], [-1.0, 0.0]])
    assert O.logits(z, W).tolist() == [[11.0, 17.0, -1.0]]
    # one-hot lm_head rows gather the hidden channel: l[m, v] = z[m, v mod H]
    H, Vv = 48, 200
    rng = np.random.default_rng(6)
    zq = bf16_of(rng.integers(-64, 64, size=(3, H)) / 8.0)
    Wq = np.zeros((Vv, H), dtype=np.float32)
    Wq[np.arange(Vv), np.arange(Vv) % H] = 1.0
    l = O.logits(zq, bf16_of(Wq), chunk=64)
    assert np.array_equal(l, O.widen(zq)[:, np.arange(Vv) % H].astype(np.float32))


def test_lse_closed_forms():
    Vv = 248320
    l = np.full((1, Vv), 2.5, dtype=np.float32)
    assert abs(O.logsumexp_rows(l)[0] - (2.5 + math.log(Vv))) < 1e-9
    # two values: n copies of a, the rest b
    n, a, b = 17, 4.0, -1.0
    l = np.full((1, 1000), b, dtype=np.float32)
    l[0, :n] = a
    exp = math.log(n * math.exp(a) + (1000 - n) * math.exp(b))
    assert abs(O.logsumexp_rows(l)[0] - exp) < 1e-12
    # cand log-prob of uniform logits is -log V
    lp = O.cand_logprob(np.full((1, 4), 2.5, np.float32), np.array([2.5 + math.log(Vv)]))
    assert np.allclose(lp, -math.log(Vv), atol=1e-6)


def test_topk_ties_to_lower_id_closed_form():
    # l[v] = -(v mod 7): the 0-valued ids are the multiples of 7, in id order
    Vv, K = 4133, 16
    l = (-(np.arange(Vv) % 7)).astype(np.float32)[None]
    ids, vals, nxt = O.topk_rows(l, K)
    assert ids[0].tolist() == [7 * i for i in range(K)]
    assert np.all(vals == 0) and nxt[0] == 0
    # mixed values: compare with an independent ordering (Python's sort on (-value, id))
    rng = np.random.default_rng(7)
    l = (rng.integers(-20, 20, size=(5, 3000)) / 4.0).astype(np.float32)
    ids, vals, _ = O.topk_rows(l, 16)
    for m in range(5):
        ref = sorted(range(3000), key=lambda v: (-float(l[m, v]), v))[:16]
        assert ids[m].tolist() == ref


# ---------------------------------------------------------------- transitions


def test_transitions_roles_of_u_and_v():
    # U[v] = e_{v mod R}, V[v] = 2 e_{(v+1) mod R}: tau(i, j) = 2 [prev_i mod R == (cur_j + 1) mod R]
    R, Vv, B, T, K = 8, 64, 2, 3, 4
    U = np.zeros((Vv, R), np.float32)
    V = np.zeros((Vv, R), np.float32)
    U[np.arange(Vv), np.arange(Vv) % R] = 1.0
    V[np.arange(Vv), (np.arange(Vv) + 1) % R] = 2.0
    rng = np.random.default_rng(8)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    tau = O.transitions(anchor, cand, bf16_of(U), bf16_of(V))
    for b in range(B):
        for t in range(T):
            for i in range(K):
                prev = anchor[b] if t == 0 else cand[b, t - 1, i]
                for j in range(K):
                    exp = 2.0 if prev % R == (cand[b, t, j] + 1) % R else 0.0
                    assert tau[b, t, i, j] == exp


# ---------------------------------------------------------------- context gate


def test_context_gate_hand_case():
    # g[m, r] = sum_h z[m, h] gate_w[r, h] with small integers (exact in bf16 and fp32)
    z = bf16_of([[1.0, 2.0, 3.0], [0.0, -1.0, 4.0]])
    gw = bf16_of([[1.0, 0.0, 1.0], [2.0, 1.0, -1.0]])
    g = O.context_gate(z, gw)
    assert g.dtype == np.float32
    assert np.array_equal(g, np.array([[4.0, 1.0], [4.0, -5.0]], np.float32))


def _gate_case(seed=9, R=16, Vv=40, B=2, T=3, K=4):
    rng = np.random.default_rng(seed)
    U = bf16_of(np.round(rng.normal(size=(Vv, R)) * 8) / 8)
    V = bf16_of(np.round(rng.normal(size=(Vv, R)) * 8) / 8)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    return U, V, cand, anchor, rng


def test_gate_of_ones_is_the_ungated_score():
    # <A(a) (.) 1, B(b)> = <A(a), B(b)>: the gate of all ones reproduces the ungated tiles bit for bit
    U, V, cand, anchor, _ = _gate_case()
    B, T, _ = cand.shape
    ones = np.ones((B, T, U.shape[1]), np.float32)
    assert np.array_equal(O.transitions(anchor, cand, U, V, ones), O.transitions(anchor, cand, U, V))


def test_gate_one_hot_selects_one_embedding_dimension():
    # gate = e_r: tau(i, j) = U[prev_i, r] * V[cur_j, r], the gate "decides which part of the match counts"
    U, V, cand, anchor, _ = _gate_case()
    B, T, K = cand.shape
    R = U.shape[1]
    r = 5
    gate = np.zeros((B, T, R), np.float32)
    gate[:, :, r] = 1.0
    tau = O.transitions(anchor, cand, U, V, gate)
    Uw, Vw = O.widen(U), O.widen(V)
    for b in range(B):
        for t in range(T):
            for i in range(K):
                prev = anchor[b] if t == 0 else cand[b, t - 1, i]
                for j in range(K):
                    assert tau[b, t, i, j] == np.float32(Uw[prev, r] * Vw[cand[b, t, j], r])


def test_gate_is_the_current_slots_and_linear():
    # the gate of slot t scales boundary t only (t-1 -> t), and tau is linear in it: g -> -2 g gives -2 tau
    U, V, cand, anchor, rng = _gate_case()
    B, T, _ = cand.shape
    R = U.shape[1]
    gate = (np.round(rng.normal(size=(B, T, R)) * 4) / 4).astype(np.float32)
    tau = O.transitions(anchor, cand, U, V, gate)
    assert np.array_equal(O.transitions(anchor, cand, U, V, -2.0 * gate), -2.0 * tau)
    g2 = gate.copy()
    g2[:, 1] = 0.0
    tau2 = O.transitions(anchor, cand, U, V, g2)
    assert np.all(tau2[:, 1] == 0.0)
    assert np.array_equal(tau2[:, [0, 2]], tau[:, [0, 2]])


def test_gated_tiny_workload_walk_is_brute_force_best():
    rc = synth.recipe(1)
    sh = rc.shape
    sh.gate = True
    inp = synth.make_inputs(rc)
    out = O.draft_tail(inp, sh)
    assert out["gate"] is not None and out["gate"].shape == (sh.batch, sh.block, sh.rank)
    # the gate is H(h_t) of the slot's conv output row
    z = out["z"].reshape(-1, sh.hidden)
    g_direct = O.widen(z) @ O.widen(inp["gate_w"]).T
    assert np.allclose(out["gate"].reshape(-1, sh.rank), g_direct, rtol=1e-6, atol=1e-6)
    bp, bs = O.brute_force_best(out["cand_lp"], out["tau"])
    assert np.array_equal(bp, out["path_idx"])
    assert np.allclose(bs, out["score"], atol=1e-5)


# ---------------------------------------------------------------- Viterbi


def _golden_case(c):
    K = len(c["cand_lp"][0])
    T = len(c["cand_lp"])
    lp = np.asarray(c["cand_lp"], np.float32)[None]
    tau = np.zeros((1, T, K, K), np.float32)
    tau[0, 0, :, :] = np.asarray(c["tau0"], np.float32)[None, :]
    for t in range(1, T):
        tau[0, t] = np.asarray(c["tau"][t - 1], np.float32)
    return lp, tau


def test_viterbi_hand_worked_golden():
    with open(os.path.join(GOLDEN, "viterbi_hand.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        lp, tau = _golden_case(c)
        path, score = O.viterbi(lp, tau)
        assert path[0].tolist() == c["viterbi_path"] and float(score[0]) == c["viterbi_score"]
        gp, gs = O.greedy_walk(lp, tau)
        assert gp[0].tolist() == c["greedy_path"] and float(gs[0]) == c["greedy_score"]
        best, second = O.viterbi_two_best(lp, tau)
        assert best[0] == c["viterbi_score"] and second[0] == c["second_best"]


@pytest.mark.parametrize("K,T", [(4, 4), (3, 6), (16, 3), (2, 9)])
def test_viterbi_equals_brute_force(K, T):
    rng = np.random.default_rng(K * 100 + T)
    B = 3
    lp = (-np.abs(rng.standard_normal((B, T, K))) * 2).astype(np.float32)
    lp = -np.sort(-lp, axis=2)
    tau = (rng.standard_normal((B, T, K, K))).astype(np.float32)
    tau[:, 0] = tau[:, 0, :1]  # slot 0: one predecessor (the anchor)
    path, score = O.viterbi(lp, tau)
    bp, bs = O.brute_force_best(lp, tau)
    assert np.array_equal(path, bp)
    assert np.allclose(score, bs, atol=1e-5)
    assert np.allclose(O.path_score(lp, tau, path), score, atol=1e-5)
    best, second = O.viterbi_two_best(lp, tau)
    assert np.allclose(best, bs, atol=1e-9)
    # the second best by enumeration
    import itertools
    for b in range(B):
        allv = sorted((O.path_score(lp[b:b + 1], tau[b:b + 1], np.asarray(c)[None])[0]
                       for c in itertools.product(range(K), repeat=T)), reverse=True)
        assert abs(allv[1] - second[b]) < 1e-9
    gp, gs = O.greedy_walk(lp, tau)
    assert np.all(gs <= bs + 1e-12)  # no path scores above the brute-force maximum
    # the greedy path by enumeration: among all paths, the one whose every step is the best
    # successor of the step before (lowest index on ties), and its float64 score
    for b in range(B):
        steps = []
        for combo in itertools.product(range(K), repeat=T):
            ok = True
            for t in range(T):
                prev = 0 if t == 0 else combo[t - 1]
                row = [float(np.float32(lp[b, t, j] + tau[b, t, prev, j])) for j in range(K)]
                if combo[t] != row.index(max(row)):
                    ok = False
                    break
            if ok:
                steps.append(combo)
        assert len(steps) == 1 and tuple(gp[b]) == steps[0]
        s = float(lp[b, 0, gp[b, 0]]) + float(tau[b, 0, 0, gp[b, 0]])
        for t in range(1, T):
            s += float(lp[b, t, gp[b, t]]) + float(tau[b, t, gp[b, t - 1], gp[b, t]])
        assert abs(gs[b] - s) < 1e-12


def test_viterbi_zero_transitions_is_per_slot_argmax():
    rng = np.random.default_rng(9)
    lp = -np.sort(np.abs(rng.standard_normal((4, 8, 16))), axis=2).astype(np.float32)
    tau = np.zeros((4, 8, 16, 16), np.float32)
    path, score = O.viterbi(lp, tau)
    assert np.all(path == 0)  # sorted candidates: candidate 0 is each slot's argmax
    assert np.allclose(score, lp[:, :, 0].astype(np.float64).sum(axis=1), atol=1e-5)


def test_viterbi_invariant_to_per_slot_constants():
    rng = np.random.default_rng(10)
    lp = rng.standard_normal((3, 6, 5)).astype(np.float32)
    tau = rng.standard_normal((3, 6, 5, 5)).astype(np.float32)
    tau[:, 0] = tau[:, 0, :1]
    shift = (rng.integers(-8, 8, size=(3, 6, 1)) * 4.0).astype(np.float32)
    p1, _ = O.viterbi(lp, tau)
    p2, _ = O.viterbi(lp + shift, tau)
    assert np.array_equal(p1, p2)


def test_viterbi_single_slot_and_exact_ties():
    rng = np.random.default_rng(12)
    lp = rng.standard_normal((2, 1, 6)).astype(np.float32)
    tau = rng.standard_normal((2, 1, 6, 6)).astype(np.float32)
    tau[:, 0] = tau[:, 0, :1]
    path, score = O.viterbi(lp, tau)
    for b in range(2):
        assert path[b, 0] == int(np.argmax(lp[b, 0] + tau[b, 0, 0]))
    # all-equal scores: every argmax takes the lowest index
    lp = np.ones((1, 5, 4), np.float32)
    tau = np.ones((1, 5, 4, 4), np.float32)
    path, score = O.viterbi(lp, tau)
    assert np.all(path == 0) and float(score[0]) == 10.0


# ---------------------------------------------------------------- whole tail


# ---------------------------------------------------------------- sampling at T > 0


def _lattice(seed, B=2, T=3, K=3):
    rng = np.random.default_rng(seed)
    lp = (-np.abs(rng.standard_normal((B, T, K)))).astype(np.float32)
    tau = (rng.standard_normal((B, T, K, K)) * 0.7).astype(np.float32)
    tau[:, 0] = tau[:, 0, :1]  # slot 0's predecessor is the anchor: one row, repeated
    return lp, tau


def test_sample_walk_logprob_is_score_over_temperature_minus_log_partition():
    # P(path) = exp(score / T) / Z: the sampler's log-probability of the path it drew equals the
    # brute-force value from all K^T paths
    import itertools
    lp, tau = _lattice(1)
    B, T, K = lp.shape
    rng = np.random.default_rng(2)
    for temp in (0.5, 1.0, 3.0):
        for _ in range(5):
            u = rng.random((B, T))
            path, logp, _ = O.sample_walk(lp, tau, temp, u)
            for b in range(B):
                scores = [O.path_score(lp[b:b + 1], tau[b:b + 1], np.asarray(c)[None])[0] / temp
                          for c in itertools.product(range(K), repeat=T)]
                logz = np.logaddexp.reduce(scores)
                s = O.path_score(lp[b:b + 1], tau[b:b + 1], path[b:b + 1])[0] / temp
                assert abs(logp[b] - (s - logz)) < 1e-9


def test_log_partition_is_brute_force():
    import itertools
    lp, tau = _lattice(4, B=2, T=3, K=3)
    for temp in (0.7, 2.0):
        z = O.log_partition(lp, tau, temp)
        for b in range(2):
            scores = [O.path_score(lp[b:b + 1], tau[b:b + 1], np.asarray(c)[None])[0] / temp
                      for c in itertools.product(range(3), repeat=3)]
            assert abs(z[b] - np.logaddexp.reduce(scores)) < 1e-9


def test_sample_walk_frequencies_match_brute_force_distribution():
    # inverse-CDF draws on a regular grid of u reproduce the path distribution
    import itertools
    lp, tau = _lattice(3, B=1, T=2, K=3)
    temp = 0.8
    paths = list(itertools.product(range(3), repeat=2))
    scores = np.array([O.path_score(lp, tau, np.asarray(c)[None])[0] / temp for c in paths])
    prob = np.exp(scores - np.logaddexp.reduce(scores))
    n = 200
    counts = {c: 0 for c in paths}
    for a in range(n):
        for c in range(n):
            u = np.array([[(c + 0.5) / n, (a + 0.5) / n]])
            p, _, _ = O.sample_walk(lp, tau, temp, u)
            counts[tuple(int(x) for x in p[0])] += 1
    freq = np.array([counts[c] for c in paths]) / n ** 2
    assert np.abs(freq - prob).max() < 0.02


def test_sample_walk_low_temperature_is_viterbi():
    lp, tau = _lattice(5, B=3, T=4, K=4)
    rng = np.random.default_rng(6)
    vp, _ = O.viterbi(lp, tau)
    for _ in range(5):
        p, _, _ = O.sample_walk(lp, tau, 1e-4, rng.random((3, 4)) * 0.98 + 0.01)
        assert np.array_equal(p, vp)


def test_sample_walk_without_transitions_is_independent_softmax():
    # tau = 0: each slot is drawn from softmax(lp_t / T) by inverse CDF, independently
    lp, _ = _lattice(7, B=2, T=3, K=4)
    tau = np.zeros((2, 3, 4, 4), np.float32)
    u = np.array([[0.1, 0.5, 0.95], [0.7, 0.02, 0.33]])
    temp = 1.5
    p, _, _ = O.sample_walk(lp, tau, temp, u)
    for b in range(2):
        for t in range(3):
            w = np.exp(lp[b, t].astype(np.float64) / temp)
            c = np.cumsum(w / w.sum())
            assert p[b, t] == int(np.searchsorted(c, u[b, t], side="right"))


def test_first_slot_reading_selects_rows_after_the_anchor_row():
    # first_slot = 1: the conv runs over all block rows (the anchor row included, so slot 1 sees
    # it), and the selection is the all-slots selection of rows 1..block-1 with the same anchor
    rc = synth.scaled_recipe(synth.recipe(2), batch=2, block=5, hidden=64, vocab=500, rank=32, layers=2)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    sh1 = synth.Shape(**{**sh.__dict__, "first_slot": 1})
    out1 = O.draft_tail(inp, sh1)
    assert out1["path_idx"].shape == (2, 4) and out1["cand_ids"].shape == (2, 4, sh.top_k)
    z = O.conv_chain(inp["hidden"], inp["conv_w"], sh.dtype, 16)
    assert np.array_equal(O.widen(out1["z"]), O.widen(z))
    sh0 = synth.Shape(**{**sh.__dict__, "block": 4})
    out0 = O.select_from_z(z[:, 1:], inp, sh0, [0, 1])
    for k in ("cand_ids", "cand_lp", "path_idx", "path_ids", "score"):
        assert np.array_equal(out1[k], out0[k]), k
    # the anchor row matters: changing it changes slot 1's conv output
    h2 = inp["hidden"].copy()
    h2[:, 0] = O.round_bf16(-O.widen(h2[:, 0])) if sh.dtype == "bf16" else -h2[:, 0]
    z2 = O.conv_chain(h2, inp["conv_w"], sh.dtype, 16)
    assert not np.array_equal(O.widen(z2[:, 1]), O.widen(z[:, 1]))
    # and the walk over the 4 slots is the brute-force best path
    bp, _ = O.brute_force_best(out1["cand_lp"], out1["tau"])
    assert np.array_equal(bp, out1["path_idx"])


def test_tiny_fp32_workload_end_to_end_brute_force():
    rc = synth.recipe(1)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    out = O.draft_tail(inp, sh)
    # every selected id is one of that slot's candidates, and the walk is the exact best path
    bp, bs = O.brute_force_best(out["cand_lp"], out["tau"])
    assert np.array_equal(bp, out["path_idx"])
    assert np.allclose(bs, out["score"], atol=1e-5)
    # the candidates are the true top-4 of a direct dot-product evaluation of a few rows
    z = O.widen(out["z"]).reshape(-1, sh.hidden)
    W = inp["lm_head"].astype(np.float64)
    for m in range(z.shape[0]):
        direct = np.array([float(np.dot(z[m], W[v])) for v in range(sh.vocab)], dtype=np.float32)
        ref = sorted(range(sh.vocab), key=lambda v: (-float(direct[v]), v))[:sh.top_k]
        assert out["cand_ids"].reshape(-1, sh.top_k)[m].tolist() == ref
        lse = math.log(sum(math.exp(float(x)) for x in direct))
        assert abs(out["lse"].reshape(-1)[m] - lse) < 1e-9
    assert out["best"][0] >= out["second"][0]


# ---------------------------------------------------------------- draw margins and per-step sampling


def test_sample_walk_cdf_margin_hand_lattice():
    # one slot, probabilities (0.5, 0.3, 0.2): cumulative boundaries at 0.5 and 0.8; the margin is
    # the distance from u to the nearer of the two, and the draw is the first index past u
    lp = np.log(np.array([[[0.5, 0.3, 0.2]]]))
    tau = np.zeros((1, 1, 3, 3))
    for u, idx, margin in ((0.55, 1, 0.05), (0.79, 1, 0.01), (0.85, 2, 0.05), (0.1, 0, 0.4), (0.5, 1, 0.0)):
        p, _, m = O.sample_walk(lp, tau, 1.0, np.array([[u]]))
        assert p[0, 0] == idx and abs(m[0] - margin) < 1e-12, (u, p, m)
    # two slots without transitions: each slot's draw uses its own u and the margin is the smaller
    # of the two slots' margins (slot 1 has boundaries at 0.25 and 0.75)
    lp2 = np.log(np.array([[[0.5, 0.3, 0.2], [0.25, 0.5, 0.25]]]))
    tau2 = np.zeros((1, 2, 3, 3))
    p, _, m = O.sample_walk(lp2, tau2, 1.0, np.array([[0.55, 0.7]]))
    assert p[0].tolist() == [1, 1] and abs(m[0] - 0.05) < 1e-12
    p, _, m = O.sample_walk(lp2, tau2, 1.0, np.array([[0.3, 0.74]]))
    assert p[0].tolist() == [0, 1] and abs(m[0] - 0.01) < 1e-12
    # with a transition, slot 0 is drawn from its distribution given slot 1's draw: K = 2,
    # lp_0 = log(1/2, 1/2), lp_1 = 0, tau_1(i, j) = log 3 for (i, j) = (1, 0), else 0. Slot 1's
    # marginal is (2/3, 1/3); given j_1 = 0, slot 0 is (1/4, 3/4), boundary 0.25
    lp3 = np.array([[[math.log(0.5), math.log(0.5)], [0.0, 0.0]]])
    tau3 = np.zeros((1, 2, 2, 2))
    tau3[0, 1, 1, 0] = math.log(3.0)
    p, logp, m = O.sample_walk(lp3, tau3, 1.0, np.array([[0.3, 0.6]]))
    assert p[0].tolist() == [1, 0]
    assert abs(m[0] - min(abs(0.6 - 2 / 3), abs(0.3 - 0.25))) < 1e-12
    assert abs(logp[0] - math.log(2 / 3 * 3 / 4)) < 1e-12


def test_greedy_sample_walk_cdf_margin_and_draws_hand_lattice():
    # per-step draws: slot 0 from softmax(lp_0 + tau_0), slot t from softmax(lp_t + tau_t(j_{t-1}, .))
    lp = np.array([[[math.log(0.5), math.log(0.5)], [0.0, 0.0]]])
    tau = np.zeros((1, 2, 2, 2))
    tau[0, 1, 1, 0] = math.log(3.0)  # after candidate 1, slot 1 is (3/4, 1/4); after 0, (1/2, 1/2)
    p, logp, m = O.greedy_sample_walk(lp, tau, 1.0, np.array([[0.6, 0.7]]))
    assert p[0].tolist() == [1, 0] and abs(logp[0] - math.log(0.5 * 0.75)) < 1e-12
    assert abs(m[0] - min(abs(0.6 - 0.5), abs(0.7 - 0.75))) < 1e-12
    p, logp, m = O.greedy_sample_walk(lp, tau, 1.0, np.array([[0.4, 0.7]]))
    assert p[0].tolist() == [0, 1] and abs(logp[0] - math.log(0.25)) < 1e-12
    assert abs(m[0] - 0.1) < 1e-12
    # temperature 2 halves every score: slot 1 after candidate 1 is (sqrt3, 1) / (sqrt3 + 1)
    p, logp, _ = O.greedy_sample_walk(lp, tau, 2.0, np.array([[0.9, 0.62]]))
    q = math.sqrt(3.0) / (math.sqrt(3.0) + 1.0)
    assert p[0].tolist() == [1, 0] and abs(logp[0] - math.log(0.5 * q)) < 1e-12


def test_greedy_sample_walk_distribution_is_product_of_step_softmaxes():
    # draws on a regular grid of u reproduce P(path) = prod_t softmax_j(s_t(j_{t-1}, j) / T)(j_t),
    # the step probabilities written out here by enumeration
    lp, tau = _lattice(11, B=1, T=2, K=3)
    temp = 0.9
    paths = list(itertools.product(range(3), repeat=2))

    def step_p(t, prev, j):
        w = [math.exp((float(lp[0, t, c]) + float(tau[0, t, prev, c])) / temp) for c in range(3)]
        return w[j] / sum(w)
    prob = np.array([step_p(0, 0, c[0]) * step_p(1, c[0], c[1]) for c in paths])
    n = 200
    counts = {c: 0 for c in paths}
    for a in range(n):
        for c in range(n):
            u = np.array([[(a + 0.5) / n, (c + 0.5) / n]])
            pth, logp, _ = O.greedy_sample_walk(lp, tau, temp, u)
            key = tuple(int(x) for x in pth[0])
            counts[key] += 1
            assert abs(logp[0] - math.log(prob[paths.index(key)])) < 1e-9
    freq = np.array([counts[c] for c in paths]) / n ** 2
    assert np.abs(freq - prob).max() < 0.02


def test_greedy_sample_walk_low_temperature_is_greedy():
    lp, tau = _lattice(12, B=3, T=5, K=4)
    rng = np.random.default_rng(13)
    gp, _ = O.greedy_walk(lp, tau)
    for _ in range(5):
        p, _, _ = O.greedy_sample_walk(lp, tau, 1e-4, rng.random((3, 5)) * 0.98 + 0.01)
        assert np.array_equal(p, gp)
