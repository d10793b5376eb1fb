"""GPU parity of every step of the draft tail against the CPU oracle, at sizes the
oracle finishes in seconds that still span several tiles, ragged tails and the
edge cases (K < 16, block 1, duplicated anchors and candidates, exact ties, ids out
of range). Each call goes through the C ABI."""
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


# ------------------------------------------------------------------ whole tail, small

CASES = {
    # several 128-wide vocab tiles per CTA plus a narrow ragged last tile, vocab not a multiple of 16
    "b3_t8_h512_v70005": dict(batch=3, block=8, hidden=512, vocab=70_005, layers=2),
    # two row chunks of 128 (160 rows: the second chunk ragged)
    "b20_t8_h256_v20003": dict(batch=20, block=8, hidden=256, vocab=20_003, layers=1),
    # eight row chunks, block 16
    "b64_t16_h256_v8208_r64": dict(batch=64, block=16, hidden=256, vocab=8_208, rank=64, layers=5),
    # vocab smaller than the number of column partitions, K < 16, block 1
    "b4_t1_h128_v100_k4": dict(batch=4, block=1, hidden=128, vocab=100, top_k=4, rank=32, layers=3),
    # no conv layers; rank that is not a multiple of the 128-column staging chunk
    "b2_t5_h64_v999_r272_nl0": dict(batch=2, block=5, hidden=64, vocab=999, rank=272, layers=0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_draft_tail_small(name):
    rc = _recipe(**CASES[name])
    sh = rc.shape
    inp = synth.make_inputs(rc)
    ref = O.draft_tail(inp, sh)
    g = P.run_tail(P.shape_of(sh), P.upload_inputs(inp))
    rep = P.check_tail(sh, inp, ref, g)
    print(name, {k: v for k, v in rep.items() if k != "near_tie_rows"}, "ties", len(rep["near_tie_rows"]))


def test_tiny_fp32_workload():
    rc = synth.recipe(1)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    ref = O.draft_tail(inp, sh)
    g = P.run_tail(P.shape_of(sh), P.upload_inputs(inp))
    P.check_tail(sh, inp, ref, g)
    # the path is the brute-force best of all 4^4 paths over the GPU's candidates
    tau = O.transitions(inp["anchor"], g["cand_ids"], inp["U"], inp["V"])
    bp, bs = O.brute_force_best(g["cand_lp"], tau)
    assert np.array_equal(bp, g["path_idx"])
    assert abs(float(bs[0]) - float(g["score"][0])) < 1e-4


def test_fp32_small_rows():
    rc = _recipe(base=1, batch=3, block=8, vocab=5000, layers=2)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    ref = O.draft_tail(inp, sh)
    g = P.run_tail(P.shape_of(sh), P.upload_inputs(inp))
    P.check_tail(sh, inp, ref, g)


# ------------------------------------------------------------------ per-step calls


def _conv_parity(sh, inp):
    """dflash2_conv on all layers and one layer per call, against the oracle (each layer on the
    GPU's own layer input, and the chain end to end)."""
    shape = P.shape_of(sh)
    x, w = P.dev(inp["hidden"]), P.dev(inp["conv_w"])
    z = P.run_conv(shape, x, w)
    zl = P.run_conv_layers(shape, x, w)
    ref = O.conv_chain(inp["hidden"], inp["conv_w"], sh.dtype, 16, sh.taps)
    return P.check_conv_layers(inp["hidden"], inp["conv_w"], sh.dtype, sh.taps, zl, z, ref_chain=ref)


# 8 and 16 rows run the chain kernel that reads whole rows per CTA; 40, 96, 160 and 256 rows
# the split-K chain (one row tile; one tile; two tiles with a 32-row tail; two full tiles)
@pytest.mark.parametrize("layers,raw,batch", [(1, False, 1), (5, False, 1), (5, False, 2), (1, False, 5),
                                              (5, False, 5), (1, True, 5), (1, False, 12), (5, False, 12),
                                              (1, True, 12), (5, False, 20), (1, True, 20), (5, False, 32)])
def test_conv_step(layers, raw, batch):
    rc = _recipe(batch=batch, block=8, hidden=5120, vocab=64, layers=layers)
    sh = rc.shape
    if raw:
        sh.taps = "raw"
        rc.conv_std = 0.002  # keeps raw taps near unit scale
    inp = synth.make_inputs(rc, with_lm_head=True)
    print(_conv_parity(sh, inp))


def test_conv_step_block16_many_rows():
    rc = _recipe(batch=40, block=16, hidden=1024, vocab=64, layers=5)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    print(_conv_parity(sh, inp))


def test_conv_step_mix_chunks():
    # 4864 rows at hidden 2560: 38 row tiles of two tap tiles leave two K-slices of 20 blocks, so
    # each CTA's 40 channel groups are mixed in two chunks whose row boxes share the operand ring
    rc = _recipe(batch=608, block=8, hidden=2560, vocab=64, layers=2)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    print(_conv_parity(sh, inp))


# at most 8 rows in the chain kernel: sequences shorter than the rows (a sequence start inside
# the row block), fewer channel groups than SMs (one group per CTA), raw taps, one row
@pytest.mark.parametrize("batch,block,hidden,layers,raw", [(2, 4, 5120, 5, False), (1, 3, 1024, 3, False),
                                                           (1, 8, 5120, 2, True), (4, 2, 256, 4, False),
                                                           (1, 1, 512, 1, False)])
def test_conv_step_few_rows(batch, block, hidden, layers, raw):
    rc = _recipe(batch=batch, block=block, hidden=hidden, vocab=64, layers=layers)
    sh = rc.shape
    if raw:
        sh.taps = "raw"
        rc.conv_std = 0.002
    inp = synth.make_inputs(rc)
    print(_conv_parity(sh, inp))


@pytest.mark.parametrize("batch,block,hidden,layers", [(11, 12, 512, 3), (1, 8, 1088, 2), (4, 5, 1088, 2),
                                                      (6, 8, 128, 3), (20, 15, 768, 2)])
def test_conv_step_tile_edges(batch, block, hidden, layers):
    # 132 rows with block 12: sequences cross the 128-row tile boundary and the last tile has
    # 4 rows; hidden 1088 (not a multiple of 256) takes the per-layer path at 8 rows and the
    # split-K chain at 20 rows of block 5, where 136 taps per layer fill a 144-row tap tile;
    # 48 rows at hidden 128 (two K blocks), 300 rows at hidden 768 (three row tiles crossed by
    # sequences of 15)
    rc = _recipe(batch=batch, block=block, hidden=hidden, vocab=64, layers=layers)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    print(_conv_parity(sh, inp))


@pytest.mark.parametrize("B", [1, 2])
def test_conv_shift_limit_exact(B):
    # tap 0 dominant everywhere: z[t] = x[t - layers] exactly (the oracle's pinned special case),
    # for one and two sequences in the row block
    T, H, L = 8, 256, 3
    rng = np.random.default_rng(0)
    x = (rng.integers(1, 32, size=(B, T, H)) / 4.0).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    w = np.zeros((L, 2 * H // 16, H), np.float32)
    w[:, 0::2, :] = 8.0
    w[:, 1::2, :] = -8.0
    wb = (w.view(np.uint32) >> 16).astype(np.uint16)
    import block_drafter_dflash2_gb300 as df2
    shape = df2.Shape.make(B, T, H, 64, 4, 32, L)
    z = O.widen(P.run_conv(shape, P.dev(xb), P.dev(wb)))
    exp = np.zeros_like(x)
    exp[:, L:] = x[:, :T - L]
    assert np.array_equal(z, exp)


# 256 and 512 rows run two and four 128-row chunks per column range; the vocabularies near 16 x 16
# columns per range leave neighbouring ranges with different tile counts; 64 and 40 rows take
# 256-column tiles in one chunk; 200 rows end in a ragged chunk
@pytest.mark.parametrize("M,V,H", [(8, 248_320 // 8, 5120), (256, 30_011, 512), (1, 777, 64), (256, 16_400, 256),
                                   (256, 18_448, 256), (256, 19_472, 256), (512, 20_000, 256), (64, 9_001, 256),
                                   (40, 5_000, 256), (200, 12_345, 256), (300, 7_777, 256)])
def test_select_topk_step(M, V, H):
    rc = _recipe(batch=M, block=1, hidden=H, vocab=V, layers=0)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    rows = inp["hidden"].reshape(M, H)
    l32 = O.logits(rows, inp["lm_head"])
    ids_o, vals_o, _ = O.topk_rows(l32, sh.top_k)
    ref = dict(cand_ids=ids_o, cand_logit=vals_o, max_logit=l32.max(axis=1), lse=O.logsumexp_rows(l32))
    ids, lp, lse = P.run_topk(P.shape_of(sh), P.dev(rows), P.dev(inp["lm_head"]))
    rep = P.check_topk(ref, ids, lp, lse, rows, inp["lm_head"], sh.top_k)
    print(M, V, H, "near-tie rows", len(rep["near_tie_rows"]))


@pytest.mark.parametrize("M", [4, 160])
def test_select_topk_exact_ties_take_lower_ids(M):
    # every logit is an integer; many exact ties, within a column range and across ranges: the kept
    # ids must be the lowest ids among ties (160 rows: the CTA-pair kernel, a ragged second chunk)
    H, V, K = 64, 5000, 16
    z = np.zeros((M, H), np.float32)
    z[np.arange(M), np.arange(M) % 4] = 1.0
    W = np.zeros((V, H), np.float32)
    W[:, :4] = (np.arange(V)[:, None] * np.array([3, 5, 7, 11])[None, :]) % 13
    zb = (z.view(np.uint32) >> 16).astype(np.uint16)
    Wb = (W.view(np.uint32) >> 16).astype(np.uint16)
    import block_drafter_dflash2_gb300 as df2
    shape = df2.Shape.make(M, 1, H, V, K, 32, 0)
    ids, lp, lse = P.run_topk(shape, P.dev(zb), P.dev(Wb))
    l32 = O.logits(zb, Wb)
    ids_o, _, _ = O.topk_rows(l32, K)
    assert np.array_equal(ids, ids_o)
    assert np.allclose(lse, O.logsumexp_rows(l32), atol=1e-4)


@pytest.mark.parametrize("M", [4, 160])
def test_select_topk_monotone_rows(M):
    # rows whose logits rise with the column id (every column beats the kept 16th: the epilogue's
    # candidate loop runs for all 32 columns of every chunk), fall with it (nothing enters after
    # the first chunk), or are all equal (the lowest ids win every tie); exact in bf16:
    # f(v) = (128 + v % 128) * 2^(v // 128) rises strictly with v
    H, V, K = 64, 5000, 16
    v = np.arange(V, dtype=np.float64)
    f = (128 + v % 128) * np.exp2(v // 128)
    W = np.zeros((V, H), np.float32)
    W[:, 0], W[:, 1], W[:, 2] = f, -f, 1.0
    z = np.zeros((M, H), np.float32)
    z[np.arange(M), np.arange(M) % 3] = 1.0
    zb = (z.view(np.uint32) >> 16).astype(np.uint16)
    Wb = (W.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(O.widen(Wb)[:, 0], f)  # exactly representable
    import block_drafter_dflash2_gb300 as df2
    shape = df2.Shape.make(M, 1, H, V, K, 32, 0)
    ids, lp, lse = P.run_topk(shape, P.dev(zb), P.dev(Wb))
    l32 = O.logits(zb, Wb)
    ids_o, _, _ = O.topk_rows(l32, K)
    assert np.array_equal(ids, ids_o)
    assert np.array_equal(ids[0], np.arange(V - 1, V - 1 - K, -1))
    assert np.array_equal(ids[1], np.arange(K)) and np.array_equal(ids[2], np.arange(K))
    assert np.allclose(lse, O.logsumexp_rows(l32), rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("T,K,R", [(8, 16, 256), (1, 16, 256), (16, 4, 64), (32, 1, 16), (3, 16, 384)])
def test_viterbi_step(T, K, R):
    rng = np.random.default_rng(T * 1000 + K * 10 + R)
    B, Vv = 6, 3000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(5, 3, (Vv, R), 0.05)
    V = synth.normal(5, 4, (Vv, R), 0.05)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    cand[0, :, :] = cand[0, :1, :1]  # duplicated candidates everywhere in sequence 0
    lp = (-np.sort(np.abs(rng.standard_normal((B, T, K))), axis=2) * 2).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    anchor[-1] = anchor[0]  # shared anchors
    pid, pix, sc, err = P.run_viterbi(P.shape_of(sh), P.dev(anchor), P.dev(cand), P.dev(lp), P.dev(U), P.dev(V))
    assert err == 0
    P.check_walk(sh, anchor, U, V, cand, lp, pix, pid, sc)


def test_greedy_walk_step():
    rng = np.random.default_rng(3)
    B, T, K, R, Vv = 5, 8, 16, 256, 2000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(6, 3, (Vv, R), 0.3)
    V = synth.normal(6, 4, (Vv, R), 0.3)
    cand = rng.integers(0, Vv, size=(B, T, K)).astype(np.int32)
    lp = (-np.sort(np.abs(rng.standard_normal((B, T, K))), axis=2)).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    shape = P.shape_of(sh, greedy=True)
    pid, pix, sc, err = P.run_viterbi(shape, P.dev(anchor), P.dev(cand), P.dev(lp), P.dev(U), P.dev(V))
    tau = O.transitions(anchor, cand, U, V)
    gp, gs = O.greedy_walk(lp, tau)
    vp, vs = O.viterbi(lp, tau)
    assert np.array_equal(pix, gp)
    assert np.allclose(sc, gs, atol=1e-4)
    assert np.all(sc <= vs + 1e-4)


def test_out_of_range_ids_set_the_error_word_and_clamp():
    B, T, K, R, Vv = 2, 4, 4, 32, 100
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0)
    U = synth.normal(7, 3, (Vv, R), 0.05)
    V = synth.normal(7, 4, (Vv, R), 0.05)
    cand = np.tile(np.arange(K, dtype=np.int32), (B, T, 1))
    lp = np.zeros((B, T, K), np.float32)
    anchor = np.array([5, Vv + 7], np.int32)
    import block_drafter_dflash2_gb300 as df2
    pid, pix, sc, err = P.run_viterbi(P.shape_of(sh), P.dev(anchor), P.dev(cand), P.dev(lp), P.dev(U), P.dev(V))
    assert err == df2.DEVERR_ANCHOR_RANGE
    cand[1, 2, 3] = -4
    anchor[1] = 3
    pid, pix, sc, err = P.run_viterbi(P.shape_of(sh), P.dev(anchor), P.dev(cand), P.dev(lp), P.dev(U), P.dev(V))
    assert err == df2.DEVERR_CANDIDATE_RANGE
    assert np.all((pid >= 0) & (pid < Vv))


def test_argument_errors_return_before_launch():
    import ctypes
    import block_drafter_dflash2_gb300 as df2
    rc = _recipe(batch=1, block=8, hidden=256, vocab=1000, layers=1)
    shape = P.shape_of(rc.shape)
    inp = synth.make_inputs(rc)
    d = P.upload_inputs(inp)
    ws = P.workspace(shape)
    B, T, K = 1, 8, 16
    o = [torch.empty((B, T), dtype=torch.int32, device="cuda"), torch.empty((B, T), dtype=torch.int32, device="cuda"),
         torch.empty((B,), dtype=torch.float32, device="cuda")]
    with pytest.raises(df2.DFlash2Error) as e:
        df2.draft_tail(shape, d["hidden"], d["lm_head"], d["U"], d["V"], d["conv_w"], d["anchor"], *o,
                       (ws.data_ptr(), ws.numel() - 1))
    assert e.value.status == df2.ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(df2.DFlash2Error) as e:
        df2.draft_tail(shape, d["hidden"].data_ptr() + 2, d["lm_head"], d["U"], d["V"], d["conv_w"], d["anchor"],
                       *o, ws)
    assert e.value.status == df2.ERR_INVALID_ARGUMENT
    lib = df2.load()
    st = lib.dflash2_draft_tail(ctypes.byref(shape), d["hidden"].data_ptr(), None, d["U"].data_ptr(),
                                d["V"].data_ptr(), d["conv_w"].data_ptr(), d["anchor"].data_ptr(),
                                o[0].data_ptr(), o[1].data_ptr(), o[2].data_ptr(), None, None, None,
                                ws.data_ptr(), ws.numel(), None)
    assert st == df2.ERR_INVALID_ARGUMENT
    torch.cuda.synchronize()
    assert df2.read_device_error(ws) == 0


@pytest.mark.parametrize("greedy", [False, True])
def test_draft_tail_score_on_logits(greedy):
    # DFLASH2_SCORE_LOGITS: same candidates and path; the score is the log-softmax score plus the
    # slots' lse (the pages' per-slot score is the drafter's raw logit)
    import block_drafter_dflash2_gb300 as df2
    rc = _recipe(batch=3, block=8, hidden=512, vocab=20_011, layers=2)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    d = P.upload_inputs(inp)
    base = P.shape_of(sh, greedy=greedy)
    flagged = df2.Shape.make(sh.batch, sh.block, sh.hidden, sh.vocab, sh.top_k, sh.rank, sh.layers,
                             greedy=greedy, score_logits=True)
    g0 = P.run_tail(base, d)
    g1 = P.run_tail(flagged, d)
    for k in ("path_ids", "path_idx", "cand_ids", "cand_lp", "lse"):
        assert np.array_equal(g0[k], g1[k]), k
    lse_sum = g1["lse"].astype(np.float64).sum(axis=1)
    assert np.allclose(g1["score"].astype(np.float64), g0["score"].astype(np.float64) + lse_sum, atol=1e-4, rtol=0)
    # against the oracle end to end: its path score on its own raw logits
    ref = O.draft_tail(inp, sh)
    raw = O.path_score(ref["cand_logit"].astype(np.float64), ref["tau"], ref["path_idx"]) if not greedy else None
    if raw is not None:
        for b in range(sh.batch):
            if np.array_equal(g1["path_idx"][b], ref["path_idx"][b]):
                assert abs(float(g1["score"][b]) - raw[b]) <= P.SCORE_TOL
    # the walk-only call has no lse: the flag is refused there
    ws = P.workspace(flagged)
    B, T, K = sh.batch, sh.block, sh.top_k
    o = [torch.empty((B, T), dtype=torch.int32, device="cuda"), torch.empty((B, T), dtype=torch.int32, device="cuda"),
         torch.empty((B,), dtype=torch.float32, device="cuda")]
    with pytest.raises(df2.DFlash2Error) as e:
        df2.viterbi(flagged, d["anchor"], P.dev(g1["cand_ids"]), P.dev(g1["cand_lp"]), d["U"], d["V"], *o, ws)
    assert e.value.status == df2.ERR_UNSUPPORTED
