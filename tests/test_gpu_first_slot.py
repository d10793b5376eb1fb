"""GPU parity of the first_slot = 1 block reading (DFLASH2_FIRST_SLOT_1: row 0 of each block is
the anchor's own position, block = 1 + the speculative tokens, "RTX 4090 ... DFlash2 vs MTP",
section 4): the conv over every row, candidates and the walk over rows 1..block-1 from the
anchor; with the context gate and with sampling as well. Each call goes through the C ABI."""
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


CASES = {
    # 7 slots after the anchor row; several vocab tiles per CTA, vocab not a multiple of 16
    "b3_t8_h512_v70005": dict(batch=3, block=8, hidden=512, vocab=70_005, layers=2),
    # one slot per sequence (block 2), two row chunks (272 rows)
    "b136_t2_h256_v9001": dict(batch=136, block=2, hidden=256, vocab=9_001, layers=1),
    # the page's hidden size at block 8 (7 slots: the fused select + walk's early gathers)
    "b1_t8_h5120_v30011": dict(batch=1, block=8, hidden=5120, vocab=30_011, layers=5),
    # block 16 (15 slots), rank 272 (two staged chunks per tile)
    "b4_t16_h128_v2000_r272": dict(batch=4, block=16, hidden=128, vocab=2_000, rank=272, layers=3),
}


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("name", sorted(CASES))
def test_draft_tail_first_slot(name, gated):
    rc = synth.scaled_recipe(synth.recipe(2), **CASES[name])
    sh = rc.shape
    sh.first_slot = 1
    sh.gate = gated
    inp = synth.make_inputs(rc)
    ref = O.draft_tail(inp, sh)
    g = P.run_tail(P.shape_of(sh), P.upload_inputs(inp), gated=gated)
    assert g["path_idx"].shape == (sh.batch, sh.block - 1)
    rep = P.check_tail(sh, inp, ref, g)
    print(name, gated, {k: v for k, v in rep.items() if k != "near_tie_rows"})


def test_viterbi_first_slot_takes_slot_arrays():
    # the walk call with the flag takes per-slot arrays of block - 1 slots
    rng = np.random.default_rng(71)
    B, T, K, R, Vv = 5, 9, 16, 256, 2000
    sh = synth.Shape(batch=B, block=T, hidden=64, vocab=Vv, top_k=K, rank=R, layers=0, first_slot=1)
    S = T - 1
    U = synth.normal(13, 3, (Vv, R), 0.2)
    V = synth.normal(13, 4, (Vv, R), 0.2)
    cand = rng.integers(0, Vv, size=(B, S, K)).astype(np.int32)
    lp = (-np.sort(np.abs(rng.standard_normal((B, S, K))), axis=2)).astype(np.float32)
    anchor = rng.integers(0, Vv, size=B).astype(np.int32)
    pid, pix, sc, err = P.run_viterbi(P.shape_of(sh), P.dev(anchor), P.dev(cand), P.dev(lp), P.dev(U), P.dev(V))
    assert err == 0 and pix.shape == (B, S)

    class _S:
        batch, block, top_k = B, S, K
    P.check_walk(_S, anchor, U, V, cand, lp, pix, pid, sc)


def test_first_slot_rejects_block_one():
    import block_drafter_dflash2_gb300 as df2
    shape = df2.Shape.make(2, 1, 64, 100, 4, 16, 1, first_slot=1)
    assert df2.workspace_size(shape) == 0
