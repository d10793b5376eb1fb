"""dflash2_select_topk_noalloc: the top-K selection with the library's own fixed device
scratch, for callers that cannot allocate device memory at the call. Checked through the C
ABI against dflash2_select_topk (which uses a caller workspace) on two calls in a row, so the
second call also shows that what the first left in the shared scratch does not leak into it.
Kept in a file of its own that runs last."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import core as O
from tests import parity as P

pytestmark = pytest.mark.gpu


def _inputs(M, V, H, seed):
    rc = synth.scaled_recipe(synth.recipe(2), batch=M, block=1, hidden=H, vocab=V, layers=0)
    rc.seed = seed
    inp = synth.make_inputs(rc)
    return rc.shape, inp["hidden"].reshape(M, H), inp["lm_head"]


def _call_noalloc(lib, shape, rows, lm_head, M, K, with_lse=True):
    ids = torch.full((M, K), -1, dtype=torch.int32, device="cuda:0")
    lp = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda:0")
    lse = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda:0")
    st = lib.dflash2_select_topk_noalloc(ctypes.byref(shape), rows.data_ptr(), lm_head.data_ptr(), ids.data_ptr(),
                                         lp.data_ptr(), lse.data_ptr() if with_lse else None,
                                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0, f"status {st}"
    return P.host(ids), P.host(lp), P.host(lse)


def test_noalloc_matches_workspace_call_twice():
    import block_drafter_dflash2_gb300 as df2
    lib = df2.load()
    cases = [(8, 31040 + 7, 5120, 11), (40, 20011, 512, 12)]  # two different shapes, back to back
    for M, V, H, seed in cases:
        sh, rows, lm_head = _inputs(M, V, H, seed)
        shape = P.shape_of(sh)
        d_rows, d_w = P.dev(rows), P.dev(lm_head)
        ids_ref, lp_ref, lse_ref = P.run_topk(shape, d_rows, d_w)
        for _ in range(2):
            ids, lp, lse = _call_noalloc(lib, shape, d_rows, d_w, M, sh.top_k)
            assert np.array_equal(ids, ids_ref)
            assert np.abs(lp - lp_ref).max() <= P.LP_TOL
            assert np.abs(lse - lse_ref).max() <= P.LSE_TOL
        # without an lse output (the merge keeps it in the scratch): same ids and log-probs
        ids_n, lp_n, _ = _call_noalloc(lib, shape, d_rows, d_w, M, sh.top_k, with_lse=False)
        assert np.array_equal(ids_n, ids_ref)
        assert np.abs(lp_n - lp_ref).max() <= P.LP_TOL
        # and it is the right selection: same comparator as the other top-K tests
        l32 = O.logits(rows, lm_head)
        i_o, v_o, _ = O.topk_rows(l32, sh.top_k)
        ref = dict(cand_ids=i_o, cand_logit=v_o, max_logit=l32.max(axis=1), lse=O.logsumexp_rows(l32))
        P.check_topk(ref, ids, lp, lse, rows, lm_head, sh.top_k)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import block_drafter_dflash2_gb300 as df2
    lib = df2.load()
    # 65536 rows: the partials need about twice the 4 MiB scratch
    shape = df2.Shape.make(8192, 8, 512, 100_000, 16, 256, 0)
    x = torch.zeros(16, dtype=torch.int16, device="cuda:0")
    st = lib.dflash2_select_topk_noalloc(ctypes.byref(shape), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                         x.data_ptr(), None, None)
    assert st == df2.ERR_WORKSPACE_TOO_SMALL
