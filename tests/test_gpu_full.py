"""Parity at the full workload sizes (vocabulary 248,320, hidden 5120, 5 conv layers), in the
launch configuration the benchmark times (dflash2_draft_tail on the same shapes).

The oracle recomputes a sample of sequences end to end; on every sequence the properties
that hold at any size are checked: candidates are distinct, sorted, valid log-probabilities
(sum of their probabilities <= 1, the largest one matching a direct dot product), the path is
made of the slot candidates, and the walk is exact on the GPU's own candidates (the oracle
Viterbi over transitions recomputed from U and V).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import core as O
from tests import parity as P

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# workload -> sequences the oracle recomputes end to end
SAMPLES = {2: [0], 3: list(range(8)), 4: [0, 9, 26, 31], 5: [0, 1, 32, 63]}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import block_drafter_dflash2_gb300 as df2
    assert torch.cuda.is_available()
    df2.load()


@pytest.mark.parametrize("config", [2, 3, 4, 5])
def test_full_size_workload(config):
    rc = synth.recipe(config)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    B, T, K, H = sh.batch, sh.block, sh.top_k, sh.hidden
    g = P.run_tail(P.shape_of(sh), P.upload_inputs(inp))
    assert g["device_error"] == 0

    # --- properties on every sequence
    ids = g["cand_ids"].reshape(B * T, K)
    lp = g["cand_lp"].reshape(B * T, K)
    assert np.all((ids >= 0) & (ids < sh.vocab))
    assert all(len(set(r.tolist())) == K for r in ids)
    assert np.all(np.diff(lp, axis=1) <= 0)             # sorted by logit, descending
    assert np.all(lp <= 1e-4)                           # log-probabilities (fp32 rounding allowed)
    assert np.all(np.exp(lp.astype(np.float64)).sum(axis=1) <= 1 + 1e-4)
    P.check_walk(sh, inp["anchor"], inp["U"], inp["V"], g["cand_ids"], g["cand_lp"], g["path_idx"],
                 g["path_ids"], g["score"])

    # --- end-to-end oracle on the sampled sequences
    seqs = SAMPLES[config]
    ref = O.draft_tail(inp, sh, seqs=seqs)
    rep = P.check_tail(sh, inp, ref, g, seqs=seqs)
    print(f"workload {config}: near-tie rows {len(rep['near_tie_rows'])}, lse err {rep['lse_max_err']:.2e}, "
          f"lp err {rep['lp_max_err']:.2e}, conv row rel {rep['conv_row_rel_max']:.2e}, paths differing at "
          f"small margins {rep['path_vs_oracle_mismatch_small_margin']}; end to end: same ids "
          f"{rep['e2e_rows_same_ids']:.3f}, same sets {rep['e2e_rows_same_set']:.3f}, same paths "
          f"{rep['e2e_paths_same']:.3f}, lse err {rep['e2e_lse_max_err']:.2e}")


@pytest.mark.parametrize("config", [2, 4])
def test_full_size_workload_gated(config):
    # the context gate at full size: the gate rows formed in the LM-head pass over the whole
    # vocabulary plus the 256 gate columns, the gated walk exact on the GPU's own candidates
    # and gate rows, and the oracle end to end on sampled sequences
    rc = synth.recipe(config)
    sh = rc.shape
    sh.gate = True
    inp = synth.make_inputs(rc)
    B, T, R = sh.batch, sh.block, sh.rank
    g = P.run_tail(P.shape_of(sh), P.upload_inputs(inp), gated=True)
    assert g["device_error"] == 0
    assert g["gate"].shape == (B, T, R) and np.all(np.isfinite(g["gate"]))
    P.check_walk(sh, inp["anchor"], inp["U"], inp["V"], g["cand_ids"], g["cand_lp"], g["path_idx"],
                 g["path_ids"], g["score"], gate=g["gate"])
    seqs = SAMPLES[config]
    ref = O.draft_tail(inp, sh, seqs=seqs)
    rep = P.check_tail(sh, inp, ref, g, seqs=seqs)
    print(f"workload {config} gated: gate err {rep['gate_max_abs_err']:.2e}, paths differing at small margins "
          f"{rep['path_vs_oracle_mismatch_small_margin']}, same paths {rep['e2e_paths_same']:.3f}")
