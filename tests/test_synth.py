"""The seeded input generator: Philox4x32-10 known-answer vectors (Salmon et al., SC'11,
published test vectors), distribution moments, determinism and the bf16 rounding."""
import numpy as np
import pytest

import synth
from oracle import core as O


def test_philox_known_answers():
    assert synth.philox4x32_10([0, 0, 0, 0], [0, 0]) == (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)
    assert synth.philox4x32_10([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2) == (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)
    assert synth.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344],
                               [0xA4093822, 0x299F31D0]) == (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)


def test_normal_moments_and_determinism():
    a = synth.normal(7, 3, (400_000,), 0.05, "f64")
    assert abs(a.mean()) < 0.05 * 0.01 and abs(a.std() - 0.05) < 0.05 * 0.01
    b = synth.normal(7, 3, (400_000,), 0.05, "f64")
    assert np.array_equal(a, b)
    c = synth.normal(7, 4, (400_000,), 0.05, "f64")
    assert not np.array_equal(a, c)
    # the bf16 and f32 forms are roundings of the same draws
    u = synth.normal(7, 3, (1000,), 0.05, "bf16")
    assert np.array_equal(u, O.round_bf16(a[:1000]))


def test_uniform_int_range_and_anchor_duplicates():
    x = synth.uniform_int(1, 2, 100_000, 248320)
    assert x.min() >= 0 and x.max() < 248320
    rc = synth.recipe(4)
    inp = synth.make_inputs(synth.scaled_recipe(rc, vocab=1000, hidden=64, rank=16), with_lm_head=True)
    anc = inp["anchor"]
    assert len(anc) == 32 and set(anc[24:].tolist()) <= set(anc[:24].tolist())


def test_hidden_rows_rms_normalised():
    rc = synth.scaled_recipe(synth.recipe(2), vocab=512)
    inp = synth.make_inputs(rc)
    h = O.widen(inp["hidden"])
    rms = np.sqrt((h * h).mean(axis=-1))
    assert np.allclose(rms, 1.0, atol=1e-2)


def test_conv_comparator_catches_planted_errors():
    # the comparator used by the GPU tests, fed the oracle's own per-layer outputs with a mistake
    # planted in them: one element of a middle layer 3 % of its scale off, one element of a layer
    # three bf16 units of its operands off (the bound is two), one whole channel of the chain
    # output scaled by 1.5, and a chain output that differs from its last layer by one unit
    from oracle import core as O
    from tests import parity as P
    rc = synth.scaled_recipe(synth.recipe(2), batch=2, block=8, hidden=256, vocab=64, layers=3)
    inp = synth.make_inputs(rc)
    h, w = inp["hidden"], inp["conv_w"]
    layers = []
    x = h
    for l in range(3):
        x = O.conv_chain(x, w[l:l + 1], "bf16", 16)
        layers.append(x)
    ref = O.conv_chain(h, w, "bf16", 16)
    P.check_conv_layers(h, w, "bf16", "softmax", layers, layers[-1], ref_chain=ref)  # the oracle itself: passes

    def planted(l, fn):
        out = [a.copy() for a in layers]
        v = O.widen(out[l]).copy()
        fn(v, O.widen(h if l == 0 else layers[l - 1]))
        out[l] = O.round_bf16(v)
        return out
    bad = planted(1, lambda v, x: v.__setitem__((1, 5, 17), v[1, 5, 17] + 0.03 * max(
        np.sqrt(np.mean(v[1, 5] ** 2)), abs(v[1, 5, 17]), abs(x[1, 5, 17]), abs(x[1, 4, 17]))))
    with pytest.raises(AssertionError):
        P.check_conv_layers(h, w, "bf16", "softmax", bad, bad[-1], ref_chain=ref)

    def three_units(v, x):
        op = max(abs(x[0, 3, 40]), abs(x[0, 2, 40]))
        v[0, 3, 40] += 3 * float(P.bf16_ulp(np.array([op]))[0])
    bad = planted(0, three_units)
    with pytest.raises(AssertionError):
        P.check_conv_layers(h, w, "bf16", "softmax", bad, bad[-1], ref_chain=ref)
    chain = O.widen(layers[-1]).copy()
    chain[:, :, 99] *= 1.5
    with pytest.raises(AssertionError):
        P.check_conv_layers(h, w, "bf16", "softmax", layers, O.round_bf16(chain), ref_chain=ref)
    chain = layers[-1].copy()
    chain[0, 0, 0] ^= 1
    with pytest.raises(AssertionError):
        P.check_conv_layers(h, w, "bf16", "softmax", layers, chain, ref_chain=ref)


def test_planted_rows_reach_the_stated_peaks():
    # the B=8 planted workload: the stored deltas move only the planted tokens' rows, and at a few
    # planted slots (the oracle's own logits over the whole vocabulary) the planted token takes
    # about 85 % of the mass and tops the slot, while its logit at the sequence's other rows stays
    # where it was before planting
    rc = synth.recipe(3)
    sh = rc.shape
    planted = synth.planted_slots(rc)
    assert (planted >= 0).sum() >= 0.95 * planted.size
    inp = synth.make_inputs(rc, apply_planting=False)  # the rows as drawn
    drawn = inp["lm_head"].copy()
    synth.apply_planted_rows(rc, inp["lm_head"], planted)  # what make_inputs returns by default
    changed = np.nonzero(np.any(inp["lm_head"] != drawn, axis=1))[0]
    assert set(changed.tolist()) <= set(planted[planted >= 0].tolist())
    z = O.conv_chain(inp["hidden"], inp["conv_w"], "bf16", 16)
    slots = ((0, 1), (3, 5), (6, 7))
    ls = O.logits(np.stack([z[b, t] for b, t in slots]), inp["lm_head"]).astype(np.float64)  # one pass
    for (b, t), l in zip(slots, ls):
        p = int(planted[b, t])
        assert p >= 0
        lse = l.max() + np.log(np.exp(l - l.max()).sum())
        assert abs(np.exp(l[p] - lse) - synth.PLANT_MASS) < 0.02
        assert int(np.argmax(l)) == p
        others = np.stack([z[b, tt] for tt in range(sh.block) if tt != t])
        before = O.logits(others, drawn[p:p + 1])[:, 0]
        after = O.logits(others, inp["lm_head"][p:p + 1])[:, 0]
        assert np.abs(after.astype(np.float64) - before).max() < 1.0
