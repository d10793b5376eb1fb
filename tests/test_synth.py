"""The seeded input generator: Philox4x32-10 known-answer vectors (Salmon et al., SC'11,
published test vectors), distribution moments, determinism and the bf16 rounding."""
import numpy as np

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
