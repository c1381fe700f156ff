"""The seeded input generators: determinism, ranges, bfloat16 storage rounding."""

import json
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_bf16_round_golden():
    g = json.load(open(os.path.join(GOLDEN, "worked_examples.json")))["bf16_rne"]
    out = synth.bf16_round(np.array(g["in"], np.float32))
    assert out.tolist() == g["out"]


def test_bf16_round_is_representable_and_nearest():
    r = np.random.default_rng(0)
    a = r.standard_normal(10000).astype(np.float32)
    b = synth.bf16_round(a)
    assert np.all(b.view(np.uint32) & 0xFFFF == 0)
    # nearest: error at most half a bf16 ulp (2^-8 relative to the binade)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(a))) - 7)
    assert np.all(np.abs(b.astype(np.float64) - a) <= ulp / 2 + 1e-30)


def test_deterministic_and_step_indexed():
    A, D, bias = synth.mamba2_params(2, 8)
    s1 = synth.mamba2_step_inputs(2, 5, 3, 8, 1, 4, 16, bias)
    s2 = synth.mamba2_step_inputs(2, 5, 3, 8, 1, 4, 16, bias)
    s3 = synth.mamba2_step_inputs(2, 6, 3, 8, 1, 4, 16, bias)
    for k in s1:
        assert np.array_equal(s1[k], s2[k])
        assert not np.array_equal(s1[k], s3[k])


def test_mamba2_ranges():
    A, D, bias = synth.mamba2_params(2, 128)
    assert np.all((A <= -1.0) & (A >= -16.0))
    s = synth.mamba2_step_inputs(2, 0, 64, 128, 1, 8, 128, bias, "bf16")
    assert s["x"].shape == (64, 128, 8) and s["B"].shape == (64, 1, 128)
    assert np.all((s["dt"] >= 1e-3) & (s["dt"] <= 0.1))
    assert np.all(s["x"].view(np.uint32) & 0xFFFF == 0)
    h = synth.mamba2_initial_state(2, 2, 4, 8, 16)
    assert h.dtype == np.float32 and abs(h.std() - 0.1) < 0.02


def test_delta_ranges():
    for kind in ("gdn", "kda"):
        s = synth.delta_step_inputs(3, 0, 16, 4, 128, 64, kind, "f32")
        assert np.allclose(np.linalg.norm(s["k"], axis=-1), 1.0, atol=1e-5)
        assert np.allclose(np.linalg.norm(s["q"], axis=-1), 1.0, atol=1e-5)
        assert s["alpha"].shape == ((16, 4) if kind == "gdn" else (16, 4, 128))
        assert np.all((s["alpha"] > 0.9) & (s["alpha"] < 1.0))
        assert np.all((s["beta"] > 0.0) & (s["beta"] < 1.0))
    d = synth.spec_draft_inputs(4, 0, 8, 4, 2, 128, 128)
    assert d["q"].shape == (8, 4, 2, 128)
    m = synth.accept_counts(4, 0, 10000, 4)
    assert m.min() == 0 and m.max() == 4 and m.dtype == np.int32
