"""The fused Gated DeltaNet / KDA fold + decode step (replayssm_gdn_fold_decode).

Each call must give what consolidate(k_next=1) followed by a decode gives:
outputs within the parity tolerances of the oracle, ring bytes and pointers
bit-exact, the folded checkpoint within the checkpoint tolerance, and the
read copy equal to the BF16 rounding of the checkpoint. Cases cover lockstep
folds, staggered folds mixed with plain decodes in one call, W = 1, both
read paths, FP32 and BF16 inputs, d_k = 64 with d_v = 96, a d_v of 256 (two
row chunks per head in the fold), long rings, the full-size layer, and a
comparison with the two calls on an identical state.
"""

import numpy as np
import pytest
import torch

import synth
from gpu_harness import Session, bf16_close, f32_close, host, spread
from recurrent_state_fp32_b300 import api

pytestmark = pytest.mark.gpu


def run(s, steps, check_every=8, joins=False, all_units_at=()):
    folds = 0
    for t in range(steps):
        if joins and t % 3 == 0:  # a slot changes hands: ring phases spread
            s.join([(t // 3) % s.wl.batch], seed=4000 + t)
        snap = s.snapshot() if t in all_units_at else None
        y, _, fold = s.fold_decode(t)
        folds += int(fold.sum())
        if snap is not None:
            s.check_all_units(snap, s.last_tok, y, f"fused step {t}")
        if t % check_every == 0:
            s.check_pointers(f"step {t}")
            s.check_ring(f"step {t}")
    s.check_pointers("end")
    s.check_ring("end")
    s.consolidate(1, force=True)
    s.check_pointers("after forced fold")
    s.check_checkpoint("after forced fold")
    return folds


CASES = {
    "small": dict(batch=3, heads=4, dk=128, dv=128, window=16, steps=40, in_dtype="bf16", seed=71),
    "ragged_f32in": dict(batch=5, heads=3, dk=64, dv=96, window=7, steps=25, in_dtype="f32",
                         seed=72),
    "w1": dict(batch=3, heads=2, dk=128, dv=64, window=1, steps=9, in_dtype="bf16", seed=73),
    "dv256": dict(batch=2, heads=2, dk=128, dv=256, window=5, steps=17, in_dtype="bf16", seed=74),
    "long_ring": dict(batch=2, heads=2, dk=128, dv=128, window=40, steps=84, in_dtype="f32",
                      seed=75),
}


@pytest.mark.parametrize("read", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["gdn", "kda"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_matches_oracle(case, kind, read):
    wl = synth.DeltaWorkload(kind, **CASES[case])
    folds = run(Session(kind, wl, read, scale=0.8), wl.steps, check_every=5)
    assert folds > 0


@pytest.mark.parametrize("kind,read", [("gdn", "bf16"), ("kda", "f32")])
def test_staggered_phases(kind, read):
    """Slots change hands, so each call mixes folding and plain sequences."""
    wl = synth.DeltaWorkload(kind, batch=12, heads=4, dk=128, dv=128, window=8, steps=30,
                             in_dtype="bf16", seed=76)
    run(Session(kind, wl, read), wl.steps, check_every=3, joins=True)


def test_no_optional_ring_fields():
    wl = synth.DeltaWorkload("gdn", batch=2, heads=3, dk=128, dv=64, window=4, steps=11, seed=77)
    run(Session("gdn", wl, "bf16", store_optional=False), wl.steps, check_every=2)


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_same_as_two_calls(kind):
    """Against consolidate + decode on an identical state: ring bytes and
    pointers equal; checkpoints equal up to FP32 rounding order; outputs held
    to the BF16 read-path bar (a different rounding order can move a folded
    element across a BF16 rounding boundary)."""
    wl = synth.DeltaWorkload(kind, batch=6, heads=4, dk=128, dv=128, window=16, steps=40,
                             in_dtype="bf16", seed=78)
    a, b = Session(kind, wl, "bf16"), Session(kind, wl, "bf16")
    for t in range(wl.steps):
        tok = a._to_dev(a.token(t))
        ya = torch.empty((wl.batch, wl.heads, wl.dv), device="cuda")
        yb = torch.empty_like(ya)
        api.consolidate(a.dims, a.state, None, 1, False)
        api.gdn_decode(a.dims, a.state, tok["q"], tok["k"], tok["v"], tok["alpha"], tok["beta"],
                       1.0, ya)
        api.gdn_fold_decode(b.dims, b.state, tok["q"], tok["k"], tok["v"], tok["alpha"],
                            tok["beta"], 1.0, yb)
        bf16_close(host(yb), host(ya), f"step {t}: y")
        for name in ("ring_head", "ring_len", "status", "sync"):
            assert torch.equal(getattr(a.state, name), getattr(b.state, name)), f"step {t}: {name}"
        for k in a.state.ring:
            assert torch.equal(a.state.ring[k], b.state.ring[k]), f"step {t}: ring {k}"
    f32_close(host(b.state.S_ckpt), host(a.state.S_ckpt), "checkpoint", atol=1e-6, rtol=1e-6)
    rd = b.state.S_read.view(torch.int16)
    assert torch.equal(rd, b.state.S_ckpt.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_full_size_sampled(kind):
    """b256, H32, d_k = d_v = 128, W16, 256 steps (16 lockstep folds), BF16
    read copy; every head of 8 spread sequences against the oracle, every
    unit at three steps that fold nothing."""
    wl = synth.DeltaWorkload(kind, batch=256, heads=32, dk=128, dv=128, window=16, steps=256,
                             in_dtype="bf16", seed=3 if kind == "gdn" else 5)
    s = Session(kind, wl, "bf16", seqs=spread(wl.batch))
    assert run(s, wl.steps, check_every=37, all_units_at=(3, 77, 250)) > 0


def test_full_size_staggered_sampled():
    """The GDN layer with sequence s at ring phase s mod W (a sixteenth of
    the batch folds in every call)."""
    wl = synth.DeltaWorkload("gdn", batch=256, heads=32, dk=128, dv=128, window=16, steps=24,
                             in_dtype="bf16", seed=3)
    s = Session("gdn", wl, "bf16", seqs=list(range(0, 256, 17)))
    phase = np.arange(wl.batch) % wl.window
    for t in range(wl.window):
        s.join(np.nonzero(phase == t)[0], seed=5000 + t)
        s.fold_decode(t)
    assert len(set(host(s.state.ring_len).tolist())) == wl.window
    for t in range(wl.window, wl.steps):
        s.fold_decode(t)
        s.check_pointers(f"step {t}")
    s.check_ring("end")
    s.consolidate(1, force=True)
    s.check_checkpoint("end")
