"""The fused Mamba-2 fold + decode step (replayssm_mamba2_fold_decode).

Each call must give what consolidate(k_next=1) followed by a decode gives:
outputs within the parity tolerances of the oracle, ring bytes and pointers
bit-exact, the folded checkpoint within the checkpoint tolerance, and the
read copy equal to the BF16 rounding of the checkpoint. Cases cover the
fused kernel (lockstep folds, staggered folds mixed with plain decodes in one
call, W = 1, FP32 and BF16 read, FP32 and BF16 inputs, two B/C groups,
N = 64) and the two-launch path it takes for W > 16 or a read-copy row block
that is not a multiple of 64 rows.
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
            s.join([(t // 3) % s.wl.batch], seed=2000 + t)
        snap = s.snapshot() if t in all_units_at else None
        y, _, fold = s.fold_decode(t)
        if snap is not None:
            s.check_all_units(snap, s.last_tok, y, f"fused step {t}")
        folds += int(fold.sum())
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
    # the small Mamba-2 workload: FP32 inputs, 64 steps (four lockstep folds)
    "tiny": dict(batch=4, heads=8, P=64, N=128, window=16, steps=64, in_dtype="f32", seed=1),
    # two B/C groups, N = 64, W = 8
    "groups_n64": dict(batch=3, heads=6, P=64, N=64, groups=2, window=8, steps=30,
                       in_dtype="bf16", seed=21),
    # P = 128: two 64-row blocks per head
    "p128": dict(batch=2, heads=4, P=128, N=128, window=6, steps=20, in_dtype="bf16", seed=22),
    # W = 1: every step after the first folds
    "w1": dict(batch=3, heads=4, P=64, N=128, window=1, steps=9, in_dtype="bf16", seed=23),
    # P = 96: the BF16 read copy takes the two-launch path, the FP32 read the fused one
    "p96": dict(batch=5, heads=6, P=96, N=64, groups=2, window=5, steps=23, in_dtype="bf16",
                seed=24),
    # W = 20 > 16: two launches
    "w20": dict(batch=2, heads=4, P=64, N=128, window=20, steps=45, in_dtype="bf16", seed=25),
}


@pytest.mark.parametrize("read", ["f32", "bf16"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_matches_oracle(case, read):
    wl = synth.Mamba2Workload(**CASES[case])
    folds = run(Session("mamba2", wl, read), wl.steps, check_every=5)
    assert folds > 0


@pytest.mark.parametrize("read", ["f32", "bf16"])
@pytest.mark.parametrize("case", ["tiny", "groups_n64", "p128", "w1"])
def test_tensor_core_fold_matches_oracle(case, read, monkeypatch):
    """The same parity bar with the fold units' update on the tensor cores
    (REPLAYSSM_FOLD_TENSOR_CORES=1: mma.sync with TF32 operands split in two)."""
    monkeypatch.setenv("REPLAYSSM_FOLD_TENSOR_CORES", "1")
    wl = synth.Mamba2Workload(**CASES[case])
    assert run(Session("mamba2", wl, read), wl.steps, check_every=5) > 0


@pytest.mark.parametrize("read", ["f32", "bf16"])
@pytest.mark.parametrize("batch,heads", [(6, 4), (24, 32)])
def test_staggered_phases(read, batch, heads):
    """Slots change hands, so each call mixes folding and plain sequences;
    with 24 x 32 heads every block holds several units of both kinds."""
    wl = synth.Mamba2Workload(batch=batch, heads=heads, P=64, N=128, window=8, steps=30,
                              seed=26)
    run(Session("mamba2", wl, read), wl.steps, check_every=3, joins=True)


def test_no_optional_ring_fields():
    wl = synth.Mamba2Workload(batch=2, heads=4, P=64, N=128, window=4, steps=11, seed=27)
    run(Session("mamba2", wl, "bf16", store_optional=False), wl.steps, check_every=2)


@pytest.mark.parametrize("read", ["f32", "bf16"])
def test_same_as_two_calls(read):
    """Against consolidate + decode on an identical state: ring bytes and
    pointers equal; checkpoints equal up to FP32 rounding order; outputs too
    with the FP32 read path. With the BF16 read copy a different rounding
    order can move a folded element across a BF16 rounding boundary (one
    BF16 ulp, about 0.8% of the element), so outputs are held to the BF16
    read-path bar there."""
    wl = synth.Mamba2Workload(batch=8, heads=16, P=64, N=128, window=16, steps=40, seed=28)
    a = Session("mamba2", wl, read)
    b = Session("mamba2", wl, read)
    for t in range(wl.steps):
        tok = a._to_dev(a.token(t))
        ya = torch.empty((wl.batch, wl.heads, wl.P), device="cuda")
        yb = torch.empty_like(ya)
        api.consolidate(a.dims, a.state, a.dA, 1, False)
        api.mamba2_decode(a.dims, a.state, a.dA, a.dD, tok["x"], tok["B"], tok["C"], tok["dt"], ya)
        api.mamba2_fold_decode(b.dims, b.state, b.dA, b.dD, tok["x"], tok["B"], tok["C"],
                               tok["dt"], yb)
        if read == "f32":
            f32_close(host(yb), host(ya), f"step {t}: y", atol=1e-5, rtol=1e-5)
        else:
            bf16_close(host(yb), host(ya), f"step {t}: y")
        for name in ("ring_head", "ring_len", "status", "sync"):
            assert torch.equal(getattr(a.state, name), getattr(b.state, name)), f"step {t}: {name}"
        for k in a.state.ring:
            assert torch.equal(a.state.ring[k], b.state.ring[k]), f"step {t}: ring {k}"
    f32_close(host(b.state.S_ckpt), host(a.state.S_ckpt), "checkpoint", atol=1e-6, rtol=1e-6)
    if read == "bf16":
        rd = b.state.S_read.view(torch.int16)
        assert torch.equal(rd, b.state.S_ckpt.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("read", ["bf16", "f32"])
def test_full_size_sampled(read):
    """b256, H128, P64, N128, W16, 256 steps (16 lockstep folds), BF16 read
    copy or FP32 read path. The oracle follows every head of 8 sequences
    spread over the batch; at three steps that fold nothing every (sequence,
    head) output is also checked against the replay formula on the GPU's own
    checkpoint copy and ring."""
    wl = synth.Mamba2Workload(batch=256, heads=128, P=64, N=128, window=16, steps=256,
                              in_dtype="bf16", seed=2)
    s = Session("mamba2", wl, read, seqs=spread(wl.batch))
    assert run(s, wl.steps, check_every=37, all_units_at=(3, 77, 250)) > 0


def test_full_size_staggered_sampled():
    """The same layer with sequence s at ring phase s mod W (a sixteenth of
    the batch folds in every call); oracle on a sample of all phases."""
    wl = synth.Mamba2Workload(batch=256, heads=128, P=64, N=128, window=16, steps=20,
                              in_dtype="bf16", seed=2)
    seqs = list(range(0, 256, 17))
    s = Session("mamba2", wl, "bf16", seqs=seqs, heads=[0, 127])
    # phases: slot s restarts from its checkpoint before step s mod W
    phase = np.arange(wl.batch) % wl.window
    for t in range(wl.window):
        s.join(np.nonzero(phase == t)[0], seed=3000 + t)
        s.fold_decode(t)
    lens = host(s.state.ring_len)
    assert len(set(lens.tolist())) == wl.window
    for t in range(wl.window, wl.steps):
        _, _, fold = s.fold_decode(t)
        s.check_pointers(f"step {t}")
    s.check_ring("end")
    s.consolidate(1, force=True)
    s.check_checkpoint("end")
