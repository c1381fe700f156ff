"""Mamba-2 replay decode, consolidate and conventional step: CUDA path vs oracle."""

import numpy as np
import pytest
import torch

import synth
from gpu_harness import Session, dev, f32_close, host, spread
from oracle import recurrences as rec
from recurrent_state_fp32_b300 import api

pytestmark = pytest.mark.gpu


def run(s, steps, check_every=8, all_units_at=()):
    for t in range(steps):
        s.consolidate(1)
        snap = s.snapshot() if t in all_units_at else None
        y, _ = s.decode(t)
        if snap is not None:
            s.check_all_units(snap, s.last_tok, y, f"step {t}")
        if t % check_every == 0:
            s.check_pointers(f"step {t}")
            s.check_ring(f"step {t}")
    s.check_pointers("end")
    s.check_ring("end")
    s.consolidate(1, force=True)
    s.check_pointers("after forced fold")
    s.check_checkpoint("after forced fold")


@pytest.mark.parametrize("read", ["f32", "bf16"])
def test_tiny_layer(read):
    """b4, H8, P64, N128, W16, 64 steps, FP32 inputs (the small Mamba-2 workload)."""
    wl = synth.Mamba2Workload(batch=4, heads=8, P=64, N=128, window=16, steps=64,
                              in_dtype="f32", seed=1)
    run(Session("mamba2", wl, read), wl.steps)


@pytest.mark.parametrize("read", ["f32", "bf16"])
def test_ragged_shapes(read):
    """Heads not a multiple of the block's head group, 2 B/C groups, P = 96, N = 64, W = 5."""
    wl = synth.Mamba2Workload(batch=5, heads=6, P=96, N=64, groups=2, window=5, steps=23,
                              in_dtype="bf16", seed=7)
    run(Session("mamba2", wl, read), wl.steps, check_every=3)


def test_window_one_folds_every_token():
    wl = synth.Mamba2Workload(batch=3, heads=4, P=64, N=128, window=1, steps=9,
                              in_dtype="bf16", seed=8)
    s = Session("mamba2", wl, "f32")
    for t in range(wl.steps):
        fold = s.consolidate(1)
        assert fold.all() == (t > 0)
        s.decode(t)
        s.check_pointers()
        s.check_ring()
    s.consolidate(1, force=True)
    s.check_checkpoint()


def test_no_optional_ring_fields():
    wl = synth.Mamba2Workload(batch=2, heads=4, P=64, N=128, window=4, steps=11, seed=9)
    run(Session("mamba2", wl, "bf16", store_optional=False), wl.steps, check_every=2)


def test_full_ring_is_refused_and_untouched():
    wl = synth.Mamba2Workload(batch=3, heads=4, P=64, N=128, window=4, steps=6, seed=10)
    s = Session("mamba2", wl, "bf16")
    for t in range(4):
        s.decode(t)
    ring = {k: v.clone() for k, v in s.state.ring.items()}
    y, ref = s.decode(4)  # no consolidate: every ring is full
    assert torch.isnan(y).all()
    s.check_pointers()
    assert all(torch.equal(ring[k], s.state.ring[k]) for k in ring)
    assert (s.state.status.cpu().numpy() == api._abi.SEQ_RING_FULL).all()
    s.consolidate(1)
    s.decode(5)  # recovers after consolidating
    s.check_pointers()


def test_forced_fold_with_empty_ring_is_a_noop():
    wl = synth.Mamba2Workload(batch=2, heads=4, P=64, N=128, window=16, seed=11)
    s = Session("mamba2", wl, "bf16")
    before = s.state.S_ckpt.clone()
    fold = s.consolidate(1, force=True)
    assert not fold.any()
    assert torch.equal(before, s.state.S_ckpt)
    s.check_pointers()


@pytest.mark.parametrize("read", ["bf16", "f32"])
def test_full_size_sampled(read):
    """b256, H128, P64, N128, W16, 256 steps, BF16 inputs, BF16 read copy or
    FP32 read path. The oracle follows every head of 8 sequences spread over
    the batch; at three steps every (sequence, head) output is also checked
    against the replay formula on the GPU's own checkpoint copy and ring."""
    wl = synth.Mamba2Workload(batch=256, heads=128, P=64, N=128, window=16, steps=256,
                              in_dtype="bf16", seed=2)
    s = Session("mamba2", wl, read, seqs=spread(wl.batch))
    run(s, wl.steps, check_every=37, all_units_at=(5, 120, 250))


@pytest.mark.parametrize("N,P", [(128, 64), (64, 96)])
def test_conventional_step(N, P):
    b, H, G = 3, 4, 2
    A, D, bias = synth.mamba2_params(5, H)
    S0 = synth.mamba2_initial_state(5, b, H, P, N)
    dims = api.LayerDims("mamba2", b, H, dk=N, dv=P, groups=G, in_dtype="bf16")
    S = dev(S0)
    ref = S0.astype(np.float64)
    for t in range(20):
        tok = synth.mamba2_step_inputs(5, t, b, H, G, P, N, bias, "bf16")
        y = torch.empty((b, H, P), device="cuda")
        api.conventional_mamba2_step(dims, S, dev(A), dev(D), dev(tok["x"], torch.bfloat16),
                                     dev(tok["B"], torch.bfloat16), dev(tok["C"], torch.bfloat16),
                                     dev(tok["dt"]), y)
        ref, yr = rec.mamba2_step(ref, tok["x"], tok["B"], tok["C"], tok["dt"], A, D)
        f32_close(host(y), yr, f"conventional y step {t}")
    f32_close(host(S), ref, "conventional state")


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait that nothing completes ends after its limit with TIMEOUT set, and the
    same context then decodes normally."""
    import ctypes

    from recurrent_state_fp32_b300 import _abi

    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    rc = _abi.lib.replayssm_selftest_wait_timeout(ctypes.c_void_p(st.data_ptr()), None)
    assert rc == _abi.OK
    torch.cuda.synchronize()
    assert int(st[0]) == _abi.SEQ_TIMEOUT
    wl = synth.Mamba2Workload(batch=2, heads=4, P=64, N=128, window=4, steps=6, seed=12)
    run(Session("mamba2", wl, "f32"), wl.steps)
