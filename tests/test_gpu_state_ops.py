"""Sequence state copies (prefix caching / continuous batching): a sequence
forked mid-stream into another slot continues exactly like its source."""

import numpy as np
import pytest
import torch

import synth
from gpu_harness import Session, dev, host

from recurrent_state_fp32_b300 import api

pytestmark = pytest.mark.gpu


def _fork_and_continue(s, steps_before, steps_after, src, dst):
    for t in range(steps_before):
        s.consolidate(1)
        s.decode(t, check=False)
    api.copy_sequences(s.dims, s.state, dev(np.array(src, np.int32), torch.int32), s.state,
                       dev(np.array(dst, np.int32), torch.int32))
    for t in range(steps_before, steps_before + steps_after):
        tok = s.token(t)
        # the forked sequences get their sources' tokens
        for k, v in tok.items():
            if s.kind == "mamba2" and k in ("B", "C"):
                v[dst] = v[src]
            else:
                v[dst] = v[src]
        g = s._to_dev(tok)
        api.consolidate(s.dims, s.state, s.dA if s.kind == "mamba2" else None, 1, False)
        rows = s.wl.P if s.kind == "mamba2" else s.wl.dv
        y = torch.full((s.wl.batch, s.wl.heads, rows), float("nan"), device="cuda")
        if s.kind == "mamba2":
            api.mamba2_decode(s.dims, s.state, s.dA, s.dD, g["x"], g["B"], g["C"], g["dt"], y)
        else:
            api.gdn_decode(s.dims, s.state, g["q"], g["k"], g["v"], g["alpha"], g["beta"], 1.0, y)
        yh = host(y)
        assert np.array_equal(yh[dst], yh[src]), f"step {t}: forked outputs differ"
    st = s.state
    for name in ("ring_head", "ring_len", "status"):
        a = host(getattr(st, name))
        assert np.array_equal(a[dst], a[src]), name
    for k, v in st.ring.items():
        a = host(v)
        assert np.array_equal(a[dst], a[src]), f"ring {k}"
    S = host(st.S_ckpt)
    assert np.array_equal(S[dst], S[src])


def test_mamba2_fork_mid_ring():
    wl = synth.Mamba2Workload(batch=6, heads=4, P=64, N=128, window=8, steps=20, seed=41)
    _fork_and_continue(Session("mamba2", wl, "bf16"), 11, 9, [0, 2], [4, 5])


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_delta_fork_mid_ring(kind):
    wl = synth.DeltaWorkload(kind, batch=5, heads=3, dk=128, dv=64, window=8, seed=42)
    _fork_and_continue(Session(kind, wl, "f32"), 13, 7, [1], [3])


JOIN_CASES = [("mamba2", "bf16"), ("mamba2", "f32"), ("gdn", "bf16"), ("kda", "f32")]


@pytest.mark.parametrize("kind,read", JOIN_CASES)
def test_staggered_joins(kind, read):
    """Continuous batching: new sequences take over slots at different steps,
    so the sequences sit at different ring phases and each consolidate folds a
    different subset of the batch. Every output, pointer, ring byte and the
    final checkpoint match the oracle."""
    if kind == "mamba2":
        wl = synth.Mamba2Workload(batch=6, heads=4, P=64, N=128, window=8, steps=30, seed=43)
    else:
        wl = synth.DeltaWorkload(kind, batch=6, heads=3, dk=128, dv=64, window=8, seed=44)
    s = Session(kind, wl, read)
    folded = set()
    for t in range(30):
        if t % 3 == 0:  # one slot changes hands every third step
            s.join([(t // 3) % wl.batch], seed=1000 + t)
        fold = s.consolidate(1)
        if fold.any() and not fold.all():
            folded.add(tuple(fold))
        s.decode(t)
        s.check_pointers(f"step {t}")
    assert len(set(host(s.state.ring_len).tolist())) > 2, "phases did not spread"
    assert folded, "no consolidate folded a strict subset of the batch"
    s.check_ring("end")
    s.consolidate(1, force=True)
    s.check_checkpoint("end")
