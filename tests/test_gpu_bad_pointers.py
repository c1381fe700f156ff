"""Sequences whose ring pointers are out of range are refused on the GPU.

A head or length outside [0, W) / [0, W] can only come from a caller that
wrote the pointer arrays itself. Every kernel checks the pointers before it
uses them: such a sequence gets REPLAYSSM_SEQ_BAD_POINTER, no output and no
change to its state, and every other sequence of the call is computed exactly
as it is in an identical state without the bad sequence (bit for bit: the
same kernels on the same inputs).
"""

import numpy as np
import pytest
import torch

import synth
from gpu_harness import Session, host
from recurrent_state_fp32_b300 import _abi

pytestmark = pytest.mark.gpu

BAD = 2  # the sequence whose pointers are corrupted

CALLS = {
    "mamba2_decode": ("mamba2", 1),
    "mamba2_fold_decode": ("mamba2", 1),
    "mamba2_verify": ("mamba2", 3),
    "gdn_decode": ("gdn", 1),
    "kda_decode": ("kda", 1),
    "gdn_verify": ("gdn", 3),
    "gdn_fold_decode": ("gdn", 1),
    "kda_fold_decode": ("kda", 1),
}


def _session(kind, K):
    if kind == "mamba2":
        wl = synth.Mamba2Workload(batch=5, heads=4, P=64, N=128, window=8, steps=6, K=K,
                                  in_dtype="bf16", seed=61)
    else:
        wl = synth.DeltaWorkload(kind, batch=5, heads=3, dk=128, dv=64, window=8, K=K,
                                 in_dtype="bf16", seed=62)
    return Session(kind, wl, "bf16")


def _call(s, call, t):
    if call.endswith("fold_decode"):
        return s.fold_decode(t, check=False)[0]
    if call.endswith("verify"):
        s.consolidate(3)
        return s.verify(t, 3, check=False)[0]
    s.consolidate(1)
    return s.decode(t, check=False)[0]


@pytest.mark.parametrize("call", sorted(CALLS))
@pytest.mark.parametrize("field,value", [("ring_head", 11), ("ring_len", 9), ("ring_len", -1)])
def test_refused_and_untouched(call, field, value):
    kind, K = CALLS[call]
    a, b = _session(kind, K), _session(kind, K)
    for t in range(3):  # a few buffered entries first
        for s in (a, b):
            _call(s, call if not call.endswith("verify") else "plain", t)
    getattr(b.state, field)[BAD] = value
    before = {k: v[BAD].clone() for k, v in b.state.ring.items()}
    S_before = b.state.S_ckpt[BAD].clone()
    R_before = b.state.S_read[BAD].clone()
    ptr_before = (int(b.state.ring_head[BAD]), int(b.state.ring_len[BAD]))
    ya = _call(a, call, 3)
    yb = _call(b, call, 3)
    torch.cuda.synchronize()
    sa, sb = host(a.state.status).astype(np.int64), host(b.state.status).astype(np.int64)
    assert not sa.any(), "the clean state reports status bits"
    assert sb[BAD] & _abi.SEQ_BAD_POINTER, "the bad sequence is not flagged"
    assert not np.delete(sb, BAD).any(), "another sequence was flagged"
    assert torch.isnan(yb[BAD]).all(), "an output was written for the bad sequence"
    keep = [q for q in range(b.wl.batch) if q != BAD]
    assert torch.equal(yb[keep], ya[keep]), "the other sequences' outputs changed"
    assert (int(b.state.ring_head[BAD]), int(b.state.ring_len[BAD])) == ptr_before
    assert torch.equal(b.state.S_ckpt[BAD], S_before)
    assert torch.equal(b.state.S_read[BAD], R_before)
    for k, v in before.items():
        assert torch.equal(b.state.ring[k][BAD], v), f"ring {k} of the bad sequence changed"
    for name in ("ring_head", "ring_len"):
        g_a, g_b = getattr(a.state, name), getattr(b.state, name)
        assert torch.equal(g_b[keep], g_a[keep]), f"{name} of the other sequences differs"
    for k in a.state.ring:
        assert torch.equal(b.state.ring[k][keep], a.state.ring[k][keep]), f"ring {k} differs"
    assert int(b.state.sync.abs().sum()) == 0, "arrival counters not back at zero"
