"""Sequence state copies (prefix caching / continuous batching): a sequence
forked mid-stream into another slot resumes from the copied checkpoint, ring
and pointers; the oracle forks the same way and both sides must agree."""

import pytest

import synth
from gpu_harness import Session, host

pytestmark = pytest.mark.gpu


def _fork_and_continue(s, steps_before, steps_after, src, dst):
    """Decode, fork src into dst mid-ring (dst at another ring phase: it
    restarted earlier), and decode on; the oracle forks too, and every
    output, pointer, ring byte and the final checkpoint match it, for the
    sources and the copies alike."""
    for t in range(steps_before):
        if t == 2:
            s.join(dst, seed=700)  # the destination slots take a new sequence
        s.consolidate(1, force=(t == 4))  # a partial fold moves the ring head
        s.decode(t)
    h, ln = host(s.state.ring_head), host(s.state.ring_len)
    assert all(ln[q] > 0 for q in src), "fork taken mid-ring"
    assert any((h[a], ln[a]) != (h[b], ln[b]) for a, b in zip(src, dst)), "phases differ"
    s.check_pointers("before the fork")
    s.fork(src, dst)
    s.check_pointers("after the fork")
    s.check_ring("after the fork")
    for t in range(steps_before, steps_before + steps_after):
        s.consolidate(1)
        s.decode(t)
        s.check_pointers(f"step {t}")
        s.check_ring(f"step {t}")
    s.consolidate(1, force=True)
    s.check_checkpoint("end")


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
