"""Speculative verify + accept (pointer rollback) on the delta kinds: CUDA path vs oracle."""

import numpy as np
import pytest

import synth
from gpu_harness import Session

pytestmark = pytest.mark.gpu


def run(s, rounds, K, check_every=4):
    wl = s.wl
    for r in range(rounds):
        s.consolidate(K)
        s.verify(r, K)
        m = synth.accept_counts(wl.seed, r, wl.batch, K)
        s.accept(m, K)
        if r % check_every == 0:
            s.check_pointers(f"round {r}")
            s.check_ring(f"round {r}")
    s.check_pointers("end")
    s.check_ring("end")
    s.consolidate(1, force=True)
    s.check_pointers("after forced fold")
    s.check_checkpoint("after forced fold")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
@pytest.mark.parametrize("read", ["f32", "bf16"])
def test_small_spec(kind, read):
    wl = synth.DeltaWorkload(kind, batch=6, heads=3, dk=128, dv=128, window=16, K=4,
                             in_dtype="bf16", seed=4)
    run(Session(kind, wl, read, scale=0.9), 30, 4)


@pytest.mark.parametrize("K", [1, 3, 8])
def test_draft_counts(K):
    wl = synth.DeltaWorkload("gdn", batch=4, heads=2, dk=64, dv=64, window=9, K=K,
                             in_dtype="f32", seed=16)
    run(Session("gdn", wl, "f32"), 12, K, check_every=1)


def test_spec_then_plain_decode():
    """Rounds of verify/accept interleaved with plain decode steps on one state."""
    wl = synth.DeltaWorkload("kda", batch=3, heads=2, dk=128, dv=128, window=16, K=4, seed=17)
    s = Session("kda", wl, "bf16")
    for r in range(10):
        s.consolidate(4)
        s.verify(r, 4)
        s.accept(synth.accept_counts(wl.seed, r, wl.batch, 4), 4)
        s.consolidate(1)
        s.decode(r)
        s.check_pointers(f"round {r}")
        s.check_ring(f"round {r}")


def test_bad_accept_and_full_ring():
    wl = synth.DeltaWorkload("gdn", batch=3, heads=2, dk=128, dv=128, window=6, K=4, seed=18)
    s = Session("gdn", wl, "bf16")
    s.verify(0, 4)
    s.accept(np.array([5, -1, 4], np.int32), 4)     # two bad counts, one good
    s.check_pointers()
    s.verify(1, 4)                                  # len 4 for seq 2: 4 + 4 > 6, refused
    s.check_pointers()
    s.check_ring()


def test_full_size_sampled():
    """b512, H32, d_k = d_v = 128, K = 4, W = 16 (the speculative workload), 24 rounds."""
    wl = synth.DeltaWorkload("gdn", batch=512, heads=32, dk=128, dv=128, window=16, K=4,
                             in_dtype="bf16", seed=4)
    s = Session("gdn", wl, "bf16", seqs=[0, 311, 511], heads=[0, 16, 31])
    run(s, 24, 4, check_every=7)
