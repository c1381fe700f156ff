"""Speculative verify + accept (pointer rollback) on the delta kinds: CUDA path vs oracle."""

import numpy as np
import pytest

import synth
from gpu_harness import Session, spread

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
    """b512, H32, d_k = d_v = 128, K = 4, W = 16 (the speculative workload), its
    128 rounds; the oracle follows every head of 4 sequences spread over the
    batch."""
    wl = synth.DeltaWorkload("gdn", batch=512, heads=32, dk=128, dv=128, window=16, K=4,
                             in_dtype="bf16", seed=4)
    s = Session("gdn", wl, "bf16", seqs=spread(wl.batch, 4))
    run(s, 128, 4, check_every=17)


@pytest.mark.parametrize("kind,dk,dv,in_dtype", [("gdn", 128, 128, "bf16"), ("kda", 64, 96, "f32")])
def test_conventional_snapshot_verify_and_accept(kind, dk, dv, in_dtype):
    """The baseline spec path: per-draft snapshots and outputs against the oracle's
    conventional recurrence stepped through the drafts; accept restores snapshot m - 1."""
    import torch

    from gpu_harness import dev, f32_close, host
    from oracle import recurrences as rec
    from recurrent_state_fp32_b300 import api

    b, H, K, seed = 5, 3, 4, 23
    dims = api.LayerDims(kind, b, H, dk=dk, dv=dv, window=16, in_dtype=in_dtype)
    S0 = synth.delta_initial_state(seed, b, H, dv, dk)
    drafts = synth.spec_draft_inputs(seed, 0, b, K, H, dk, dv, kind, in_dtype)
    vt = torch.bfloat16 if in_dtype == "bf16" else torch.float32
    d = {n: dev(v, vt if n in ("q", "k", "v") else torch.float32) for n, v in drafts.items()}
    S = dev(S0)
    snaps = torch.empty((b, K, H, dv, dk), device="cuda")
    o = torch.empty((b, K, H, dv), device="cuda")
    api.conventional_gdn_verify(dims, S, K, d["q"], d["k"], d["v"], d["alpha"], d["beta"], 0.8,
                                snaps, o)
    torch.cuda.synchronize()
    assert np.array_equal(host(S), S0), "verify must not modify S"
    ref = np.asarray(S0, np.float64)
    for i in range(K):
        ref, o_ref = rec.delta_step(ref, drafts["q"][:, i], drafts["k"][:, i], drafts["v"][:, i],
                                    drafts["alpha"][:, i], drafts["beta"][:, i], scale=0.8)
        f32_close(host(o[:, i]), o_ref, f"draft {i} output")
        f32_close(host(snaps[:, i]), ref, f"draft {i} snapshot")
    m = np.array([0, 1, 2, 4, 3], np.int32)
    status = torch.zeros(b, dtype=torch.int32, device="cuda")
    api.conventional_accept(dims, S, snaps, dev(m, torch.int32), K, status)
    got, sn = host(S), host(snaps)
    for q in range(b):
        want = S0[q] if m[q] == 0 else sn[q, m[q] - 1]
        assert np.array_equal(got[q], want), f"sequence {q}: accept of {m[q]} drafts"
    assert int(status.abs().sum()) == 0
    before = host(S)
    api.conventional_accept(dims, S, snaps, dev(np.array([5, -1, 0, 4, 1], np.int32), torch.int32),
                            K, status)
    st = host(status).astype(np.int64)
    assert st[0] & 2 and st[1] & 2 and not st[2:].any()
    after = host(S)
    assert np.array_equal(after[:2], before[:2]), "a refused accept leaves S unchanged"
    assert np.array_equal(after[3], sn[3, 3]) and np.array_equal(after[4], sn[4, 0])


@pytest.mark.parametrize("read", ["f32", "bf16"])
def test_mamba2_spec(read):
    """Mamba-2 verify (K drafts from one state read) + pointer accept, with folds."""
    wl = synth.Mamba2Workload(batch=4, heads=8, P=64, N=128, window=16, K=4, in_dtype="bf16",
                              seed=31)
    run(Session("mamba2", wl, read), 20, 4)


def test_mamba2_spec_ragged():
    """P = 96, N = 64, two B/C groups, W = 7, K = 3, FP32 inputs and read path."""
    wl = synth.Mamba2Workload(batch=3, heads=6, P=96, N=64, groups=2, window=7, K=3,
                              in_dtype="f32", seed=32)
    run(Session("mamba2", wl, "f32"), 14, 3, check_every=1)


def test_mamba2_spec_then_plain_decode():
    wl = synth.Mamba2Workload(batch=3, heads=4, P=64, N=128, window=16, K=4, seed=33)
    s = Session("mamba2", wl, "bf16")
    for r in range(8):
        s.consolidate(4)
        s.verify(r, 4)
        s.accept(synth.accept_counts(wl.seed, r, wl.batch, 4), 4)
        s.consolidate(1)
        s.decode(r)
        s.check_pointers(f"round {r}")
        s.check_ring(f"round {r}")
    s.consolidate(1, force=True)
    s.check_checkpoint("end")
