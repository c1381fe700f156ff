"""Gated DeltaNet / KDA replay decode, consolidate and conventional step: CUDA path vs oracle."""

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


@pytest.mark.parametrize("kind", ["gdn", "kda"])
@pytest.mark.parametrize("read", ["f32", "bf16"])
def test_small_layer(kind, read):
    """b3, H4, d_k = d_v = 128, W16, 40 steps, BF16 vector inputs."""
    wl = synth.DeltaWorkload(kind, batch=3, heads=4, dk=128, dv=128, window=16, steps=40,
                             in_dtype="bf16", seed=3)
    run(Session(kind, wl, read, scale=0.75), wl.steps)


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_ragged_and_fp32_inputs(kind):
    """d_k = 64, d_v = 96 (3 row passes), W = 7, FP32 inputs."""
    wl = synth.DeltaWorkload(kind, batch=5, heads=3, dk=64, dv=96, window=7, steps=25,
                             in_dtype="f32", seed=12)
    run(Session(kind, wl, "f32"), wl.steps, check_every=4)


@pytest.mark.parametrize("batch", [1, 8])
def test_small_batch_row_split(batch):
    """Small batches split each head into row blocks to fill the SMs."""
    wl = synth.DeltaWorkload("kda", batch=batch, heads=2, dk=128, dv=128, window=16, steps=20,
                             in_dtype="bf16", seed=13)
    run(Session("kda", wl, "bf16"), wl.steps, check_every=5)


def test_fold_row_chunks():
    """d_v = 160 at d_k = 128: each folding head is two row chunks (128 + 32
    rows) of the prefetching consolidate, each unit re-staging the ring."""
    wl = synth.DeltaWorkload("gdn", batch=3, heads=3, dk=128, dv=160, window=16, steps=36,
                             in_dtype="bf16", seed=16)
    run(Session("gdn", wl, "bf16"), wl.steps, check_every=7)


@pytest.mark.parametrize("kind,window,in_dtype,steps", [
    ("gdn", 20, "bf16", 44),   # a longer ring, still prefetched
    ("kda", 16, "f32", 36),    # staging too large for two blocks per SM: synchronous fold
    ("kda", 40, "f32", 84),    # synchronous fold, longer ring
])
def test_fold_forms(kind, window, in_dtype, steps):
    """Consolidate shapes on both sides of the prefetching fold's shared-memory limit."""
    wl = synth.DeltaWorkload(kind, batch=3, heads=2, dk=128, dv=128, window=window,
                             steps=steps, in_dtype=in_dtype, seed=17)
    run(Session(kind, wl, "bf16"), wl.steps, check_every=11)


def test_window_one_and_no_optional_fields():
    wl = synth.DeltaWorkload("gdn", batch=2, heads=3, dk=128, dv=64, window=1, steps=8, seed=14)
    run(Session("gdn", wl, "f32", store_optional=False), wl.steps, check_every=1)


def test_full_ring_is_refused():
    wl = synth.DeltaWorkload("gdn", batch=2, heads=2, dk=128, dv=128, window=3, seed=15)
    s = Session("gdn", wl, "bf16")
    for t in range(3):
        s.decode(t)
    y, _ = s.decode(3)
    assert torch.isnan(y).all()
    s.check_pointers()
    s.check_ring()


@pytest.mark.parametrize("read", ["bf16", "f32"])
@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_full_size_sampled(kind, read):
    """b256, H32, d_k = d_v = 128, W16, 256 steps, BF16 inputs, BF16 read copy
    or FP32 read path. The oracle follows every head of 8 sequences spread
    over the batch; at three steps every (sequence, head) output is also
    checked against the replay formula on the GPU's own checkpoint copy and
    ring."""
    wl = synth.DeltaWorkload(kind, batch=256, heads=32, dk=128, dv=128, window=16, steps=256,
                             in_dtype="bf16", seed=3 if kind == "gdn" else 5)
    s = Session(kind, wl, read, seqs=spread(wl.batch))
    run(s, wl.steps, check_every=41, all_units_at=(6, 130, 249))


@pytest.mark.parametrize("batch", [1, 8, 64, 512])
def test_kda_batch_sweep_sizes(batch):
    """The KDA layer at the other batch sizes of the batch sweep (1, 8, 64,
    512; 256 is above), 256 steps, BF16 read copy; every head of up to 8
    sequences against the oracle, every unit at two steps."""
    wl = synth.DeltaWorkload("kda", batch=batch, heads=32, dk=128, dv=128, window=16, steps=256,
                             in_dtype="bf16", seed=5)
    s = Session("kda", wl, "bf16", seqs=spread(batch, min(8, batch)))
    run(s, wl.steps, check_every=53, all_units_at=(11, 200))


@pytest.mark.parametrize("kind", ["gdn", "kda"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 96)])
def test_conventional_step(kind, dk, dv):
    b, H = 3, 4
    S0 = synth.delta_initial_state(6, b, H, dv, dk)
    dims = api.LayerDims(kind, b, H, dk=dk, dv=dv, in_dtype="bf16")
    S = dev(S0)
    ref = S0.astype(np.float64)
    for t in range(20):
        tok = synth.delta_step_inputs(6, t, b, H, dk, dv, kind, "bf16")
        o = torch.empty((b, H, dv), device="cuda")
        api.conventional_gdn_step(dims, S, dev(tok["q"], torch.bfloat16),
                                  dev(tok["k"], torch.bfloat16), dev(tok["v"], torch.bfloat16),
                                  dev(tok["alpha"]), dev(tok["beta"]), 0.5, o)
        ref, orf = rec.delta_step(ref, tok["q"], tok["k"], tok["v"], tok["alpha"], tok["beta"], 0.5)
        f32_close(host(o), orf, f"conventional o step {t}")
    f32_close(host(S), ref, "conventional state")
