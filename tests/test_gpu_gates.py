"""Gates at the edge of their range: a gate of exactly 0 (the layer forgets
its state at that entry) and gates so small that their product over a window
falls below the smallest FP32 normal. GDN (scalar gate) and KDA (per key
channel) through decode, consolidate, the fused fold + decode step and
speculative verify, against the float64 oracle (gated delta rule, "NVIDIA y
Princeton aceleran modelos híbridos…", paragraph 2: S_t = S_{t-1} A_t +
beta_t v_t k_t^T with A_t = Diag(alpha_t)(I - beta_t k_t k_t^T); alpha_t = 0
keeps only the new entry's beta v k^T)."""

import numpy as np
import pytest

import synth
from gpu_harness import Session

pytestmark = pytest.mark.gpu


def plant(alpha, t, kind, draft_axis=False):
    """Zero and tiny gates at fixed (step, sequence) positions; every other
    gate keeps its synthetic value."""
    a = np.array(alpha, copy=True)
    if draft_axis:  # [b, K, H(, d_k)]: draft i counts as step t + i
        for i in range(a.shape[1]):
            a[:, i] = plant(a[:, i], t + i, kind)
        return a
    if t % 3 == 0:
        a[0] = 0.0                         # sequence 0 forgets everything
    if t % 2 == 1:
        a[1] = 1e-20                       # two steps: 1e-40, below the FP32 normals
    if kind == "kda" and a.ndim == 3 and t % 4 == 2:
        a[2, :, : a.shape[2] // 4] = 0.0   # a quarter of sequence 2's channels forget
    return a.astype(np.float32)


class GateSession(Session):
    def token(self, t):
        tok = super().token(t)
        tok["alpha"] = plant(tok["alpha"], t, self.kind)
        return tok


@pytest.fixture
def planted_drafts(monkeypatch):
    real = synth.spec_draft_inputs

    def drafts(seed, r, batch, K, H, dk, dv, kind, in_dtype):
        d = real(seed, r, batch, K, H, dk, dv, kind, in_dtype)
        d["alpha"] = plant(d["alpha"], 2 * r, kind, draft_axis=True)
        return d

    monkeypatch.setattr(synth, "spec_draft_inputs", drafts)


@pytest.mark.parametrize("read", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_decode_and_fold(kind, read):
    wl = synth.DeltaWorkload(kind, batch=4, heads=3, dk=128, dv=128, window=6, steps=20,
                             in_dtype="bf16", seed=81)
    s = GateSession(kind, wl, read)
    for t in range(wl.steps):
        s.consolidate(1)
        s.decode(t)
    s.consolidate(1, force=True)
    s.check_pointers("end")
    s.check_checkpoint("after forced fold")


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_fused_step(kind):
    wl = synth.DeltaWorkload(kind, batch=4, heads=3, dk=128, dv=128, window=5, steps=17,
                             in_dtype="bf16", seed=82)
    s = GateSession(kind, wl, "bf16")
    for t in range(wl.steps):
        s.fold_decode(t)
    s.consolidate(1, force=True)
    s.check_checkpoint("after forced fold")


@pytest.mark.parametrize("tensor_cores", ["1", "0"])
@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_verify(kind, tensor_cores, planted_drafts, monkeypatch):
    monkeypatch.setenv("REPLAYSSM_DELTA_TENSOR_CORES", tensor_cores)
    wl = synth.DeltaWorkload(kind, batch=4, heads=3, dk=128, dv=128, window=12, K=4,
                             in_dtype="bf16", seed=83)
    s = GateSession(kind, wl, "bf16")
    for r in range(8):
        s.consolidate(4)
        s.verify(r, 4)
        s.accept(synth.accept_counts(wl.seed, r, wl.batch, 4), 4)
    s.consolidate(1, force=True)
    s.check_checkpoint("after forced fold")
