"""The tensor-core form of Gated DeltaNet speculative verify.

With a BF16 read copy and BF16 inputs, verify (K > 1) of a GDN layer with
windows up to 16 runs the tensor-core kernel: S [q | k]^T by mma.sync and the
sweep coefficients from a Gram tile. REPLAYSSM_DELTA_TENSOR_CORES=0 selects
the FFMA kernel. Both are held to the oracle's parity bar over rounds of
consolidate + verify + accept, on shapes that cover d_k 64 and 128, d_v of
one to three 64-row units, every draft count up to 8, short windows, and
batches that spread many heads over each block; and the two kernels agree on
the outputs of the same calls.
"""

import pytest
import torch

import synth
from gpu_harness import Session, bf16_close, host

pytestmark = pytest.mark.gpu

CASES = {
    "d128": dict(batch=6, heads=3, dk=128, dv=128, window=16, K=4, seed=41),
    "d64_dv192": dict(batch=5, heads=4, dk=64, dv=192, window=16, K=3, seed=42),
    "dv64_w5": dict(batch=7, heads=2, dk=128, dv=64, window=5, K=2, seed=43),
    "k8_w12": dict(batch=4, heads=3, dk=128, dv=128, window=12, K=8, seed=44),
    "many_heads": dict(batch=24, heads=32, dk=128, dv=128, window=16, K=4, seed=45),
}


def rounds(s, n, K):
    wl = s.wl
    for r in range(n):
        s.consolidate(K)
        s.verify(r, K)
        s.accept(synth.accept_counts(wl.seed, r, wl.batch, K), K)
        if r % 3 == 0:
            s.check_pointers(f"round {r}")
            s.check_ring(f"round {r}")
    s.consolidate(1, force=True)
    s.check_checkpoint("after forced fold")


@pytest.mark.parametrize("tensor_cores", ["1", "0"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_verify_matches_oracle(case, tensor_cores, monkeypatch):
    monkeypatch.setenv("REPLAYSSM_DELTA_TENSOR_CORES", tensor_cores)
    wl = synth.DeltaWorkload("gdn", in_dtype="bf16", **CASES[case])
    n = 12 if case != "many_heads" else 6
    rounds(Session("gdn", wl, "bf16", scale=0.85), n, wl.K)


def test_kernels_agree(monkeypatch):
    """Identical states, the same rounds through each kernel: outputs within
    the BF16 read-path bar of each other, ring bytes and pointers equal."""
    wl = synth.DeltaWorkload("gdn", batch=10, heads=8, dk=128, dv=128, window=16, K=4,
                             in_dtype="bf16", seed=46)
    a, b = Session("gdn", wl, "bf16"), Session("gdn", wl, "bf16")
    for r in range(10):
        m = synth.accept_counts(wl.seed, r, wl.batch, wl.K)
        outs = []
        for s, tc in ((a, "1"), (b, "0")):
            monkeypatch.setenv("REPLAYSSM_DELTA_TENSOR_CORES", tc)
            s.consolidate(wl.K)
            outs.append(s.verify(r, wl.K, check=False)[0])
            s.accept(m, wl.K)
        torch.cuda.synchronize()
        bf16_close(host(outs[0]), host(outs[1]), f"round {r}")
        for name in ("ring_head", "ring_len", "status"):
            assert torch.equal(getattr(a.state, name), getattr(b.state, name)), f"round {r}: {name}"
        for k in a.state.ring:
            assert torch.equal(a.state.ring[k], b.state.ring[k]), f"round {r}: ring {k}"
