"""The bench's algorithmic byte counts (the numerator of its roofline figure).

Checked against the per-token traffic the method must move, written out here
from the layer sizes, on a stand-in layer that needs no GPU. Per sequence and
token, averaged over a cycle of W = 16 steps in which the ring fills once:

- decode: the state read once (read copy, or the FP32 checkpoint without
  one); the token's inputs read and written to the ring; the n buffered
  entries read back (n = 0..15, mean 7.5); the output written;
- fold, once per cycle: the FP32 checkpoint read and written, the read copy
  written (when there is one) and the 16 ring entries read;
- the fused fold + decode step does not read the read copy of a sequence it
  folds (the output comes from the new rows).
"""

import numpy as np
import torch

import bench

B = 2  # sequences of the stand-in layer; every count below is per sequence


def layer(kind, read, fused=False):
    wl = dict(bench.WORKLOADS[kind])
    wl["batch"] = B
    L = object.__new__(bench.Layer)
    L.np, L.torch, L.wl, L.fused = np, torch, wl, fused and kind == "mamba2"
    H, dk, dv, G = wl["heads"], wl["dk"], wl["dv"], wl["groups"]

    class State:
        S_read = object() if read == "bf16" else None

    L.state = State()
    bf = lambda *s: torch.zeros((B,) + s, dtype=torch.bfloat16)  # noqa: E731
    f32 = lambda *s: torch.zeros((B,) + s, dtype=torch.float32)  # noqa: E731
    if kind == "mamba2":
        L.pool = [{"x": bf(H, dv), "B": bf(G, dk), "C": bf(G, dk), "dt": f32(H)}]
    else:
        gate = f32(H) if kind == "gdn" else f32(H, dk)
        L.pool = [{"q": bf(H, dk), "k": bf(H, dk), "v": bf(H, dv), "alpha": gate, "beta": f32(H)}]
    L.out = f32(H, dv)
    return L


def per_token(L, cycles=4):
    """Bytes per sequence and token over whole cycles: starting from full
    rings, every W-th step folds (the first one included)."""
    W = L.wl["window"]
    dec, fold = L.account(np.full(B, W, np.int64), W * cycles)
    return (dec + fold) / (B * W * cycles)


def test_mamba2_bytes_per_token():
    H, P, N = 128, 64, 128
    state = H * P * N                                   # 1,048,576 elements
    token = H * P * 2 + 2 * N * 2 + H * 4               # x, B, C (bf16), dt
    entry = H * P * 2 + N * 2 + H * 4                   # x, B, dt read back
    out = H * P * 4
    decode = lambda ts: state * ts + 2 * token + 7.5 * entry + out  # noqa: E731
    fold = lambda rd: (state * (4 + 4 + rd) + 16 * entry) / 16     # noqa: E731
    assert decode(2) + fold(2) == 2_965_888
    assert decode(4) + fold(0) == 4_931_968
    assert per_token(layer("mamba2", "bf16")) == 2_965_888
    assert per_token(layer("mamba2", "f32")) == 4_931_968
    # fused step: no read-copy read for the folded sequence (once per cycle)
    assert per_token(layer("mamba2", "bf16", fused=True)) == 2_965_888 - state * 2 / 16
    # conventional step: FP32 state read and written, token in, output out
    assert layer("mamba2", "bf16").conventional_bytes() / B == state * 8 + token + out == 8_438_784


def test_delta_bytes_per_token():
    H, d = 32, 128
    state = H * d * d
    for kind, gate in (("gdn", H * 4), ("kda", H * d * 4)):
        token = 3 * H * d * 2 + gate + H * 4            # q, k, v (bf16), alpha, beta
        entry = 2 * H * d * 2 + gate + H * 4            # k, v, alpha, beta read back
        out = H * d * 4
        want = state * 2 + 2 * token + 7.5 * entry + out + (state * 10 + 16 * entry) / 16
        assert per_token(layer(kind, "bf16")) == want
        # bytes per sequence and token of the b256 layers, BF16 read copy
        assert want == {"gdn": 1_583_744, "kda": 1_754_432}[kind]


def test_staggered_phases_move_the_same_bytes():
    """Sequences at ring phases s mod W move, per step, the cycle average."""
    L = layer("mamba2", "bf16")
    W = L.wl["window"]
    lock = L.account(np.full(B, W, np.int64), W)
    L2 = layer("mamba2", "bf16")
    L2.wl["batch"] = W
    L2.pool = [{k: torch.zeros((W,) + tuple(v.shape[1:]), dtype=v.dtype) for k, v in L.pool[0].items()}]
    L2.out = torch.zeros((W,) + tuple(L.out.shape[1:]))
    stag = L2.account(W - np.arange(W), W)
    assert np.isclose(sum(stag) / (W * W), sum(lock) / (B * W))


def test_fold_cycle_rate():
    """The steady state of one fold cycle: W - 1 plain calls and one folding
    call, each followed by the median gap, whatever share of folds the timed
    window held."""
    W, tokens = 16, 256
    dec_ms = [0.100, 0.102, 0.400, 0.098, 0.100, 0.101, 0.099, 0.100]
    folds = [False, False, True, False, False, False, False, False]
    gaps = [2.0, 3.0, 2.0, 2.5, 2.0, 4.0, 2.0]
    st = bench.call_stats(dec_ms, gaps, folds, W, tokens)
    assert st["plain_call_us_median"] == 100.0 and st["fold_call_us"] == 400.0
    assert st["fold_calls"] == 1 and st["host_gap_us_median"] == 2.0
    cycle = (15 * 100.0 + 400.0) / 16
    assert st["cycle_call_us"] == round(cycle, 2)
    assert st["cycle_tokens_per_s"] == round(tokens / ((cycle + 2.0) * 1e-6), 1)
    # every call folds (staggered phases) or none does: no cycle figure
    assert "cycle_call_us" not in bench.call_stats(dec_ms, gaps, [True] * 8, W, tokens)
    assert "cycle_call_us" not in bench.call_stats(dec_ms, gaps, [False] * 8, W, tokens)


def test_traffic_of_changed_kernels_is_not_reported_as_current():
    """A capture taken before its kernel changed is reported beside the
    roofline's traffic, never as it; unchanged captures scale with the batch."""
    for (kind, read, fused), why in bench.TRAFFIC_STALE.items():
        wl = dict(bench.WORKLOADS[kind])
        rec = bench.traffic_per_call(wl, read, fused)
        assert rec["traffic"] is None
        table = bench.TRAFFIC_B64_FUSED if fused else bench.TRAFFIC_B64
        assert rec["traffic_last_capture"]["bytes"] == round(table[(kind, read)] * wl["batch"] / 64)
        assert rec["traffic_last_capture"]["changed_since"] == why
    wl = dict(bench.WORKLOADS["mamba2"])
    cur = bench.traffic_per_call(wl, "bf16", False)
    assert set(cur) == {"traffic"} and cur["traffic"] == round(bench.TRAFFIC_B64[("mamba2", "bf16")] * wl["batch"] / 64)
    wl["batch"] = 128
    assert bench.traffic_per_call(wl, "bf16", False)["traffic"] == round(bench.TRAFFIC_B64[("mamba2", "bf16")] * 2)
    assert bench.traffic_per_call(dict(bench.WORKLOADS["kda"]), "bf16", False) == {"traffic": None}
