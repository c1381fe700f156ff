"""The allocation-free Mamba-2 decode entry point against the ordinary one.

Some callers cannot allocate device memory when they decode: a plugin whose
host framework owns all device memory and allows no allocation while it
executes, or a serving loop that reserved the whole device for its state pool
up front. replayssm_mamba2_decode_noalloc serves them: it computes what
replayssm_mamba2_decode computes but takes its scratch (the per-head workspace
and the per-sequence arrival counters) from one fixed 16 MiB array inside the
library, so state.work and state.sync may be NULL.

The GPU tests call it through the C ABI twice in a row (the second call finds
the array as the first left it) and check each output, ring and pointer
against replayssm_mamba2_decode on an identical state, with the tolerance of
the other parity tests; and run decodes through it alone against the oracle.
The file's name makes pytest collect it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_harness import Session, f32_close, host
from recurrent_state_fp32_b300 import _abi, api

FAKE = 0x10000  # 16-byte aligned, never dereferenced


def _state(**over):
    f = {name: FAKE for name, _ in _abi.State._fields_}
    f.update(over)
    return _abi.State(**f)


def _noalloc(d, s, A=FAKE, y=FAKE):
    r = ctypes.byref
    return _abi.lib.replayssm_mamba2_decode_noalloc(
        r(d) if d is not None else None, r(s) if s is not None else None,
        A, FAKE, FAKE, FAKE, FAKE, FAKE, y, None)


# One sequence of P = 64 heads: each head takes a 68-float workspace row
# (P + 1 rounded up to 4); BOUNDARY_HEADS is the most the 16 MiB array holds.
BOUNDARY_HEADS = 61679


def _size(batch, heads, P=64, N=128, W=16):
    d = _abi.Dims(_abi.MAMBA2, batch, heads, 1, N, P, W, _abi.BF16)
    return _abi.lib.replayssm_mamba2_decode_noalloc_bytes(ctypes.byref(d))


def test_scratch_size_query():
    """The size query follows the documented formula and puts the refusal
    boundary where the call does."""
    def formula(b, H, P):
        rows = b * H * ((P + 1 + 3) // 4 * 4) * 4 + (4 * b + 15) // 16 * 16
        return (rows + 255) // 256 * 256 + 4 * b

    for b, H, P in ((1, 8, 64), (256, 128, 64), (5, 6, 96), (3, 1, 32), (1, BOUNDARY_HEADS, 64)):
        assert _size(b, H, P) == formula(b, H, P), (b, H, P)
    assert _size(256, 128) < 9 << 20
    assert _size(1, BOUNDARY_HEADS) <= _abi.NOALLOC_SCRATCH_BYTES < _size(1, BOUNDARY_HEADS + 1)
    r = ctypes.byref
    assert _abi.lib.replayssm_mamba2_decode_noalloc_bytes(None) == 0
    gdn = _abi.Dims(_abi.GDN, 2, 8, 1, 128, 64, 16, _abi.BF16)
    assert _abi.lib.replayssm_mamba2_decode_noalloc_bytes(r(gdn)) == 0
    bad = _abi.Dims(_abi.MAMBA2, 2, 8, 1, 96, 64, 16, _abi.BF16)
    assert _abi.lib.replayssm_mamba2_decode_noalloc_bytes(r(bad)) == 0


def test_arguments_and_the_size_limit():
    """Argument errors and the scratch limit are reported before any CUDA call."""
    no_scratch = dict(work=None, sync=None)
    big = _abi.Dims(_abi.MAMBA2, 4096, 128, 1, 128, 256, 16, _abi.BF16)
    assert _noalloc(big, _state(**no_scratch)) == _abi.ERR_SCRATCH_LIMIT
    assert b"16 MiB" in _abi.lib.replayssm_status_string(_abi.ERR_SCRATCH_LIMIT)
    over = _abi.Dims(_abi.MAMBA2, 1, BOUNDARY_HEADS + 1, 1, 128, 64, 16, _abi.BF16)
    assert _noalloc(over, _state(**no_scratch)) == _abi.ERR_SCRATCH_LIMIT
    empty = _abi.Dims(_abi.MAMBA2, 0, 8, 1, 128, 64, 16, _abi.BF16)
    assert _noalloc(empty, _state(**no_scratch)) == _abi.OK
    assert _noalloc(None, _state()) == _abi.ERR_INVALID_ARG
    assert _noalloc(empty, None) == _abi.ERR_INVALID_ARG
    gdn = _abi.Dims(_abi.GDN, 0, 8, 1, 128, 64, 16, _abi.BF16)
    assert _noalloc(gdn, _state()) == _abi.ERR_INVALID_ARG
    assert _noalloc(empty, _state(ring_len=None)) == _abi.ERR_INVALID_ARG
    assert _noalloc(empty, _state(S_read=FAKE + 8)) == _abi.ERR_MISALIGNED
    assert _noalloc(empty, _state(), A=None) == _abi.ERR_INVALID_ARG


CASES = {
    # ragged: P = 96, N = 64, 2 B/C groups, W = 5, FP32 inputs, FP32 read
    "ragged": dict(batch=5, heads=6, P=96, N=64, groups=2, window=5, in_dtype="f32",
                   read=False),
    # 64 sequences of the 128-head, P = 64, N = 128, W = 16 layer, BF16 read copy
    "layer": dict(batch=64, heads=128, P=64, N=128, groups=1, window=16, in_dtype="bf16",
                  read=True),
    # one sequence with as many heads as the fixed array holds (2 GB of state)
    "boundary": dict(batch=1, heads=BOUNDARY_HEADS, P=64, N=128, groups=1, window=3,
                     in_dtype="bf16", read=False),
}


def _compare(case):
    """Decodes a few buffered tokens through the ordinary entry point on two
    identical states, then makes two allocation-free calls in a row (the second
    finds the array as the first left it) and one on a full ring, each against
    replayssm_mamba2_decode on the twin state: outputs within the parity
    tolerance, ring bytes, pointers and status bit-exact."""
    c = CASES[case]
    b, H, P, N, G, W = (c[k] for k in ("batch", "heads", "P", "N", "groups", "window"))
    seed = 11
    dims = api.LayerDims("mamba2", b, H, dk=N, dv=P, window=W, groups=G, in_dtype=c["in_dtype"])
    assert api.mamba2_decode_noalloc_bytes(dims) <= _abi.NOALLOC_SCRATCH_BYTES
    vt = torch.float32 if c["in_dtype"] == "f32" else torch.bfloat16
    A, D, bias = synth.mamba2_params(seed, H)
    A, D = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    ref = api.LayerState(dims, read_copy=c["read"])
    new = api.LayerState(dims, read_copy=c["read"])
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    S0 = torch.empty_like(ref.S_ckpt).normal_(0.0, 0.1, generator=gen)
    for st in (ref, new):
        st.set_checkpoint(S0)
    del S0

    def token(t):
        tok = synth.mamba2_step_inputs(seed, t, b, H, G, P, N, bias, c["in_dtype"])
        return {k: torch.from_numpy(np.ascontiguousarray(tok[k])).cuda().to(
            torch.float32 if k == "dt" else vt) for k in ("x", "B", "C", "dt")}

    def args(tok, y):
        return [tok["x"].data_ptr(), tok["B"].data_ptr(), tok["C"].data_ptr(),
                tok["dt"].data_ptr(), y.data_ptr()]

    # a few buffered tokens first, so that the replay sums are not trivial
    for t in range(W - 2):
        tok = token(t)
        y = torch.empty((b, H, P), device="cuda")
        for st in (ref, new):
            api.mamba2_decode(dims, st, A, D, tok["x"], tok["B"], tok["C"], tok["dt"], y)

    # the caller's scratch is withheld from the allocation-free call
    c_new = _abi.State.from_buffer_copy(new.c())
    c_new.work = None
    c_new.sync = None
    for t in (W - 2, W - 1, W):  # two calls in a row, then one on a full ring
        tok = token(t)
        y_ref = torch.full((b, H, P), float("nan"), device="cuda")
        y_new = torch.full((b, H, P), float("nan"), device="cuda")
        _abi.check("replayssm_mamba2_decode", _abi.lib.replayssm_mamba2_decode(
            ctypes.byref(dims.c()), ctypes.byref(ref.c()), A.data_ptr(), D.data_ptr(),
            *args(tok, y_ref), None))
        _abi.check("replayssm_mamba2_decode_noalloc", _abi.lib.replayssm_mamba2_decode_noalloc(
            ctypes.byref(dims.c()), ctypes.byref(c_new), A.data_ptr(), D.data_ptr(),
            *args(tok, y_new), None))
        torch.cuda.synchronize()
        for name in ("ring_len", "ring_head", "status"):
            assert torch.equal(getattr(new, name), getattr(ref, name)), f"{case} token {t}: {name}"
        for k, v in ref.ring.items():
            assert torch.equal(new.ring[k], v), f"{case} token {t}: ring {k}"
        if t < W:
            f32_close(host(y_new), host(y_ref), f"{case} token {t}: y")
            assert int(ref.status.abs().sum()) == 0
            assert (host(ref.ring_len) == t + 1).all()
        else:  # refused: status bit set, output not written, state untouched
            assert torch.isnan(y_new).all() and torch.isnan(y_ref).all(), f"{case}: y written"
            assert (host(new.status) == _abi.SEQ_RING_FULL).all()
            assert (host(new.ring_len) == W).all()
    del ref, new
    torch.cuda.empty_cache()


@pytest.mark.gpu
def test_matches_the_allocating_entry_point():
    """The cases one after another in one process, so that each call finds the
    array holding the previous case's rows, of another layout: the small
    ragged layer, the 128-head layer, the small one again, then the largest
    size the array holds."""
    for case in ("ragged", "layer", "ragged", "boundary"):
        _compare(case)


@pytest.mark.gpu
@pytest.mark.parametrize("read", ["f32", "bf16"])
def test_against_the_oracle(read):
    """Decodes through the allocation-free entry point alone (the caller's
    scratch withheld), with consolidates between them, held to the oracle
    like every other decode: outputs within the parity tolerance, ring and
    pointers bit-exact, the checkpoint after a forced fold."""
    wl = synth.Mamba2Workload(batch=5, heads=6, P=64, N=128, window=8, steps=20,
                              in_dtype="bf16", seed=63)
    s = Session("mamba2", wl, read)
    for t in range(wl.steps):
        s.consolidate(1)
        tok = s.token(t)
        g = s._to_dev(tok)
        y = torch.full((wl.batch, wl.heads, wl.P), float("nan"), device="cuda")
        c = _abi.State.from_buffer_copy(s.state.c())
        c.work = None
        c.sync = None
        _abi.check("replayssm_mamba2_decode_noalloc", _abi.lib.replayssm_mamba2_decode_noalloc(
            ctypes.byref(s.dims.c()), ctypes.byref(c), s.dA.data_ptr(), s.dD.data_ptr(),
            g["x"].data_ptr(), g["B"].data_ptr(), g["C"].data_ptr(), g["dt"].data_ptr(),
            y.data_ptr(), None))
        ref = s.oracle.decode(s._sub(tok))
        torch.cuda.synchronize()
        s.compare_out(host(y)[s.seqs][:, s.heads], ref, f"token {t}")
        s.check_pointers(f"token {t}")
        s.check_ring(f"token {t}")
    s.consolidate(1, force=True)
    s.check_checkpoint("after forced fold")
