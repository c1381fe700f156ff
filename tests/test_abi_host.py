"""The C-ABI library on the host: it loads, exports every declared entry point,
and rejects bad arguments before any CUDA call (no GPU needed).

Every call here either fails validation or has batch == 0, so nothing is ever
launched; fake device addresses are never dereferenced.
"""

import ctypes
import os
import re

import pytest

from recurrent_state_fp32_b300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "replayssm.h")

FAKE = 0x10000  # 16-byte aligned, never dereferenced
MISALIGNED = 0x10008


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"REPLAYSSM_API\s+[\w\s\*]+?\b(replayssm_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("replayssm_mamba2_decode", "replayssm_gdn_decode", "replayssm_consolidate",
              "replayssm_spec_verify", "replayssm_accept"):
        assert n in names
    assert set(names) == set(_abi.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(_abi.LIB_PATH)
    for n in declared_symbols():
        assert hasattr(lib, n), n


def test_version_and_strings():
    assert _abi.lib.replayssm_version() == 100
    for code in range(5):
        assert _abi.lib.replayssm_status_string(code)
    assert b"unknown" in _abi.lib.replayssm_status_string(99)


def dims(kind=_abi.MAMBA2, batch=2, heads=4, groups=1, dk=128, dv=64, window=16,
         in_dtype=_abi.BF16):
    return _abi.Dims(kind, batch, heads, groups, dk, dv, window, in_dtype)


def state(**over):
    f = {name: FAKE for name, _ in _abi.State._fields_}
    f.update(over)
    return _abi.State(**f)


def m2_decode(d, s, y=FAKE, A=FAKE):
    r = ctypes.byref
    return _abi.lib.replayssm_mamba2_decode(r(d) if d is not None else None,
                                            r(s) if s is not None else None,
                                            A, FAKE, FAKE, FAKE, FAKE, FAKE, y, None)


def test_null_and_bad_dims():
    assert m2_decode(None, state()) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(), None) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(kind=7), state()) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(kind=_abi.GDN), state()) == _abi.ERR_INVALID_ARG  # wrong entry point
    assert m2_decode(dims(batch=-1), state()) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(heads=0), state()) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(groups=3), state()) == _abi.ERR_INVALID_ARG   # 3 does not divide 4
    assert m2_decode(dims(in_dtype=5), state()) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(window=0), state()) == _abi.ERR_INVALID_ARG


def test_unsupported_sizes():
    assert m2_decode(dims(dk=96), state()) == _abi.ERR_UNSUPPORTED
    assert m2_decode(dims(dv=48), state()) == _abi.ERR_UNSUPPORTED
    assert m2_decode(dims(dv=288), state()) == _abi.ERR_UNSUPPORTED
    assert m2_decode(dims(window=65), state()) == _abi.ERR_UNSUPPORTED


def test_null_and_misaligned_pointers():
    assert m2_decode(dims(), state(S_ckpt=None)) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(), state(ring_len=None)) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(), state(sync=None)) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(), state(), y=None) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(), state(), A=None) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(), state(S_read=MISALIGNED)) == _abi.ERR_MISALIGNED
    assert m2_decode(dims(), state(ring_x=MISALIGNED)) == _abi.ERR_MISALIGNED
    assert m2_decode(dims(), state(), y=MISALIGNED) == _abi.ERR_MISALIGNED


def test_empty_batch_is_a_noop():
    assert m2_decode(dims(batch=0), state()) == _abi.OK
    r = ctypes.byref
    d = dims(kind=_abi.GDN, batch=0, dv=128)
    assert _abi.lib.replayssm_gdn_decode(r(d), r(state()), FAKE, FAKE, FAKE, FAKE, FAKE,
                                         1.0, FAKE, None) == _abi.OK
    assert _abi.lib.replayssm_consolidate(r(d), r(state()), None, 1, 0, None) == _abi.OK
    assert _abi.lib.replayssm_spec_verify(r(d), r(state()), 4, FAKE, FAKE, FAKE, FAKE, FAKE,
                                          1.0, FAKE, None) == _abi.OK
    assert _abi.lib.replayssm_accept(r(d), r(state()), FAKE, 4, None) == _abi.OK


def test_call_specific_checks():
    r = ctypes.byref
    g = dims(kind=_abi.GDN, dv=128)
    m = dims()
    # consolidate: k_next in [0, W], force in {0, 1}, A required for Mamba-2
    assert _abi.lib.replayssm_consolidate(r(g), r(state()), None, 17, 0, None) == _abi.ERR_INVALID_ARG
    assert _abi.lib.replayssm_consolidate(r(g), r(state()), None, -1, 0, None) == _abi.ERR_INVALID_ARG
    assert _abi.lib.replayssm_consolidate(r(g), r(state()), None, 1, 2, None) == _abi.ERR_INVALID_ARG
    assert _abi.lib.replayssm_consolidate(r(m), r(state()), None, 1, 0, None) == _abi.ERR_INVALID_ARG
    # verify: K in [1, 8] and K <= W; Mamba-2 not built
    sv = _abi.lib.replayssm_spec_verify
    assert sv(r(g), r(state()), 0, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, None) == _abi.ERR_INVALID_ARG
    assert sv(r(g), r(state()), 9, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, None) == _abi.ERR_INVALID_ARG
    g4 = dims(kind=_abi.GDN, dv=128, window=3)
    assert sv(r(g4), r(state()), 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, None) == _abi.ERR_INVALID_ARG
    assert sv(r(m), r(state()), 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, None) == _abi.ERR_UNSUPPORTED
    # accept: K >= 0, m required
    assert _abi.lib.replayssm_accept(r(g), r(state()), FAKE, -1, None) == _abi.ERR_INVALID_ARG
    assert _abi.lib.replayssm_accept(r(g), r(state()), None, 4, None) == _abi.ERR_INVALID_ARG
    # refresh needs a read copy
    assert _abi.lib.replayssm_refresh_read_copy(r(g), r(state(S_read=None)), None) == _abi.ERR_INVALID_ARG
    # conventional steps check their kind
    assert _abi.lib.replayssm_conventional_mamba2_step(r(g), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                                       FAKE, FAKE, None) == _abi.ERR_INVALID_ARG
    assert _abi.lib.replayssm_conventional_gdn_step(r(m), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0,
                                                    FAKE, None) == _abi.ERR_INVALID_ARG


@pytest.mark.parametrize("missing", ["ring_k", "ring_v", "ring_alpha", "ring_beta"])
def test_delta_state_requires_its_ring(missing):
    r = ctypes.byref
    g = dims(kind=_abi.KDA, dv=128)
    st = state(**{missing: None})
    assert _abi.lib.replayssm_gdn_decode(r(g), r(st), FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE,
                                         None) == _abi.ERR_INVALID_ARG


def test_fold_decode_arguments():
    """The fused fold + decode entry point validates like the plain decode."""
    r = ctypes.byref

    def call(d, s, A=FAKE, y=FAKE):
        return _abi.lib.replayssm_mamba2_fold_decode(
            r(d) if d is not None else None, r(s) if s is not None else None,
            A, FAKE, FAKE, FAKE, FAKE, FAKE, y, None)

    assert call(None, state()) == _abi.ERR_INVALID_ARG
    assert call(dims(), None) == _abi.ERR_INVALID_ARG
    assert call(dims(kind=_abi.GDN), state()) == _abi.ERR_INVALID_ARG
    assert call(dims(), state(), A=None) == _abi.ERR_INVALID_ARG
    assert call(dims(), state(), y=None) == _abi.ERR_INVALID_ARG
    assert call(dims(), state(ring_len=None)) == _abi.ERR_INVALID_ARG
    assert call(dims(), state(S_ckpt=FAKE + 4)) == _abi.ERR_MISALIGNED
    assert call(dims(dk=96), state()) == _abi.ERR_UNSUPPORTED
    assert call(dims(batch=0), state()) == _abi.OK


def test_workspace_size():
    r = ctypes.byref
    # Mamba-2: the fused fold + decode step's rows (16 decode weights, the
    # token's weight, two decays, padding, 16 fold weights: 36 floats) and 16
    # B rows per (sequence, group); verify rows for K = 4
    m = dims(batch=2, heads=4, dk=128, dv=64)
    step = 2 * 4 * 36 * 4 + 2 * 16 * 128 * 4
    assert _abi.lib.replayssm_workspace_bytes(r(m), 1) == step
    assert _abi.lib.replayssm_workspace_bytes(r(m), 4) == max(4 * 2 * 4 * 68 * 4 + 16, step)
    g = dims(kind=_abi.GDN, batch=3, heads=2, dk=128, dv=96)
    assert _abi.lib.replayssm_workspace_bytes(r(g), 1) == 3 * 2 * 224 * 4 + 16
    assert _abi.lib.replayssm_workspace_bytes(r(g), 4) == 3 * 4 * 2 * 224 * 4 + 16
    assert _abi.lib.replayssm_workspace_bytes(r(dims(dk=96)), 1) == 0
    assert _abi.lib.replayssm_workspace_bytes(None, 1) == 0
    assert m2_decode(dims(), state(work=None)) == _abi.ERR_INVALID_ARG
    assert m2_decode(dims(), state(work=MISALIGNED)) == _abi.ERR_MISALIGNED


def test_conventional_spec_arguments():
    r = ctypes.byref
    g = dims(kind=_abi.GDN, dv=128)
    cv = _abi.lib.replayssm_conventional_gdn_verify
    assert cv(r(g), FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, FAKE, None) == _abi.ERR_INVALID_ARG
    assert cv(r(g), FAKE, 9, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, FAKE, None) == _abi.ERR_INVALID_ARG
    assert cv(r(dims()), FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, FAKE, None) == _abi.ERR_INVALID_ARG
    assert cv(r(g), FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, None, FAKE, None) == _abi.ERR_INVALID_ARG
    assert cv(r(g), MISALIGNED, 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, FAKE, None) == _abi.ERR_MISALIGNED
    g0 = dims(kind=_abi.GDN, batch=0, dv=128)
    assert cv(r(g0), FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, FAKE, None) == _abi.OK
    ca = _abi.lib.replayssm_conventional_accept
    assert ca(r(g), FAKE, FAKE, None, 4, None, None) == _abi.ERR_INVALID_ARG
    assert ca(r(g), FAKE, FAKE, FAKE, 0, None, None) == _abi.ERR_INVALID_ARG
    assert ca(r(g), FAKE, FAKE, FAKE, 4, MISALIGNED, None) == _abi.ERR_MISALIGNED
    assert ca(r(g0), FAKE, FAKE, FAKE, 4, None, None) == _abi.OK


def test_mamba2_spec_arguments():
    r = ctypes.byref
    mv = _abi.lib.replayssm_mamba2_spec_verify
    m = dims()
    assert mv(r(dims(kind=_abi.GDN, dv=128)), r(state()), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
              None) == _abi.ERR_INVALID_ARG
    assert mv(r(m), r(state()), 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == _abi.ERR_INVALID_ARG
    assert mv(r(m), r(state()), 9, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == _abi.ERR_INVALID_ARG
    assert mv(r(dims(window=3)), r(state()), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
              None) == _abi.ERR_INVALID_ARG
    assert mv(r(m), r(state()), 4, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == _abi.ERR_INVALID_ARG
    assert mv(r(m), r(state()), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, MISALIGNED,
              None) == _abi.ERR_MISALIGNED
    assert mv(r(dims(batch=0)), r(state()), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
              None) == _abi.OK


def test_selftest_arguments():
    assert _abi.lib.replayssm_selftest_wait_timeout(None, None) == _abi.ERR_INVALID_ARG
    assert _abi.lib.replayssm_selftest_wait_timeout(MISALIGNED, None) == _abi.ERR_MISALIGNED


def test_copy_sequences_arguments():
    r = ctypes.byref
    cs = _abi.lib.replayssm_copy_sequences
    g = dims(kind=_abi.GDN, dv=128)
    assert cs(r(g), r(state()), FAKE, r(state()), FAKE, -1, None) == _abi.ERR_INVALID_ARG
    assert cs(r(g), r(state()), FAKE, r(state()), FAKE, 0, None) == _abi.OK
    assert cs(r(g), r(state()), None, r(state()), FAKE, 2, None) == _abi.ERR_INVALID_ARG
    assert cs(r(g), r(state(S_read=None)), FAKE, r(state()), FAKE, 2, None) == _abi.ERR_INVALID_ARG
    assert cs(r(g), r(state()), FAKE, r(state(ring_k=None)), FAKE, 2, None) == _abi.ERR_INVALID_ARG


def test_binding_refuses_bad_index_tensors():
    """The Python binding checks count and index tensors (int32, one per
    sequence, equal lengths) before it builds any call."""
    import torch

    from recurrent_state_fp32_b300 import api

    dims = api.LayerDims("gdn", 3, 2, dk=128, dv=128)
    with pytest.raises(TypeError):
        api.accept(dims, None, torch.zeros(3, dtype=torch.int64), 4)
    with pytest.raises(ValueError):
        api.accept(dims, None, torch.zeros(2, dtype=torch.int32), 4)
    with pytest.raises(TypeError):
        api.conventional_accept(dims, None, None, [0, 1, 2], 4)
    with pytest.raises(ValueError):
        api.copy_sequences(dims, None, torch.zeros(2, dtype=torch.int32), None,
                           torch.zeros(3, dtype=torch.int32))
