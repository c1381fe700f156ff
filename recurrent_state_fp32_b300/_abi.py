"""ctypes view of the C ABI declared in include/replayssm.h (marshalling only).

Loads the in-tree ``libreplayssm.so`` on first use and raises ImportError if
it has not been built (there is no fallback implementation).
"""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libreplayssm.so")

# Return codes and per-sequence status bits (values fixed by the header).
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_CUDA = 0, 1, 2, 3, 4
ERR_SCRATCH_LIMIT = 5
NOALLOC_SCRATCH_BYTES = 16 << 20  # fixed scratch of replayssm_mamba2_decode_noalloc
SEQ_RING_FULL, SEQ_BAD_ACCEPT, SEQ_TIMEOUT, SEQ_BAD_POINTER = 1, 2, 4, 8
MAMBA2, GDN, KDA = 0, 1, 2
F32, BF16 = 0, 1


class Dims(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("groups", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("window", ctypes.c_int32), ("in_dtype", ctypes.c_int32)]


_P = ctypes.c_void_p


class State(ctypes.Structure):
    _fields_ = [("S_ckpt", _P), ("S_read", _P), ("ring_x", _P), ("ring_B", _P), ("ring_C", _P),
                ("ring_dt", _P), ("ring_q", _P), ("ring_k", _P), ("ring_v", _P),
                ("ring_alpha", _P), ("ring_beta", _P), ("ring_head", _P), ("ring_len", _P),
                ("status", _P), ("sync", _P), ("work", _P)]


class DeltaConfig(ctypes.Structure):
    _fields_ = [("tensor_cores", ctypes.c_int32), ("prep_warps", ctypes.c_int32),
                ("depth", ctypes.c_int32), ("state_stages", ctypes.c_int32),
                ("vector_slots", ctypes.c_int32), ("consumer_groups", ctypes.c_int32),
                ("consumer_warps_per_group", ctypes.c_int32), ("rows_per_unit", ctypes.c_int32),
                ("units_per_head", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int64)]


_DP = ctypes.POINTER(Dims)
_SP = ctypes.POINTER(State)
_I = ctypes.c_int32
_F = ctypes.c_float

# name -> argtypes (every entry point returns int32 except the two helpers)
SIGNATURES = {
    "replayssm_mamba2_decode": [_DP, _SP, _P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_mamba2_decode_noalloc": [_DP, _SP, _P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_mamba2_decode_noalloc_bytes": [_DP],
    "replayssm_gdn_decode": [_DP, _SP, _P, _P, _P, _P, _P, _F, _P, _P],
    "replayssm_gdn_fold_decode": [_DP, _SP, _P, _P, _P, _P, _P, _F, _P, _P],
    "replayssm_consolidate": [_DP, _SP, _P, _I, _I, _P],
    "replayssm_mamba2_fold_decode": [_DP, _SP, _P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_spec_verify": [_DP, _SP, _I, _P, _P, _P, _P, _P, _F, _P, _P],
    "replayssm_mamba2_spec_verify": [_DP, _SP, _I, _P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_accept": [_DP, _SP, _P, _I, _P],
    "replayssm_refresh_read_copy": [_DP, _SP, _P],
    "replayssm_conventional_mamba2_step": [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_conventional_gdn_step": [_DP, _P, _P, _P, _P, _P, _P, _F, _P, _P],
    "replayssm_conventional_gdn_verify": [_DP, _P, _I, _P, _P, _P, _P, _P, _F, _P, _P, _P],
    "replayssm_conventional_accept": [_DP, _P, _P, _P, _I, _P, _P],
    "replayssm_copy_sequences": [_DP, _SP, _P, _SP, _P, _I, _P],
    "replayssm_selftest_wait_timeout": [_P, _P],
    "replayssm_workspace_bytes": [_DP, _I],
    "replayssm_delta_kernel_config": [_DP, _I, _I, ctypes.c_int64, ctypes.POINTER(DeltaConfig)],
    "replayssm_status_string": [_I],
    "replayssm_version": [],
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"the ReplaySSM CUDA library is not built ({path} is missing); run "
            "`python -m recurrent_state_fp32_b300.build`")
    lib = ctypes.CDLL(path)
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = {"replayssm_status_string": ctypes.c_char_p,
                      "replayssm_workspace_bytes": ctypes.c_int64,
                      "replayssm_mamba2_decode_noalloc_bytes": ctypes.c_int64}.get(name, ctypes.c_int32)
    return lib


class _LazyLib:
    """Loads the library on first use, so that building it needs no prior build."""

    _lib = None

    def __getattr__(self, name):
        if _LazyLib._lib is None:
            _LazyLib._lib = load()
        return getattr(_LazyLib._lib, name)


lib = _LazyLib()


class ReplaySSMError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = lib.replayssm_status_string(code).decode()
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


def check(fn: str, code: int) -> None:
    if code != OK:
        raise ReplaySSMError(fn, code)
