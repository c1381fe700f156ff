"""Python binding of the ReplaySSM C ABI (same names, argument marshalling only).

Every function takes torch CUDA tensors, passes their device pointers and the
current CUDA stream to the library, and raises ReplaySSMError on a non-OK
return code. All arithmetic happens in the CUDA kernels; torch only provides
device memory and streams. ``LayerState`` allocates the caller-owned state
buffers with the layouts the header documents.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _abi
from ._abi import ReplaySSMError  # noqa: F401

_KINDS = {"mamba2": _abi.MAMBA2, "gdn": _abi.GDN, "kda": _abi.KDA}
_DTYPES = {"f32": _abi.F32, "bf16": _abi.BF16}
_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class LayerDims:
    """Sizes of one SSM layer (``dk`` = N or d_k, ``dv`` = P or d_v)."""

    kind: str
    batch: int
    heads: int
    dk: int
    dv: int
    window: int = 16
    groups: int = 1
    in_dtype: str = "bf16"

    def c(self) -> _abi.Dims:
        c = self.__dict__.get("_c")
        if c is None:
            c = _abi.Dims(_KINDS[self.kind], self.batch, self.heads, self.groups, self.dk,
                          self.dv, self.window, _DTYPES[self.in_dtype])
            object.__setattr__(self, "_c", c)  # frozen dataclass: cache the C struct once
        return c

    @property
    def vec_dtype(self) -> torch.dtype:
        return _TORCH[self.in_dtype]


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _int32(t, name: str):
    """Index and count tensors are int32 [n] on the device; anything else
    would be misread by the kernels, so it is refused here."""
    if not isinstance(t, torch.Tensor) or t.dtype != torch.int32:
        raise TypeError(f"{name} must be an int32 tensor")
    return t


def ring_wd(W: int) -> int:
    """Entries per (sequence, head) of a scalar ring field: W rounded up to 4."""
    return (W + 3) & ~3


class LayerState:
    """Caller-owned device buffers of one layer's decode state.

    S_ckpt f32 [b,H,dv,dk]; S_read bf16 (optional); per-head ring fields
    [b,H,W,...] (scalar ones [b,H,Wd]); Mamba-2 B/C [b,W,G,N]; ring_head,
    ring_len, status, sync int32 [b], zero-initialised.
    """

    def __init__(self, dims: LayerDims, device="cuda", read_copy: bool = True,
                 store_optional: bool = True, max_drafts: int = 1):
        d = dims
        b, W, H = d.batch, d.window, d.heads
        z = dict(device=device)
        self.dims = d
        self.S_ckpt = torch.zeros((b, H, d.dv, d.dk), dtype=torch.float32, **z)
        self.S_read = torch.zeros_like(self.S_ckpt, dtype=torch.bfloat16) if read_copy else None
        vt = d.vec_dtype
        Wd = ring_wd(W)
        self.ring = {}
        if d.kind == "mamba2":
            self.ring["x"] = torch.zeros((b, H, W, d.dv), dtype=vt, **z)
            self.ring["B"] = torch.zeros((b, W, d.groups, d.dk), dtype=vt, **z)
            if store_optional:
                self.ring["C"] = torch.zeros((b, W, d.groups, d.dk), dtype=vt, **z)
            self.ring["dt"] = torch.zeros((b, H, Wd), dtype=torch.float32, **z)
        else:
            if store_optional:
                self.ring["q"] = torch.zeros((b, H, W, d.dk), dtype=vt, **z)
            self.ring["k"] = torch.zeros((b, H, W, d.dk), dtype=vt, **z)
            self.ring["v"] = torch.zeros((b, H, W, d.dv), dtype=vt, **z)
            ashape = (b, H, Wd) if d.kind == "gdn" else (b, H, W, d.dk)
            self.ring["alpha"] = torch.zeros(ashape, dtype=torch.float32, **z)
            self.ring["beta"] = torch.zeros((b, H, Wd), dtype=torch.float32, **z)
        self.ring_head = torch.zeros(b, dtype=torch.int32, **z)
        self.ring_len = torch.zeros(b, dtype=torch.int32, **z)
        self.status = torch.zeros(b, dtype=torch.int32, **z)
        self.sync = torch.zeros(b, dtype=torch.int32, **z)
        nbytes = workspace_bytes(d, max_drafts)
        self.work = torch.empty((nbytes + 3) // 4, dtype=torch.float32, **z)
        self._c = None

    def c(self) -> _abi.State:
        """The C struct of device pointers (built once; the buffers never move)."""
        if self._c is not None:
            return self._c
        r = self.ring
        g = lambda k: _ptr(r.get(k))  # noqa: E731
        self._c = _abi.State(_ptr(self.S_ckpt), _ptr(self.S_read), g("x"), g("B"), g("C"),
                             g("dt"), g("q"), g("k"), g("v"), g("alpha"), g("beta"),
                             _ptr(self.ring_head), _ptr(self.ring_len), _ptr(self.status),
                             _ptr(self.sync), _ptr(self.work))
        return self._c

    def set_checkpoint(self, S: torch.Tensor, stream=None) -> None:
        """Copies S into the FP32 checkpoint and refreshes the read copy, both on
        `stream` (default: the current stream), so the refresh sees the copy."""
        if stream is None:
            self.S_ckpt.copy_(S)
        else:
            s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(int(stream))
            with torch.cuda.stream(s):
                self.S_ckpt.copy_(S)
        if self.S_read is not None:
            refresh_read_copy(self.dims, self, stream)


def _call(name, *args):
    _abi.check(name, getattr(_abi.lib, name)(*args))


def _refs(dims, state):
    return ctypes.byref(dims.c()), ctypes.byref(state.c())


def mamba2_decode(dims, state, A, D, x, B, C, dt, y, stream=None):
    d, s = _refs(dims, state)
    _call("replayssm_mamba2_decode", d, s, _ptr(A), _ptr(D), _ptr(x), _ptr(B), _ptr(C),
          _ptr(dt), _ptr(y), _stream(stream))


def mamba2_decode_noalloc(dims, state, A, D, x, B, C, dt, y, stream=None):
    """mamba2_decode for callers that cannot allocate device memory when they
    decode (a plugin whose host framework owns all device memory, a serving
    loop that reserved the device for its state pool): the scratch comes from
    the library's fixed 16 MiB array instead of state.work and state.sync.
    Calls that overlap on the GPU share that array and race."""
    d, s = _refs(dims, state)
    _call("replayssm_mamba2_decode_noalloc", d, s, _ptr(A), _ptr(D), _ptr(x), _ptr(B), _ptr(C),
          _ptr(dt), _ptr(y), _stream(stream))


def mamba2_decode_noalloc_bytes(dims: LayerDims) -> int:
    """Bytes of the fixed scratch mamba2_decode_noalloc needs for these sizes
    (at most NOALLOC_SCRATCH_BYTES, else the call is refused); 0 if invalid."""
    return int(_abi.lib.replayssm_mamba2_decode_noalloc_bytes(ctypes.byref(dims.c())))


def mamba2_fold_decode(dims, state, A, D, x, B, C, dt, y, stream=None):
    """consolidate(k_next=1) then mamba2_decode in one call: a full ring is
    folded while its state rows stream past."""
    d, s = _refs(dims, state)
    _call("replayssm_mamba2_fold_decode", d, s, _ptr(A), _ptr(D), _ptr(x), _ptr(B), _ptr(C),
          _ptr(dt), _ptr(y), _stream(stream))


def gdn_decode(dims, state, q, k, v, alpha, beta, scale, o, stream=None):
    d, s = _refs(dims, state)
    _call("replayssm_gdn_decode", d, s, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
          float(scale), _ptr(o), _stream(stream))


def gdn_fold_decode(dims, state, q, k, v, alpha, beta, scale, o, stream=None):
    """consolidate(k_next=1) + gdn_decode in one call: full rings are folded
    and their token decoded from the new rows."""
    d, s = _refs(dims, state)
    _call("replayssm_gdn_fold_decode", d, s, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
          float(scale), _ptr(o), _stream(stream))


def consolidate(dims, state, A=None, k_next=1, force=False, stream=None):
    d, s = _refs(dims, state)
    _call("replayssm_consolidate", d, s, _ptr(A), int(k_next), int(bool(force)), _stream(stream))


def spec_verify(dims, state, K, q, k, v, alpha, beta, scale, o, stream=None):
    d, s = _refs(dims, state)
    _call("replayssm_spec_verify", d, s, int(K), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
          _ptr(beta), float(scale), _ptr(o), _stream(stream))


def mamba2_spec_verify(dims, state, K, A, D, x, B, C, dt, y, stream=None):
    d, s = _refs(dims, state)
    _call("replayssm_mamba2_spec_verify", d, s, int(K), _ptr(A), _ptr(D), _ptr(x), _ptr(B),
          _ptr(C), _ptr(dt), _ptr(y), _stream(stream))


def accept(dims, state, m, K, stream=None):
    _int32(m, "m")
    if m.numel() != dims.batch:
        raise ValueError("m must hold one count per sequence")
    d, s = _refs(dims, state)
    _call("replayssm_accept", d, s, _ptr(m), int(K), _stream(stream))


def refresh_read_copy(dims, state, stream=None):
    d, s = _refs(dims, state)
    _call("replayssm_refresh_read_copy", d, s, _stream(stream))


def conventional_mamba2_step(dims, S, A, D, x, B, C, dt, y, stream=None):
    _call("replayssm_conventional_mamba2_step", ctypes.byref(dims.c()), _ptr(S), _ptr(A),
          _ptr(D), _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(y), _stream(stream))


def conventional_gdn_step(dims, S, q, k, v, alpha, beta, scale, o, stream=None):
    _call("replayssm_conventional_gdn_step", ctypes.byref(dims.c()), _ptr(S), _ptr(q), _ptr(k),
          _ptr(v), _ptr(alpha), _ptr(beta), float(scale), _ptr(o), _stream(stream))


def conventional_gdn_verify(dims, S, K, q, k, v, alpha, beta, scale, snapshots, o, stream=None):
    """Baseline speculative verify: K drafts stepped with a state snapshot each."""
    _call("replayssm_conventional_gdn_verify", ctypes.byref(dims.c()), _ptr(S), int(K), _ptr(q),
          _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), float(scale), _ptr(snapshots), _ptr(o),
          _stream(stream))


def conventional_accept(dims, S, snapshots, m, K, status=None, stream=None):
    """Baseline accept: S = snapshot m - 1 per sequence (m = 0: unchanged)."""
    _int32(m, "m")
    if m.numel() != dims.batch:
        raise ValueError("m must hold one count per sequence")
    _call("replayssm_conventional_accept", ctypes.byref(dims.c()), _ptr(S), _ptr(snapshots),
          _ptr(m), int(K), _ptr(status), _stream(stream))


def copy_sequences(dims, src, src_idx, dst, dst_idx, stream=None):
    """Copy whole sequences (checkpoint, read copy, ring, pointers) between states."""
    n = int(_int32(src_idx, "src_idx").numel())
    if _int32(dst_idx, "dst_idx").numel() != n:
        raise ValueError("src_idx and dst_idx must have the same length")
    _call("replayssm_copy_sequences", ctypes.byref(dims.c()), ctypes.byref(src.c()),
          _ptr(src_idx), ctypes.byref(dst.c()), _ptr(dst_idx), n, _stream(stream))


def workspace_bytes(dims: LayerDims, K: int = 1) -> int:
    """Bytes of scratch a state needs for decode (K = 1) and verify with up to K drafts."""
    return int(_abi.lib.replayssm_workspace_bytes(ctypes.byref(dims.c()), int(K)))


def delta_kernel_config(dims: LayerDims, K: int = 1, read_copy: bool = True,
                        smem_limit: int = 0) -> dict:
    """Launch configuration of the GDN/KDA decode (K = 1) or verify kernel for
    these sizes (host only; smem_limit 0 means the B300's), as a dict."""
    out = _abi.DeltaConfig()
    _call("replayssm_delta_kernel_config", ctypes.byref(dims.c()), int(K), int(bool(read_copy)),
          int(smem_limit), ctypes.byref(out))
    return {name: int(getattr(out, name)) for name, _ in _abi.DeltaConfig._fields_}


def version() -> int:
    return int(_abi.lib.replayssm_version())
