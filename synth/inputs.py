"""Seeded generators for the decode workloads (no decode arithmetic here).

Every draw comes from ``numpy.random.default_rng([seed, stream, index])``, so a
step's (or a speculative round's) inputs can be regenerated on their own, in
any order, on any machine. Values are drawn in float32; fields that the
workloads store as bfloat16 are rounded to the nearest bfloat16 (ties to
even) *here*, before either side sees them, so the CUDA path and the oracle
consume bit-identical numbers.

Distributions (the layer types are the ones the pages name: Mamba-2, Gated
DeltaNet and a Kimi-Delta-Attention-style per-channel gate):

Mamba-2 (per head: state P x N, scalar A_h < 0, skip D_h)
  x ~ N(0, 1)                      [batch, H, P]
  B, C ~ N(0, 1) / sqrt(N)         [batch, G, N]
  dt = clamp(softplus(dt_raw + dt_bias_h), 1e-3, 0.1), dt_raw ~ N(0, 1)
  dt_bias_h = softplus^-1(dt0_h),  dt0_h log-uniform in [1e-3, 0.1]
  A_h = -exp(U(0, ln 16)),  D_h ~ N(0, 1),  h_c at start ~ N(0, 0.1)

Gated DeltaNet / KDA (per head: state d_v x d_k)
  q, k = z / ||z||, z ~ N(0, I)    [batch, H, d_k]
  v ~ N(0, 1)                      [batch, H, d_v]
  alpha = 0.9 + 0.1 * exp(-softplus(z)), z ~ N(0, 1): per head (GDN) or per
          head and key channel (KDA), so alpha lies in (0.9, 1)
  beta = sigmoid(z), z ~ N(0, 1)   [batch, H]
  S_c at start ~ N(0, 0.1)
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Stream labels: one independent random stream per kind of draw.
_PARAMS, _STATE, _STEP, _DRAFTS, _ACCEPT = 0, 1, 2, 3, 4


def _rng(seed: int, stream: int, index: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream), int(index)])


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); float32 out."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).reshape(a.shape)


def _vec(a: np.ndarray, in_dtype: str) -> np.ndarray:
    if in_dtype == "bf16":
        return bf16_round(a)
    if in_dtype == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    raise ValueError(f"unknown input dtype {in_dtype!r}")


def _softplus(z: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, z)


def _l2norm(z: np.ndarray) -> np.ndarray:
    return z / np.linalg.norm(z, axis=-1, keepdims=True)


@dataclass(frozen=True)
class Mamba2Workload:
    """Shape and seed of a Mamba-2 decode workload."""

    batch: int
    heads: int
    P: int
    N: int
    groups: int = 1
    window: int = 16
    steps: int = 64
    in_dtype: str = "bf16"
    seed: int = 1
    K: int = 1  # drafts per speculative round

    @property
    def name(self) -> str:
        return (f"mamba2_b{self.batch}_h{self.heads}_p{self.P}_n{self.N}_g{self.groups}"
                f"_w{self.window}_{self.in_dtype}")


@dataclass(frozen=True)
class DeltaWorkload:
    """Shape and seed of a Gated DeltaNet ("gdn") or KDA-gate ("kda") workload."""

    kind: str
    batch: int
    heads: int
    dk: int
    dv: int
    window: int = 16
    steps: int = 64
    in_dtype: str = "bf16"
    seed: int = 3
    K: int = 0  # draft tokens per speculative round (0: plain decode)

    @property
    def name(self) -> str:
        s = (f"{self.kind}_b{self.batch}_h{self.heads}_dk{self.dk}_dv{self.dv}"
             f"_w{self.window}_{self.in_dtype}")
        return s + (f"_k{self.K}" if self.K else "")


# ---------------------------------------------------------------- Mamba-2


def mamba2_params(seed: int, heads: int):
    """Per-head constants: (A [H], D [H], dt_bias [H]), all float32."""
    r = _rng(seed, _PARAMS)
    A = -np.exp(r.uniform(0.0, np.log(16.0), size=heads))
    D = r.standard_normal(heads)
    dt0 = np.exp(r.uniform(np.log(1e-3), np.log(0.1), size=heads))
    dt_bias = dt0 + np.log(-np.expm1(-dt0))  # inverse softplus
    return A.astype(np.float32), D.astype(np.float32), dt_bias.astype(np.float32)


def mamba2_initial_state(seed: int, batch: int, heads: int, P: int, N: int) -> np.ndarray:
    """Initial checkpoint h_c ~ N(0, 0.1), float32 [batch, H, P, N]."""
    r = _rng(seed, _STATE)
    return (0.1 * r.standard_normal((batch, heads, P, N), dtype=np.float32)).astype(np.float32)


def mamba2_step_inputs(seed: int, step: int, batch: int, heads: int, groups: int,
                       P: int, N: int, dt_bias: np.ndarray, in_dtype: str = "bf16"):
    """One decode token for every sequence: dict x, B, C (vector fields), dt."""
    r = _rng(seed, _STEP, step)
    x = r.standard_normal((batch, heads, P), dtype=np.float32)
    inv = np.float32(1.0 / np.sqrt(N))
    B = r.standard_normal((batch, groups, N), dtype=np.float32) * inv
    C = r.standard_normal((batch, groups, N), dtype=np.float32) * inv
    dt_raw = r.standard_normal((batch, heads))
    dt = np.clip(_softplus(dt_raw + dt_bias.astype(np.float64)), 1e-3, 0.1)
    return {
        "x": _vec(x, in_dtype),
        "B": _vec(B, in_dtype),
        "C": _vec(C, in_dtype),
        "dt": dt.astype(np.float32),
    }


# ---------------------------------------------------------- GDN / KDA


def delta_initial_state(seed: int, batch: int, heads: int, dv: int, dk: int) -> np.ndarray:
    """Initial checkpoint S_c ~ N(0, 0.1), float32 [batch, H, d_v, d_k]."""
    r = _rng(seed, _STATE)
    return (0.1 * r.standard_normal((batch, heads, dv, dk), dtype=np.float32)).astype(np.float32)


def _delta_token(r: np.random.Generator, lead: tuple, heads: int, dk: int, dv: int,
                 kind: str, in_dtype: str):
    shp = lead + (heads,)
    q = _l2norm(r.standard_normal(shp + (dk,), dtype=np.float32))
    k = _l2norm(r.standard_normal(shp + (dk,), dtype=np.float32))
    v = r.standard_normal(shp + (dv,), dtype=np.float32)
    gshape = shp if kind == "gdn" else shp + (dk,)
    if kind not in ("gdn", "kda"):
        raise ValueError(f"unknown delta kind {kind!r}")
    alpha = 0.9 + 0.1 * np.exp(-_softplus(r.standard_normal(gshape)))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal(shp)))
    return {
        "q": _vec(q, in_dtype),
        "k": _vec(k, in_dtype),
        "v": _vec(v, in_dtype),
        "alpha": alpha.astype(np.float32),
        "beta": beta.astype(np.float32),
    }


def delta_step_inputs(seed: int, step: int, batch: int, heads: int, dk: int, dv: int,
                      kind: str = "gdn", in_dtype: str = "bf16"):
    """One decode token per sequence: dict q, k, v [b,H,d], alpha, beta."""
    return _delta_token(_rng(seed, _STEP, step), (batch,), heads, dk, dv, kind, in_dtype)


def spec_draft_inputs(seed: int, rnd: int, batch: int, K: int, heads: int, dk: int, dv: int,
                      kind: str = "gdn", in_dtype: str = "bf16"):
    """K draft tokens per sequence for one speculative round: fields [b, K, H, ...]."""
    return _delta_token(_rng(seed, _DRAFTS, rnd), (batch, K), heads, dk, dv, kind, in_dtype)


def mamba2_draft_inputs(seed: int, rnd: int, batch: int, K: int, heads: int, groups: int,
                        P: int, N: int, dt_bias: np.ndarray, in_dtype: str = "bf16"):
    """K Mamba-2 draft tokens per sequence for one speculative round:
    x [b, K, H, P], B and C [b, K, G, N], dt [b, K, H] (same distributions as
    a decode token)."""
    r = _rng(seed, _DRAFTS, rnd)
    x = r.standard_normal((batch, K, heads, P), dtype=np.float32)
    inv = np.float32(1.0 / np.sqrt(N))
    B = r.standard_normal((batch, K, groups, N), dtype=np.float32) * inv
    C = r.standard_normal((batch, K, groups, N), dtype=np.float32) * inv
    dt_raw = r.standard_normal((batch, K, heads))
    dt = np.clip(_softplus(dt_raw + dt_bias.astype(np.float64)), 1e-3, 0.1)
    return {"x": _vec(x, in_dtype), "B": _vec(B, in_dtype), "C": _vec(C, in_dtype),
            "dt": dt.astype(np.float32)}


def accept_counts(seed: int, rnd: int, batch: int, K: int) -> np.ndarray:
    """Accepted draft count per sequence for one round, uniform on {0..K}, int32."""
    return _rng(seed, _ACCEPT, rnd).integers(0, K + 1, size=batch).astype(np.int32)
