"""Conventional per-token SSM decode recurrences, float64 (oracle; tests only).

These are the plain definitions that the ReplaySSM method must reproduce:
"ReplaySSM: o ganho aparece na carga concorrente…", section "Cuidados e
limites", states that its outputs equal conventional decoding apart from
floating-point differences. The layer types are the ones named in "NVIDIA
présente ReplaySSM…", section "Pourquoi les hybrides sont devenus la norme";
each update below is the standard published decode step of that layer type,
in the orientation where a delta-rule state S is d_v x d_k and o = S q.

All arrays carry leading [batch, heads] axes; every step is one token.
"""

from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def expand_groups(BC: np.ndarray, heads: int) -> np.ndarray:
    """Map Mamba-2 B/C of shape [b, G, N] to per-head [b, H, N] (head h uses group h // (H/G))."""
    G = BC.shape[1]
    if heads % G:
        raise ValueError("heads must be a multiple of groups")
    return np.repeat(_f64(BC), heads // G, axis=1)


def mamba2_step(h, x, B, C, dt, A, D):
    """One conventional Mamba-2 decode step (scalar-per-head A).

    h [b,H,P,N]; x [b,H,P]; B, C [b,G,N]; dt [b,H] (already activated);
    A, D [H]. With dA = exp(dt*A):
        h' = dA * h + dt * x (outer) B
        y  = h' C + D * x
    Returns (h', y) in float64.
    """
    h, x, dt, A, D = _f64(h), _f64(x), _f64(dt), _f64(A), _f64(D)
    H = h.shape[1]
    Bh, Ch = expand_groups(B, H), expand_groups(C, H)
    dA = np.exp(dt * A[None, :])
    h_new = dA[:, :, None, None] * h + (dt[:, :, None] * x)[:, :, :, None] * Bh[:, :, None, :]
    y = np.matmul(h_new, Ch[:, :, :, None])[..., 0] + D[None, :, None] * x
    return h_new, y


def delta_step(S, q, k, v, alpha, beta, scale=1.0):
    """One conventional gated delta-rule decode step (GDN or KDA gate).

    S [b,H,d_v,d_k]; q, k [b,H,d_k]; v [b,H,d_v]; beta [b,H];
    alpha [b,H] (Gated DeltaNet: scalar gate) or [b,H,d_k] (KDA: per key
    channel). With A_t = Diag(alpha)(I - beta k k^T):
        S' = S A_t + beta v k^T
        o  = scale * S' q
    Returns (S', o) in float64.
    """
    S, q, k, v = _f64(S), _f64(q), _f64(k), _f64(v)
    alpha, beta = _f64(alpha), _f64(beta)
    if alpha.ndim == 2:
        G = alpha[:, :, None, None] * S          # S Diag(alpha), scalar alpha
    else:
        G = S * alpha[:, :, None, :]             # S Diag(alpha): scale key columns
    Gk = np.matmul(G, k[:, :, :, None])[..., 0]  # (S Diag(alpha)) k, [b,H,d_v]
    b = beta[:, :, None, None]
    S_new = G - b * Gk[:, :, :, None] * k[:, :, None, :] + b * v[:, :, :, None] * k[:, :, None, :]
    o = scale * np.matmul(S_new, q[:, :, :, None])[..., 0]
    return S_new, o
