"""The ReplaySSM replay formulas, evaluated naively in float64 (oracle; tests only).

"NVIDIA y Princeton aceleran modelos híbridos…", paragraph 2: on a normal
step the token's inputs are appended to the buffer and the output is computed
from the checkpoint; the persistent state is only updated when the buffer
fills. For a checkpoint taken at position c and buffered tokens c+1..t
(n = t - c, the newest one being the current token) the output is therefore
a function of the checkpoint and the buffer alone. Writing the conventional
recurrence out over the buffer gives:

Mamba-2 (dA_i = exp(dt_i A)):
    y_t = (prod_{i=1..n} dA_i) (h_c C_t)
          + sum_{j=1..n} w_j (C_t . B_j) x_j + D x_t,
    w_j = dt_j prod_{i=j+1..n} dA_i

Gated delta rule (A_j = Diag(alpha_j)(I - beta_j k_j k_j^T)):
    S_t q = S_c A_1 ... A_n q + sum_j beta_j v_j (k_j^T A_{j+1} ... A_n q)
  evaluated by the backward sweep u <- q; for j = n..1:
    s = k_j . u;  o += beta_j s v_j;  u <- A_j u;   then o += S_c u.

These are a second, independent route to the same numbers as
``oracle.recurrences``; the tests check the two against each other.
Entries are lists ordered oldest to newest; every array carries leading
[batch, heads] axes (Mamba-2 B and C carry [batch, groups]).
"""

from __future__ import annotations

import numpy as np

from .recurrences import expand_groups


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def mamba2_replay_output(h_c, entries, C_t, A, D):
    """y_t from checkpoint h_c [b,H,P,N] and n buffered entries (dicts x, B, dt)."""
    h_c, A, D = _f64(h_c), _f64(A), _f64(D)
    H = h_c.shape[1]
    n = len(entries)
    Ct = expand_groups(C_t, H)                                  # [b,H,N]
    dA = [np.exp(_f64(e["dt"]) * A[None, :]) for e in entries]  # each [b,H]
    decay_all = np.ones_like(dA[0])
    for a in dA:
        decay_all = decay_all * a
    y = decay_all[:, :, None] * np.matmul(h_c, Ct[:, :, :, None])[..., 0]
    for j in range(n):
        w = _f64(entries[j]["dt"]).copy()
        for i in range(j + 1, n):
            w = w * dA[i]
        CB = np.sum(Ct * expand_groups(entries[j]["B"], H), axis=-1)  # [b,H]
        y = y + (w * CB)[:, :, None] * _f64(entries[j]["x"])
    return y + D[None, :, None] * _f64(entries[-1]["x"])


def mamba2_replay_fold(h_c, entries, A):
    """Checkpoint after folding the n entries: (prod dA) h_c + sum_j w_j x_j (outer) B_j."""
    h_c, A = _f64(h_c), _f64(A)
    H = h_c.shape[1]
    n = len(entries)
    dA = [np.exp(_f64(e["dt"]) * A[None, :]) for e in entries]
    decay_all = np.ones_like(dA[0])
    for a in dA:
        decay_all = decay_all * a
    h = decay_all[:, :, None, None] * h_c
    for j in range(n):
        w = _f64(entries[j]["dt"]).copy()
        for i in range(j + 1, n):
            w = w * dA[i]
        xw = w[:, :, None] * _f64(entries[j]["x"])
        h = h + xw[:, :, :, None] * expand_groups(entries[j]["B"], H)[:, :, None, :]
    return h


def _apply_A(u, k, alpha, beta):
    """A_j u = Diag(alpha)(u - beta (k . u) k) for u, k [b,H,d_k]."""
    s = np.sum(k * u, axis=-1)
    r = u - (beta * s)[:, :, None] * k
    return r * (alpha[:, :, None] if alpha.ndim == 2 else alpha)


def delta_replay_output(S_c, entries, q_t, scale=1.0):
    """o_t from checkpoint S_c [b,H,d_v,d_k] and n entries (dicts k, v, alpha, beta)."""
    S_c = _f64(S_c)
    u = scale * _f64(q_t)
    o = np.zeros(S_c.shape[:3])
    for e in reversed(entries):
        k, v = _f64(e["k"]), _f64(e["v"])
        alpha, beta = _f64(e["alpha"]), _f64(e["beta"])
        s = np.sum(k * u, axis=-1)
        o = o + (beta * s)[:, :, None] * v
        u = _apply_A(u, k, alpha, beta)
    return o + np.matmul(S_c, u[:, :, :, None])[..., 0]
