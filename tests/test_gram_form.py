"""The algebra of the tensor-core GDN verify, checked on the CPU against the
oracle's replay (float64).

The kernel never runs the backward sweep "u <- A_j u" of the replay
("NVIDIA y Princeton aceleran modelos híbridos…", paragraphs 2 and 3).
It forms, for query t over the entries 0..top (top = len + t):
  - G = K K^T and P[j][t] = scale k_j . q_t (one tensor-core tile);
  - the coefficients c from scalar updates: a[j] starts at P[j][t]; entry i,
    from top down to 0, gives c_i = beta_i a[i] and then
    a[j] <- alpha_i (a[j] - c_i G[j][i]) for j < i;
  - A_i = alpha_0 ... alpha_i, the weights w_t = A_top scale (on q_t) and
    -c_i A_i (on k_i);
  - o_t = S [q | k]^T w_t + sum_i c_i v_i.
This file restates those steps in numpy and holds them to the oracle's
``delta_replay_output`` for single decodes, K drafts, short rings and gates
of 0, so that the identity the kernel relies on is pinned apart from the
GPU.
"""

import numpy as np
import pytest

from oracle.replay import delta_replay_output


def gram_form(S, ks, vs, alphas, betas, qs, length, scale, gate_in_update=True):
    """o[t] for queries t < K over entries 0..length + t, one (sequence, head):
    S [d_v, d_k]; ks [n, d_k]; vs [n, d_v]; alphas, betas [n]; qs [K, d_k]."""
    K, n = len(qs), length + len(qs)
    G = ks @ ks.T
    P = scale * ks @ qs.T
    A = np.cumprod(alphas)
    Y = S @ np.concatenate([qs, ks]).T          # [d_v, K + n]
    out = []
    for t in range(K):
        top = length + t
        a = P[:, t].copy()
        c = np.zeros(n)
        for i in range(top, -1, -1):
            c[i] = betas[i] * a[i]
            for j in range(i):
                a[j] = (alphas[i] if gate_in_update else 1.0) * (a[j] - c[i] * G[j, i])
        w = np.zeros(K + n)
        w[t] = A[top] * scale
        w[K:K + top + 1] = -c[:top + 1] * A[:top + 1]
        out.append(Y @ w + vs[:top + 1].T @ c[:top + 1])
    return np.stack(out)


def oracle_outputs(S, ks, vs, alphas, betas, qs, length, scale):
    out = []
    for t in range(len(qs)):
        entries = [{"k": ks[j][None, None], "v": vs[j][None, None],
                    "alpha": np.array([[alphas[j]]]), "beta": np.array([[betas[j]]])}
                   for j in range(length + t + 1)]
        out.append(delta_replay_output(S[None, None], entries, qs[t][None, None], scale)[0, 0])
    return np.stack(out)


def draw(seed, length, K, dk=32, dv=24):
    r = np.random.default_rng(seed)
    n = length + K
    ks = r.standard_normal((n, dk))
    ks /= np.linalg.norm(ks, axis=1, keepdims=True)
    return (r.standard_normal((dv, dk)) * 0.3, ks, r.standard_normal((n, dv)),
            r.uniform(0.9, 1.0, n), 1 / (1 + np.exp(-r.standard_normal(n))),
            r.standard_normal((K, dk)))


@pytest.mark.parametrize("length,K", [(0, 1), (8, 1), (15, 1), (0, 4), (5, 4), (12, 4), (8, 8)])
def test_matches_replay(length, K):
    S, ks, vs, al, be, qs = draw(10 + length + K, length, K)
    got = gram_form(S, ks, vs, al, be, qs, length, 0.8)
    ref = oracle_outputs(S, ks, vs, al, be, qs, length, 0.8)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_zero_and_vanishing_gates():
    """A gate of 0 forgets everything before its entry; gates of 1e-30 make
    the products underflow FP32 but not the float64 reference."""
    S, ks, vs, al, be, qs = draw(7, 9, 4)
    al[3] = 0.0
    al[6] = 1e-30
    got = gram_form(S, ks, vs, al, be, qs, 9, 1.0)
    ref = oracle_outputs(S, ks, vs, al, be, qs, 9, 1.0)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_a_dropped_update_is_caught():
    """The scalar updates are needed: leaving out the gate of the update
    (a[j] <- a[j] - c_i G[j][i]) moves the outputs away from the replay."""
    S, ks, vs, al, be, qs = draw(3, 8, 2)
    al = np.full_like(al, 0.5)
    good = gram_form(S, ks, vs, al, be, qs, 8, 1.0)
    ref = oracle_outputs(S, ks, vs, al, be, qs, 8, 1.0)
    np.testing.assert_allclose(good, ref, rtol=1e-12, atol=1e-12)
    bad = gram_form(S, ks, vs, al, be, qs, 8, 1.0, gate_in_update=False)
    assert np.abs(bad - ref).max() > 1e-3
