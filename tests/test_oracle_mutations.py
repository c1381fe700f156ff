"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each one.

A pin set that passes a wrong oracle proves nothing; every mutant below must
make at least one pin of ``tests/oracle_pins.py`` fail.
"""

import numpy as np
import pytest

import oracle.method as om
import oracle.recurrences as rec
import oracle.replay as rep
import oracle_pins

_f = rec._f64


def _m2_parts(h, x, B, C, dt, A, D):
    h, x, dt, A, D = _f(h), _f(x), _f(dt), _f(A), _f(D)
    H = h.shape[1]
    return h, x, rec.expand_groups(B, H), rec.expand_groups(C, H), dt, A, D


def m2_no_skip(h, x, B, C, dt, A, D):
    h, x, Bh, Ch, dt, A, D = _m2_parts(h, x, B, C, dt, A, D)
    hn = np.exp(dt * A)[..., None, None] * h + (dt[..., None] * x)[..., None] * Bh[:, :, None, :]
    return hn, np.einsum("bhpn,bhn->bhp", hn, Ch)


def m2_old_state_output(h, x, B, C, dt, A, D):
    h, x, Bh, Ch, dt, A, D = _m2_parts(h, x, B, C, dt, A, D)
    hn = np.exp(dt * A)[..., None, None] * h + (dt[..., None] * x)[..., None] * Bh[:, :, None, :]
    return hn, np.einsum("bhpn,bhn->bhp", h, Ch) + D[None, :, None] * x


def m2_sign_A(h, x, B, C, dt, A, D):
    return rec_m2(h, x, B, C, dt, -np.asarray(A), D)


def m2_no_dt_input(h, x, B, C, dt, A, D):
    h, x, Bh, Ch, dt, A, D = _m2_parts(h, x, B, C, dt, A, D)
    hn = np.exp(dt * A)[..., None, None] * h + x[..., None] * Bh[:, :, None, :]
    return hn, np.einsum("bhpn,bhn->bhp", hn, Ch) + D[None, :, None] * x


def m2_swap_BC(h, x, B, C, dt, A, D):
    return rec_m2(h, x, C, B, dt, A, D)


def _delta_parts(S, q, k, v, alpha, beta):
    return _f(S), _f(q), _f(k), _f(v), _f(alpha), _f(beta)


def d_transposed_output(S, q, k, v, alpha, beta, scale=1.0):
    Sn, _ = rec_delta(S, q, k, v, alpha, beta, scale)
    return Sn, scale * np.einsum("bhvk,bhv->bhk", Sn, _f(q))


def d_gate_after(S, q, k, v, alpha, beta, scale=1.0):
    S, q, k, v, alpha, beta = _delta_parts(S, q, k, v, alpha, beta)
    b = beta[..., None, None]
    P = S - b * np.einsum("bhvk,bhk->bhv", S, k)[..., None] * k[:, :, None, :]
    G = alpha[..., None, None] * P if alpha.ndim == 2 else P * alpha[:, :, None, :]
    Sn = G + b * v[..., None] * k[:, :, None, :]
    return Sn, scale * np.einsum("bhvk,bhk->bhv", Sn, q)


def d_sign_flip(S, q, k, v, alpha, beta, scale=1.0):
    S, q, k, v, alpha, beta = _delta_parts(S, q, k, v, alpha, beta)
    G = alpha[..., None, None] * S if alpha.ndim == 2 else S * alpha[:, :, None, :]
    b = beta[..., None, None]
    Sn = G + b * np.einsum("bhvk,bhk->bhv", G, k)[..., None] * k[:, :, None, :] \
        + b * v[..., None] * k[:, :, None, :]
    return Sn, scale * np.einsum("bhvk,bhk->bhv", Sn, q)


def d_no_gate(S, q, k, v, alpha, beta, scale=1.0):
    return rec_delta(S, q, k, v, np.ones_like(np.asarray(alpha)), beta, scale)


def d_old_state_output(S, q, k, v, alpha, beta, scale=1.0):
    Sn, _ = rec_delta(S, q, k, v, alpha, beta, scale)
    return Sn, scale * np.einsum("bhvk,bhk->bhv", _f(S), _f(q))


def d_beta_only_on_write(S, q, k, v, alpha, beta, scale=1.0):
    S, q, k, v, alpha, beta = _delta_parts(S, q, k, v, alpha, beta)
    G = alpha[..., None, None] * S if alpha.ndim == 2 else S * alpha[:, :, None, :]
    Sn = G - np.einsum("bhvk,bhk->bhv", G, k)[..., None] * k[:, :, None, :] \
        + beta[..., None, None] * v[..., None] * k[:, :, None, :]
    return Sn, scale * np.einsum("bhvk,bhk->bhv", Sn, q)


def r_forward_sweep(S_c, entries, q_t, scale=1.0):
    return rec_replay(S_c, list(reversed(entries)), q_t, scale)


def r_ungated_sweep(S_c, entries, q_t, scale=1.0):
    ent = [dict(e, alpha=np.ones_like(np.asarray(e["alpha"], float))) for e in entries]
    return rec_replay(S_c, ent, q_t, scale)


def r_m2_no_decay_on_checkpoint(h_c, entries, C_t, A, D):
    # drops the decay factor on the checkpoint term
    return rec_m2_replay(h_c, entries, C_t, A, D) + _ckpt_term_delta(h_c, entries, C_t, A)


def _ckpt_term_delta(h_c, entries, C_t, A):
    H = np.asarray(h_c).shape[1]
    Ct = rec.expand_groups(C_t, H)
    hc = np.matmul(_f(h_c), Ct[..., None])[..., 0]
    total = sum(_f(e["dt"]) for e in entries)
    return (1.0 - np.exp(total * _f(A)[None, :]))[..., None] * hc


rec_m2 = rec.mamba2_step
rec_delta = rec.delta_step
rec_replay = rep.delta_replay_output
rec_m2_replay = rep.mamba2_replay_output


def consolidate_off_by_one(self, k_next=1, force=False):
    fold = (self.len + k_next >= self.W) | (bool(force) & (self.len > 0))
    self.ckpt[fold] = self.committed[fold]
    self.head[fold] = (self.head[fold] + self.len[fold]) % self.W
    self.len[fold] = 0
    return fold


def consolidate_keeps_head(self, k_next=1, force=False):
    fold = (self.len + k_next > self.W) | (bool(force) & (self.len > 0))
    self.ckpt[fold] = self.committed[fold]
    self.len[fold] = 0
    return fold


_orig_write = om.ReplayOracle._write


def write_next_slot(self, mask, slot, tok):
    return _orig_write(self, mask, (slot + 1) % self.W, tok)


def restart_keeps_checkpoint(self, seqs, S0):
    seqs = np.asarray(seqs, np.int64)
    self.committed[seqs] = np.asarray(S0, np.float64)
    self.head[seqs] = 0
    self.len[seqs] = 0
    self.status[seqs] = 0


def restart_keeps_length(self, seqs, S0):
    seqs = np.asarray(seqs, np.int64)
    self.committed[seqs] = np.asarray(S0, np.float64)
    self.ckpt[seqs] = np.asarray(S0, np.float64)
    self.status[seqs] = 0


def spec_verify_unchained(self, K, drafts):
    """Every draft stepped from the committed state: drafts blind to each other."""
    ok = self.len + K <= self.W
    self.status[~ok] |= om.RING_FULL
    outs, states = [], []
    for i in range(K):
        tok = {k: np.asarray(v)[:, i] for k, v in drafts.items()}
        self._write(ok, (self.head + self.len + i) % self.W, tok)
        S, o = self._step(self.committed, tok)
        outs.append(o)
        states.append(S)
    out = np.stack(outs, axis=1)
    out[~ok] = np.nan
    self._drafts, self._verified = states, ok
    return out


_orig_accept = om.ReplayOracle.accept


def accept_moves_by_K(self, m, K):
    """The pointer advances over every verified draft, accepted or not."""
    _orig_accept(self, m, K)
    m = np.asarray(m, np.int64)
    good = (m >= 0) & (m <= K)
    self.len[good] += (K - m[good]).astype(np.int32)


def accept_clamps_silently(self, m, K):
    """An out-of-range accept count is clamped instead of flagged."""
    _orig_accept(self, np.clip(np.asarray(m, np.int64), 0, K), K)


def copy_without_ring(self, src, dst):
    """The copy takes the checkpoint and the pointers but not the ring bytes."""
    src, dst = np.asarray(src, np.int64), np.asarray(dst, np.int64)
    for arr in (self.committed, self.ckpt, self.head, self.len, self.status):
        arr[dst] = arr[src].copy()


def copy_without_pointers(self, src, dst):
    """The copy takes the states and the ring but keeps the destination's pointers."""
    src, dst = np.asarray(src, np.int64), np.asarray(dst, np.int64)
    for arr in (self.committed, self.ckpt, *self.ring.values()):
        arr[dst] = arr[src].copy()


def bf16_truncate(a):
    """Rounds toward zero (drops the low 16 bits)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return u.view(np.float32).astype(np.float64)


def bf16_ties_away(a):
    """Rounds half away from zero instead of to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.int64)
    u = ((u + 0x8000) >> 16) << 16
    return (u & 0xFFFFFFFF).astype(np.uint32).view(np.float32).astype(np.float64)


MUTANTS = [
    (rec, "mamba2_step", m2_no_skip),
    (rec, "mamba2_step", m2_old_state_output),
    (rec, "mamba2_step", m2_sign_A),
    (rec, "mamba2_step", m2_no_dt_input),
    (rec, "mamba2_step", m2_swap_BC),
    (rec, "delta_step", d_transposed_output),
    (rec, "delta_step", d_gate_after),
    (rec, "delta_step", d_sign_flip),
    (rec, "delta_step", d_no_gate),
    (rec, "delta_step", d_old_state_output),
    (rec, "delta_step", d_beta_only_on_write),
    (rep, "delta_replay_output", r_forward_sweep),
    (rep, "delta_replay_output", r_ungated_sweep),
    (rep, "mamba2_replay_output", r_m2_no_decay_on_checkpoint),
    (om.ReplayOracle, "consolidate", consolidate_off_by_one),
    (om.ReplayOracle, "consolidate", consolidate_keeps_head),
    (om.ReplayOracle, "_write", write_next_slot),
    (om.ReplayOracle, "restart", restart_keeps_checkpoint),
    (om.ReplayOracle, "restart", restart_keeps_length),
    (om.ReplayOracle, "spec_verify", spec_verify_unchained),
    (om.ReplayOracle, "accept", accept_moves_by_K),
    (om.ReplayOracle, "accept", accept_clamps_silently),
    (om.ReplayOracle, "copy_sequences", copy_without_ring),
    (om.ReplayOracle, "copy_sequences", copy_without_pointers),
    (om, "bf16_rne", bf16_truncate),
    (om, "bf16_rne", bf16_ties_away),
]


@pytest.mark.parametrize("owner,name,mutant", MUTANTS, ids=[m[2].__name__ for m in MUTANTS])
def test_mutant_is_caught(monkeypatch, owner, name, mutant):
    monkeypatch.setattr(owner, name, mutant)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {mutant.__name__}"
