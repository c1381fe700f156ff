"""Checks that pin the CPU oracle to facts outside itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
a closed form, an invariant fixed by the mathematics or the pages, an
independent published formulation, brute force on tiny inputs, or a
hand-worked fixture under ``tests/golden``. They always call the oracle
through its module attributes, so the mutation tests can swap a function for
a deliberately wrong one and check that some pin fails.
"""

from __future__ import annotations

import json
import os

import numpy as np

import oracle.method as om
import oracle.recurrences as rec
import oracle.replay as rep

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol, what):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# ----------------------------------------------------------------- inputs
def _as_f32(tok):
    """Token inputs are float32 numbers (as the ring stores them), held in float64."""
    return {k: np.asarray(v, np.float32).astype(np.float64) for k, v in tok.items()}


def m2_tokens(r, b, H, G, P, N, n):
    toks = []
    for _ in range(n):
        toks.append({
            "x": r.standard_normal((b, H, P)),
            "B": r.standard_normal((b, G, N)) / np.sqrt(N),
            "C": r.standard_normal((b, G, N)) / np.sqrt(N),
            "dt": r.uniform(1e-3, 0.1, (b, H)),
        })
    return [_as_f32(t) for t in toks]


def m2_params(r, H):
    return -np.exp(r.uniform(0, np.log(16), H)), r.standard_normal(H)


def delta_tokens(r, b, H, dk, dv, n, kda=False):
    toks = []
    for _ in range(n):
        q = r.standard_normal((b, H, dk))
        k = r.standard_normal((b, H, dk))
        toks.append({
            "q": q / np.linalg.norm(q, axis=-1, keepdims=True),
            "k": k / np.linalg.norm(k, axis=-1, keepdims=True),
            "v": r.standard_normal((b, H, dv)),
            "alpha": r.uniform(0.9, 1.0, (b, H, dk) if kda else (b, H)),
            "beta": r.uniform(0.05, 0.95, (b, H)),
        })
    return [_as_f32(t) for t in toks]


# ------------------------------------------------------------ Mamba-2 pins
def pin_mamba2_worked_examples():
    """Hand-worked P=N=1 and P=N=2 examples (tests/golden/worked_examples.json)."""
    g = _golden("worked_examples.json")
    ex = g["mamba2_scalar"]
    h = np.array(ex["h0"], float)[None, None]
    for t, tok in enumerate(ex["tokens"]):
        h, y = rec.mamba2_step(h, np.array(tok["x"])[None, None], np.array(tok["B"])[None, None],
                               np.array(tok["C"])[None, None], np.array([[tok["dt"]]]),
                               np.array([ex["A"]]), np.array([ex["D"]]))
        _close(h[0, 0], ex["h"][t], 1e-12, f"mamba2_scalar h{t + 1}")
        _close(y[0, 0], ex["y"][t], 1e-12, f"mamba2_scalar y{t + 1}")
    ex = g["mamba2_2x2"]
    h = np.array(ex["h0"], float)[None, None]
    for t, tok in enumerate(ex["tokens"]):
        h, y = rec.mamba2_step(h, np.array(tok["x"])[None, None], np.array(tok["B"])[None, None],
                               np.array(tok["C"])[None, None], np.array([[tok["dt"]]]),
                               np.array([ex["A"]]), np.array([tok["D"]]))
        _close(h[0, 0], ex["h"][t], 1e-12, f"mamba2_2x2 h{t + 1}")
        _close(y[0, 0], ex["y"][t], 1e-12, f"mamba2_2x2 y{t + 1}")


def pin_mamba2_single_token_zero_state():
    """From h = 0 one token gives h = dt x (outer) B and y = dt (C.B) x + D x."""
    r = _rng(11)
    b, H, P, N = 3, 4, 8, 16
    A, D = m2_params(r, H)
    tok = m2_tokens(r, b, H, 1, P, N, 1)[0]
    h, y = rec.mamba2_step(np.zeros((b, H, P, N)), tok["x"], tok["B"], tok["C"], tok["dt"], A, D)
    Bv, Cv = tok["B"][:, 0], tok["C"][:, 0]
    h_ref = tok["dt"][:, :, None, None] * tok["x"][:, :, :, None] * Bv[:, None, None, :]
    cb = np.sum(Cv * Bv, axis=-1)
    y_ref = (tok["dt"] * cb[:, None])[:, :, None] * tok["x"] + D[None, :, None] * tok["x"]
    _close(h, h_ref, 1e-14, "zero-state h")
    _close(y, y_ref, 1e-13, "zero-state y")


def pin_mamba2_pure_decay():
    """With x = 0 the state only decays: h_t = exp(A sum dt) h_0."""
    r = _rng(12)
    b, H, P, N, n = 2, 3, 4, 8, 9
    A, D = m2_params(r, H)
    h0 = r.standard_normal((b, H, P, N))
    h = h0
    toks = m2_tokens(r, b, H, 1, P, N, n)
    for tok in toks:
        h, y = rec.mamba2_step(h, np.zeros((b, H, P)), tok["B"], tok["C"], tok["dt"], A, D)
    total = sum(t["dt"] for t in toks)
    _close(h, np.exp(A[None, :] * total)[:, :, None, None] * h0, 1e-13, "pure decay")


def pin_mamba2_ssd_matrix_form():
    """The recurrence equals Mamba-2's quadratic ("attention-like") matrix form.

    y_t = exp(A cs_t) h_0 C_t + sum_{s<=t} (C_t . B_s) exp(A (cs_t - cs_s)) dt_s x_s + D x_t
    with cs_t the running sum of dt. This is a second, independently derived
    formula (segment sums instead of a product of per-token decays).
    """
    r = _rng(13)
    b, H, P, N, T = 2, 3, 5, 7, 12
    A, D = m2_params(r, H)
    h0 = r.standard_normal((b, H, P, N))
    toks = m2_tokens(r, b, H, 1, P, N, T)
    h, ys = h0, []
    for tok in toks:
        h, y = rec.mamba2_step(h, tok["x"], tok["B"], tok["C"], tok["dt"], A, D)
        ys.append(y)
    dt = np.stack([t["dt"] for t in toks], axis=-1)          # [b,H,T]
    cs = np.cumsum(dt, axis=-1)
    Bm = np.stack([t["B"][:, 0] for t in toks], axis=1)      # [b,T,N]
    Cm = np.stack([t["C"][:, 0] for t in toks], axis=1)
    X = np.stack([t["x"] for t in toks], axis=2)             # [b,H,T,P]
    CB = np.einsum("btn,bsn->bts", Cm, Bm)                   # [b,T,T]
    seg = cs[:, :, :, None] - cs[:, :, None, :]              # [b,H,t,s]
    L = np.where(np.tril(np.ones((T, T), bool)), np.exp(A[None, :, None, None] * seg), 0.0)
    M = L * CB[:, None] * dt[:, :, None, :]
    Y = np.einsum("bhts,bhsp->bhtp", M, X)
    Y += np.exp(A[None, :, None] * cs)[..., None] * np.einsum("bhpn,btn->bhtp", h0, Cm)
    Y += D[None, :, None, None] * X
    _close(np.stack(ys, axis=2), Y, 1e-11, "SSD matrix form")


def pin_mamba2_replay_equals_conventional():
    """Output and fold from checkpoint + buffer equal the token-by-token recurrence."""
    r = _rng(14)
    b, H, G, P, N = 2, 4, 2, 6, 10
    A, D = m2_params(r, H)
    for n in (1, 2, 7, 16):
        h0 = r.standard_normal((b, H, P, N))
        toks = m2_tokens(r, b, H, G, P, N, n)
        h = h0
        for tok in toks:
            h, y = rec.mamba2_step(h, tok["x"], tok["B"], tok["C"], tok["dt"], A, D)
        _close(rep.mamba2_replay_output(h0, toks, toks[-1]["C"], A, D), y, 1e-11, f"replay y n={n}")
        _close(rep.mamba2_replay_fold(h0, toks, A), h, 1e-11, f"replay fold n={n}")


def pin_mamba2_groups():
    """Head h uses B/C group h // (H/G): G=2 equals two G=1 runs on the head halves."""
    r = _rng(15)
    b, H, P, N = 2, 4, 3, 5
    A, D = m2_params(r, H)
    h0 = r.standard_normal((b, H, P, N))
    tok = m2_tokens(r, b, H, 2, P, N, 1)[0]
    h, y = rec.mamba2_step(h0, tok["x"], tok["B"], tok["C"], tok["dt"], A, D)
    for g in range(2):
        sl = slice(2 * g, 2 * g + 2)
        hg, yg = rec.mamba2_step(h0[:, sl], tok["x"][:, sl], tok["B"][:, g:g + 1],
                                 tok["C"][:, g:g + 1], tok["dt"][:, sl], A[sl], D[sl])
        _close(h[:, sl], hg, 1e-14, f"group {g} h")
        _close(y[:, sl], yg, 1e-14, f"group {g} y")


# ------------------------------------------------------- delta-rule pins
def _one(a):
    return np.asarray(a, float)[None, None]


def pin_delta_worked_examples():
    """Hand-worked 2x2 GDN and KDA steps (tests/golden/worked_examples.json)."""
    g = _golden("worked_examples.json")
    for key in ("gdn_2x2", "kda_2x2"):
        ex = g[key]
        alpha = np.array([[ex["alpha"]]]) if key == "gdn_2x2" else _one(ex["alpha"])
        S1, o = rec.delta_step(_one(ex["S0"]), _one(ex["q"]), _one(ex["k"]), _one(ex["v"]),
                               alpha, np.array([[ex["beta"]]]))
        _close(S1[0, 0], ex["S1"], 1e-12, f"{key} S1")
        _close(o[0, 0], ex["o"], 1e-12, f"{key} o")


def pin_delta_single_token_zero_state():
    """From S = 0 one token gives S = beta v k^T and o = scale beta (k.q) v (any gate)."""
    r = _rng(21)
    for kda in (False, True):
        tok = delta_tokens(r, 2, 3, 8, 6, 1, kda)[0]
        S, o = rec.delta_step(np.zeros((2, 3, 6, 8)), tok["q"], tok["k"], tok["v"],
                              tok["alpha"], tok["beta"], scale=0.5)
        bvk = tok["beta"][:, :, None, None] * tok["v"][:, :, :, None] * tok["k"][:, :, None, :]
        kq = np.sum(tok["k"] * tok["q"], axis=-1)
        _close(S, bvk, 1e-14, "zero-state S")
        _close(o, 0.5 * (tok["beta"] * kq)[:, :, None] * tok["v"], 1e-14, "zero-state o")


def pin_delta_rule_writes_value():
    """alpha = 1, beta = 1, |k| = 1: the new state maps k_t to v_t exactly (S_t k_t = v_t)."""
    r = _rng(22)
    S = r.standard_normal((2, 3, 6, 8))
    tok = delta_tokens(r, 2, 3, 8, 6, 1)[0]
    k = tok["k"] / np.linalg.norm(tok["k"], axis=-1, keepdims=True)  # unit norm in float64
    S1, _ = rec.delta_step(S, tok["q"], k, tok["v"], np.ones((2, 3)), np.ones((2, 3)))
    _close(np.einsum("bhvk,bhk->bhv", S1, k), tok["v"], 1e-13, "S_t k_t = v_t")


def pin_delta_beta_zero():
    """beta = 0 leaves only the gate: alpha = 1 keeps S, scalar alpha scales S, KDA scales columns."""
    r = _rng(23)
    S = r.standard_normal((2, 3, 6, 8))
    tok = delta_tokens(r, 2, 3, 8, 6, 1, kda=True)[0]
    z = np.zeros((2, 3))
    S1, _ = rec.delta_step(S, tok["q"], tok["k"], tok["v"], np.ones((2, 3)), z)
    _close(S1, S, 0.0, "beta=0, alpha=1")
    a = r.uniform(0.5, 1.0, (2, 3))
    S1, _ = rec.delta_step(S, tok["q"], tok["k"], tok["v"], a, z)
    _close(S1, a[:, :, None, None] * S, 1e-15, "beta=0, scalar alpha")
    S1, _ = rec.delta_step(S, tok["q"], tok["k"], tok["v"], tok["alpha"], z)
    _close(S1, S * tok["alpha"][:, :, None, :], 1e-15, "beta=0, channel alpha")


def pin_kda_uniform_gate_is_gdn():
    """A KDA gate vector with equal entries reproduces the scalar-gate GDN step."""
    r = _rng(24)
    S = r.standard_normal((2, 3, 6, 8))
    tok = delta_tokens(r, 2, 3, 8, 6, 1)[0]
    a_vec = np.repeat(tok["alpha"][:, :, None], 8, axis=-1)
    S1, o1 = rec.delta_step(S, tok["q"], tok["k"], tok["v"], tok["alpha"], tok["beta"])
    S2, o2 = rec.delta_step(S, tok["q"], tok["k"], tok["v"], a_vec, tok["beta"])
    _close(S1, S2, 1e-14, "KDA uniform = GDN S")
    _close(o1, o2, 1e-14, "KDA uniform = GDN o")


def pin_delta_published_orientation():
    """Same outputs as the published form with a d_k x d_v state M = S^T.

    Kimi Delta Attention and Gated DeltaNet are published as
    M_t = (I - beta k k^T) Diag(alpha) M_{t-1} + beta k v^T, o_t = M_t^T q_t,
    written here independently with explicit d_k x d_k matrices.
    """
    r = _rng(25)
    dk, dv, T = 5, 4, 10
    for kda in (False, True):
        toks = delta_tokens(r, 1, 1, dk, dv, T, kda)
        S = r.standard_normal((1, 1, dv, dk))
        M = S[0, 0].T.copy()
        for tok in toks:
            S, o = rec.delta_step(S, tok["q"], tok["k"], tok["v"], tok["alpha"], tok["beta"])
            k, v, q = tok["k"][0, 0], tok["v"][0, 0], tok["q"][0, 0]
            be = tok["beta"][0, 0]
            a = tok["alpha"][0, 0] * np.ones(dk) if not kda else tok["alpha"][0, 0]
            M = (np.eye(dk) - be * np.outer(k, k)) @ np.diag(a) @ M + be * np.outer(k, v)
            _close(o[0, 0], M.T @ q, 1e-12, "published orientation")


def pin_delta_brute_force_products():
    """Tiny d: S_t = S_0 A_1..A_t + sum_j beta_j v_j k_j^T A_{j+1}..A_t with explicit A_j matrices."""
    r = _rng(26)
    d, T = 4, 7
    for kda in (False, True):
        toks = delta_tokens(r, 1, 1, d, d, T, kda)
        S0 = r.standard_normal((1, 1, d, d))
        S = S0
        for tok in toks:
            S, o = rec.delta_step(S, tok["q"], tok["k"], tok["v"], tok["alpha"], tok["beta"])
        Am = []
        for tok in toks:
            k = tok["k"][0, 0]
            a = tok["alpha"][0, 0] * np.ones(d) if not kda else tok["alpha"][0, 0]
            Am.append(np.diag(a) @ (np.eye(d) - tok["beta"][0, 0] * np.outer(k, k)))
        total = S0[0, 0].copy()
        for Aj in Am:
            total = total @ Aj
        for j, tok in enumerate(toks):
            term = tok["beta"][0, 0] * np.outer(tok["v"][0, 0], tok["k"][0, 0])
            for Ai in Am[j + 1:]:
                term = term @ Ai
            total = total + term
        _close(S[0, 0], total, 1e-12, "brute-force product")
        _close(o[0, 0], total @ toks[-1]["q"][0, 0], 1e-12, "brute-force output")


def pin_delta_orthonormal_keys_memorise():
    """alpha = 1, beta = 1 and orthonormal keys: after m writes S k_j = v_j for every j."""
    r = _rng(27)
    dk, dv, m = 8, 5, 6
    Q, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    S = r.standard_normal((1, 1, dv, dk))
    vs = r.standard_normal((m, dv))
    for j in range(m):
        k = Q[:, j][None, None]
        S, _ = rec.delta_step(S, k, k, vs[j][None, None], np.ones((1, 1)), np.ones((1, 1)))
    for j in range(m):
        _close(S[0, 0] @ Q[:, j], vs[j], 1e-12, f"memorised key {j}")


def pin_delta_replay_equals_conventional():
    """The backward u-sweep from checkpoint + buffer equals the token-by-token output."""
    r = _rng(28)
    for kda in (False, True):
        for n in (1, 2, 5, 16):
            S0 = r.standard_normal((2, 3, 6, 8))
            toks = delta_tokens(r, 2, 3, 8, 6, n, kda)
            S = S0
            for tok in toks:
                S, o = rec.delta_step(S, tok["q"], tok["k"], tok["v"], tok["alpha"], tok["beta"],
                                      scale=0.75)
            _close(rep.delta_replay_output(S0, toks, toks[-1]["q"], scale=0.75), o, 1e-11,
                   f"u-sweep n={n} kda={kda}")


# --------------------------------------------------- ring / method pins
def _id_token(kind, t, b):
    ids = np.array([t + 100 * s for s in range(b)], np.float64)
    if kind == "gdn":
        f = {"q": ids[:, None, None], "k": ids[:, None, None], "v": ids[:, None, None],
             "alpha": np.full((b, 1), 0.5), "beta": np.full((b, 1), 0.5)}
    return f


def pin_ring_golden_w4():
    """The scripted W=4 call sequence of tests/golden/ring_w4.json, slot by slot."""
    g = _golden("ring_w4.json")
    W = g["window"]
    orc = om.ReplayOracle("gdn", np.zeros((2, 1, 1, 1)), W)
    for i, c in enumerate(g["calls"]):
        op = c["op"]
        if op == "decode":
            orc.decode(_id_token("gdn", c["token"], 2))
        elif op == "consolidate":
            fold = orc.consolidate(c["k_next"], c["force"])
            assert list(fold) == c["fold"], f"call {i}: fold {fold}"
        elif op == "verify":
            toks = [_id_token("gdn", t, 2) for t in c["drafts"]]
            drafts = {k: np.stack([t[k] for t in toks], axis=1) for k in toks[0]}
            orc.spec_verify(len(c["drafts"]), drafts)
        elif op == "accept":
            orc.accept(np.array(c["m"]), c["K"])
        assert orc.head.tolist() == c["head"], f"call {i} ({op}): head {orc.head}"
        assert orc.len.tolist() == c["len"], f"call {i} ({op}): len {orc.len}"
        assert orc.status.tolist() == c["status"], f"call {i} ({op}): status {orc.status}"
        assert orc.ring["k"][:, :, 0, 0].tolist() == c["slots"], f"call {i} ({op}): slots"


def run_plain_decode(kind, W, T, seed, b=2, H=2, rows=4, cols=6):
    """Oracle decode loop (consolidate(1) then decode per token).

    Returns (tokens, outputs, oracle, initial state, (A, D) or None).
    """
    r = _rng(seed)
    S0 = r.standard_normal((b, H, rows, cols))
    if kind == "mamba2":
        A, D = m2_params(r, H)
        toks = m2_tokens(r, b, H, 1, rows, cols, T)
        orc = om.ReplayOracle(kind, S0, W, A=A, D=D)
        params = (A, D)
    else:
        toks = delta_tokens(r, b, H, cols, rows, T, kind == "kda")
        orc = om.ReplayOracle(kind, S0, W, scale=0.9)
        params = None
    outs = []
    for tok in toks:
        orc.consolidate(1)
        outs.append(orc.decode(tok))
    return toks, outs, orc, S0, params


def pin_w1_is_conventional():
    """W = 1: every token folds first, so outputs and state follow the plain recurrence."""
    for kind in ("mamba2", "gdn", "kda"):
        toks, outs, orc, S, params = run_plain_decode(kind, 1, 9, 31)
        for t, tok in enumerate(toks):
            if kind == "mamba2":
                S, y = rec.mamba2_step(S, tok["x"], tok["B"], tok["C"], tok["dt"], *params)
            else:
                S, y = rec.delta_step(S, tok["q"], tok["k"], tok["v"], tok["alpha"], tok["beta"], 0.9)
            _close(outs[t], y, 1e-12, f"{kind} W=1 output {t}")
        _close(orc.committed, S, 1e-12, f"{kind} W=1 state")
        # the checkpoint trails the committed state by the one buffered token
        assert np.all(orc.len == 1) and np.all(orc.head == 0)


def pin_replay_reads_checkpoint_and_ring():
    """After every decode, the replay formula on (checkpoint, ring) gives the decode output."""
    for kind in ("mamba2", "gdn", "kda"):
        r = _rng(41)
        b, H, rows, cols, W, T = 2, 2, 4, 6, 5, 23
        if kind == "mamba2":
            A, D = m2_params(r, H)
            toks = m2_tokens(r, b, H, 1, rows, cols, T)
            orc = om.ReplayOracle(kind, r.standard_normal((b, H, rows, cols)), W, A=A, D=D)
        else:
            toks = delta_tokens(r, b, H, cols, rows, T, kind == "kda")
            orc = om.ReplayOracle(kind, r.standard_normal((b, H, rows, cols)), W, scale=1.1)
        for t, tok in enumerate(toks):
            orc.consolidate(1)
            y = orc.decode(tok)
            _close(orc.replay_output(tok, "f64"), y, 1e-11, f"{kind} replay step {t}")


def pin_restart_is_a_fresh_sequence():
    """A slot taken over by a new sequence from the zero state mid-stream: its
    first output is the single-token closed form, the replay formula keeps
    agreeing with decode through later folds, and the other slot runs exactly
    as it would without the restart."""
    for kind in ("mamba2", "gdn", "kda"):
        r = _rng(47)
        b, H, rows, cols, W, T, t_join = 2, 2, 4, 6, 5, 17, 7
        S0 = r.standard_normal((b, H, rows, cols))
        if kind == "mamba2":
            A, D = m2_params(r, H)
            toks = m2_tokens(r, b, H, 1, rows, cols, T)
            mk = lambda: om.ReplayOracle(kind, S0, W, A=A, D=D)  # noqa: E731
        else:
            toks = delta_tokens(r, b, H, cols, rows, T, kind == "kda")
            mk = lambda: om.ReplayOracle(kind, S0, W, scale=0.7)  # noqa: E731
        orc, plain = mk(), mk()
        for t, tok in enumerate(toks):
            if t == t_join:
                orc.restart([1], np.zeros((1, H, rows, cols)))
            orc.consolidate(1)
            plain.consolidate(1)
            y = orc.decode(tok)
            y_plain = plain.decode(tok)
            _close(y[0], y_plain[0], 0.0, f"{kind} untouched slot, step {t}")
            _close(orc.replay_output(tok, "f64"), y, 1e-11, f"{kind} replay step {t}")
            if t == t_join:
                if kind == "mamba2":
                    cb = np.sum(tok["C"][1, 0] * tok["B"][1, 0])
                    want = (tok["dt"][1] * cb + D)[:, None] * tok["x"][1]
                else:
                    kq = np.sum(tok["k"][1] * tok["q"][1], axis=-1)
                    want = 0.7 * (tok["beta"][1] * kq)[:, None] * tok["v"][1]
                _close(y[1], want, 1e-13, f"{kind} first token after the restart")
        assert orc.len[1] == (T - t_join - 1) % W + 1, f"{kind} restarted slot length"


def pin_copied_sequence_continues_its_source():
    """A sequence copied mid-ring into a slot at another ring phase, then fed
    its own tokens, gives exactly what the plain recurrence gives from its
    source's history (the source's tokens up to the copy, then its own), and
    its checkpoint, ring and pointers replay to that output. Checked through
    later folds, for every layer kind."""
    for kind in ("mamba2", "gdn", "kda"):
        r = _rng(53)
        b, H, rows, cols, W, T, t_copy = 3, 2, 4, 6, 7, 23, 7
        S0 = r.standard_normal((b, H, rows, cols))
        if kind == "mamba2":
            A, D = m2_params(r, H)
            toks = m2_tokens(r, b, H, 1, rows, cols, T)
            orc = om.ReplayOracle(kind, S0, W, A=A, D=D)
            step = lambda S, k: rec.mamba2_step(S, k["x"], k["B"], k["C"], k["dt"], A, D)  # noqa: E731
        else:
            toks = delta_tokens(r, b, H, cols, rows, T, kind == "kda")
            orc = om.ReplayOracle(kind, S0, W, scale=0.8)
            step = lambda S, k: rec.delta_step(S, k["q"], k["k"], k["v"], k["alpha"],  # noqa: E731
                                               k["beta"], 0.8)
        ref = S0.copy()  # plain recurrence of sequences 0 and 1 (and 2 after the copy)
        for t, tok in enumerate(toks):
            if t == 5:  # the destination slot starts a new sequence: another phase
                orc.restart([2], np.zeros((1, H, rows, cols)))
            if t == t_copy:
                assert orc.len[0] > 0 and (orc.head[0], orc.len[0]) != (orc.head[2], orc.len[2])
                orc.copy_sequences([0], [2])
                ref[2] = ref[0]
            orc.consolidate(1, force=(t == 3))  # an early partial fold moves the head
            y = orc.decode(tok)
            ref, y_ref = step(ref, tok)
            for q in (0, 1) if t < t_copy else (0, 1, 2):
                _close(y[q], y_ref[q], 1e-11, f"{kind} step {t} sequence {q}")
            # every sequence's checkpoint, ring and pointers replay to its output
            _close(orc.replay_output(tok, "f64"), y, 1e-11, f"{kind} replay step {t}")
        _close(orc.committed, ref, 1e-11, f"{kind} committed state")
        orc.consolidate(1, force=True)
        _close(orc.ckpt, ref, 1e-11, f"{kind} checkpoint after a forced fold")


def pin_rollback_equals_accepted_prefix():
    """Verify K drafts then accept m equals decoding only the m accepted tokens.

    The pages ("NVIDIA y Princeton aceleran…", paragraph 3) say rejected
    drafts are discarded by moving a buffer pointer, with no state copy per
    draft; the result must equal never having seen the rejected drafts.
    """
    for kind in ("gdn", "kda"):
        r = _rng(51)
        b, H, dk, dv, W, K, R = 3, 2, 6, 4, 16, 4, 12
        S0 = r.standard_normal((b, H, dv, dk))
        spec = om.ReplayOracle(kind, S0, W, scale=0.8)
        plain = om.ReplayOracle(kind, S0, W, scale=0.8)
        for rnd in range(R):
            toks = delta_tokens(r, b, H, dk, dv, K, kind == "kda")
            drafts = {k: np.stack([t[k] for t in toks], axis=1) for k in toks[0]}
            m = r.integers(0, K + 1, size=b)
            spec.consolidate(K)
            o = spec.spec_verify(K, drafts)
            spec.accept(m, K)
            for s in range(b):
                one = om.ReplayOracle(kind, plain.committed[s:s + 1], W, scale=0.8)
                for i in range(m[s]):
                    tok = {k: v[s:s + 1] for k, v in toks[i].items()}
                    y = one.decode(tok)
                    _close(o[s, i], y[0], 1e-11, f"{kind} round {rnd} seq {s} draft {i}")
                plain.committed[s] = one.committed[0]
        spec.consolidate(1, force=True)
        _close(spec.ckpt, plain.committed, 1e-11, f"{kind} checkpoint after rollback")
        assert np.all(spec.status == 0)
    # Mamba-2: the same invariant with its own recurrence
    r = _rng(52)
    b, H, G, P, N, W, K, R = 3, 4, 2, 3, 5, 16, 4, 12
    A, D = -r.uniform(1.0, 16.0, H), r.standard_normal(H)
    h0 = r.standard_normal((b, H, P, N))
    spec = om.ReplayOracle("mamba2", h0, W, A=A, D=D, groups=G)
    plain = om.ReplayOracle("mamba2", h0, W, A=A, D=D, groups=G)
    for rnd in range(R):
        toks = m2_tokens(r, b, H, G, P, N, K)
        drafts = {k: np.stack([t[k] for t in toks], axis=1) for k in toks[0]}
        m = r.integers(0, K + 1, size=b)
        spec.consolidate(K)
        o = spec.spec_verify(K, drafts)
        spec.accept(m, K)
        for s in range(b):
            one = om.ReplayOracle("mamba2", plain.committed[s:s + 1], W, A=A, D=D, groups=G)
            for i in range(m[s]):
                y = one.decode({k: v[s:s + 1] for k, v in toks[i].items()})
                _close(o[s, i], y[0], 1e-11, f"mamba2 round {rnd} seq {s} draft {i}")
            plain.committed[s] = one.committed[0]
    spec.consolidate(1, force=True)
    _close(spec.ckpt, plain.committed, 1e-11, "mamba2 checkpoint after rollback")
    assert np.all(spec.status == 0)


def pin_status_and_refusal():
    """Decoding into a full ring is refused (bit 1, nothing changes); bad accepts set bit 2."""
    toks, outs, orc, _, _ = run_plain_decode("gdn", 3, 3, 61)
    head, ln = orc.head.copy(), orc.len.copy()
    S = orc.committed.copy()
    ring = {k: v.copy() for k, v in orc.ring.items()}
    y = orc.decode(toks[0])
    assert np.all(np.isnan(y)) and np.all(orc.status == om.RING_FULL)
    assert np.array_equal(orc.head, head) and np.array_equal(orc.len, ln)
    assert np.array_equal(orc.committed, S)
    assert all(np.array_equal(ring[k], orc.ring[k]) for k in ring)
    orc.consolidate(1)
    orc.accept(np.array([5, -2]), 4)
    assert np.all(orc.status == om.RING_FULL | om.BAD_ACCEPT)
    assert np.all(orc.len == 0)


def pin_bf16_rounding():
    """Round-to-nearest-even bfloat16 on hand-checked values (worked_examples.json),
    and bit for bit against torch's float32 -> bfloat16 conversion (also
    round to nearest, ties to even) on random values, exact ties of both
    parities, values just either side of a tie, and signed zeros and
    subnormals."""
    import torch

    g = _golden("worked_examples.json")["bf16_rne"]
    _close(om.bf16_rne(np.array(g["in"], np.float32)), g["out"], 0.0, "bf16 RNE")
    r = _rng(57)
    bits = r.integers(0, 0x7F800000, 4000, dtype=np.int64)       # finite, positive
    ties = (bits & ~0xFFFF) | 0x8000                               # halfway cases
    near = np.concatenate([ties - 1, ties + 1])
    sub = r.integers(1, 0x00800000, 200, dtype=np.int64)           # subnormals
    u = np.concatenate([bits, ties, near, sub, [0]]).astype(np.uint32)
    f = np.concatenate([u, u | 0x80000000]).astype(np.uint32).view(np.float32)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float32).numpy()
    got = om.bf16_rne(f).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), "bf16 RNE vs torch"


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
