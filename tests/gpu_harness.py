"""Runs the CUDA path (through the C-ABI binding) and the CPU oracle side by side
on the same seeded inputs, and compares them.

Tolerances (the ones the parity bar states):
  FP32 read path: |gpu - ref| <= 1e-4 + 1e-4 |ref| elementwise.
  BF16 read copy: per output vector, max |gpu - ref| <= 2e-2 * max |ref|.
  Consolidated FP32 checkpoint: 1e-4 + 1e-4 |ref| elementwise.
  Ring slots, head, len, status: bit-exact.
"""

from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import replay as rep
from oracle.method import ReplayOracle
from recurrent_state_fp32_b300 import api

DEV = "cuda"


def spread(batch, n=8):
    """n sequences spread over the batch, first and last included: their units
    fall on the first, middle and last persistent blocks alike."""
    if n <= 1 or batch <= 1:
        return [0]
    return sorted({int(round(i * (batch - 1) / (n - 1))) for i in range(n)})


def dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV, dtype)


def f32_close(gpu, ref, what, atol=1e-4, rtol=1e-4):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, f"{what}: {gpu.shape} vs {ref.shape}"
    err = np.abs(gpu - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, "
                           f"max abs err {err.max():.3e}")
    return float(err.max()) if err.size else 0.0


def bf16_close(gpu, ref, what, rel=2e-2):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, f"{what}: {gpu.shape} vs {ref.shape}"
    if gpu.size == 0:
        return 0.0
    err = np.abs(gpu - ref).max(axis=-1)
    scale = np.abs(ref).max(axis=-1)
    bad = err > rel * scale
    assert not bad.any(), f"{what}: {int(bad.sum())} vectors outside 2e-2, worst {np.max(err / scale):.3e}"
    return float(np.max(err / np.maximum(scale, 1e-30)))


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


class Session:
    """One layer state on the GPU plus its oracle twin on a sample of (seq, head).

    kind: "mamba2", "gdn" or "kda"; wl: synth workload; read: "f32" or "bf16".
    seqs/heads: the sequences and heads the oracle follows (default: all).
    """

    def __init__(self, kind, wl, read="bf16", seqs=None, heads=None, scale=1.0,
                 store_optional=True):
        self.kind, self.wl, self.read, self.scale = kind, wl, read, scale
        b, H = wl.batch, wl.heads
        self.seqs = np.arange(b) if seqs is None else np.asarray(seqs)
        self.heads = np.arange(H) if heads is None else np.asarray(heads)
        if kind == "mamba2":
            self.A, self.D, self.dt_bias = synth.mamba2_params(wl.seed, H)
            S0 = synth.mamba2_initial_state(wl.seed, b, H, wl.P, wl.N)
            self.dims = api.LayerDims("mamba2", b, H, dk=wl.N, dv=wl.P, window=wl.window,
                                      groups=wl.groups, in_dtype=wl.in_dtype)
            if wl.groups > 1 and len(self.heads) != H:
                raise ValueError("head sampling needs groups == 1")
        else:
            S0 = synth.delta_initial_state(wl.seed, b, H, wl.dv, wl.dk)
            self.dims = api.LayerDims(kind, b, H, dk=wl.dk, dv=wl.dv, window=wl.window,
                                      in_dtype=wl.in_dtype)
        self.state = api.LayerState(self.dims, read_copy=(read == "bf16"),
                                    store_optional=store_optional,
                                    max_drafts=max(1, getattr(wl, "K", 1)))
        self.state.set_checkpoint(dev(S0))
        sub = S0[self.seqs][:, self.heads]
        if kind == "mamba2":
            self.dA, self.dD = dev(self.A), dev(self.D)
            self.oracle = ReplayOracle(kind, sub, wl.window, A=self.A[self.heads],
                                       D=self.D[self.heads], groups=wl.groups,
                                       store_optional=store_optional)
        else:
            self.oracle = ReplayOracle(kind, sub, wl.window, scale=scale,
                                       store_optional=store_optional)
        self.vt = self.dims.vec_dtype
        self.worst = 0.0
        self.last_tok = None

    # --------------------------------------------------------------- inputs
    def token(self, t):
        wl = self.wl
        if self.kind == "mamba2":
            return synth.mamba2_step_inputs(wl.seed, t, wl.batch, wl.heads, wl.groups, wl.P,
                                            wl.N, self.dt_bias, wl.in_dtype)
        return synth.delta_step_inputs(wl.seed, t, wl.batch, wl.heads, wl.dk, wl.dv, self.kind,
                                       wl.in_dtype)

    def _sub(self, tok, axis_heads=1):
        out = {}
        for k, v in tok.items():
            v = v[self.seqs]
            if not (self.kind == "mamba2" and k in ("B", "C")):
                v = np.take(v, self.heads, axis=axis_heads)
            out[k] = v
        return out

    def _vec(self, name):
        return name in ("x", "B", "C", "q", "k", "v")

    def _to_dev(self, tok):
        return {k: dev(v, self.vt if self._vec(k) else torch.float32) for k, v in tok.items()}

    # ---------------------------------------------------------------- calls
    def join(self, slots, seed):
        """New sequences take over ``slots``: a fresh seeded checkpoint, ring
        pointers and status zero (the per-sequence initialisation the state
        layout documents); the ring bytes stay. Sampled slots restart in the
        oracle too."""
        wl, st = self.wl, self.state
        slots = np.asarray(slots, np.int64)
        if self.kind == "mamba2":
            S = synth.mamba2_initial_state(seed, len(slots), wl.heads, wl.P, wl.N)
        else:
            S = synth.delta_initial_state(seed, len(slots), wl.heads, wl.dv, wl.dk)
        idx = torch.from_numpy(slots).to(DEV)
        st.S_ckpt[idx] = dev(S)
        for name in ("ring_head", "ring_len", "status"):
            getattr(st, name)[idx] = 0
        if st.S_read is not None:
            api.refresh_read_copy(self.dims, st)
        pos = {int(s): i for i, s in enumerate(self.seqs)}
        mine = [(pos[int(s)], i) for i, s in enumerate(slots) if int(s) in pos]
        if mine:
            o_idx, s_idx = (np.array(v) for v in zip(*mine))
            S32 = S.astype(np.float32)[s_idx][:, self.heads]
            self.oracle.restart(o_idx, S32)

    def fork(self, src, dst):
        """Sequences dst[i] become copies of sequences src[i] (replayssm_copy_sequences
        on the GPU; the oracle copies its own rows). Both lists must be sampled."""
        src, dst = np.asarray(src, np.int32), np.asarray(dst, np.int32)
        api.copy_sequences(self.dims, self.state, dev(src, torch.int32), self.state,
                           dev(dst, torch.int32))
        pos = {int(s): i for i, s in enumerate(self.seqs)}
        self.oracle.copy_sequences([pos[int(s)] for s in src], [pos[int(d)] for d in dst])

    def consolidate(self, k_next=1, force=False):
        api.consolidate(self.dims, self.state, self.dA if self.kind == "mamba2" else None,
                        k_next, force)
        return self.oracle.consolidate(k_next, force)

    def decode(self, t, check=True):
        tok = self.token(t)
        self.last_tok = tok
        g = self._to_dev(tok)
        rows = self.wl.P if self.kind == "mamba2" else self.wl.dv
        y = torch.full((self.wl.batch, self.wl.heads, rows), float("nan"), device=DEV)
        if self.kind == "mamba2":
            api.mamba2_decode(self.dims, self.state, self.dA, self.dD, g["x"], g["B"], g["C"],
                              g["dt"], y)
        else:
            api.gdn_decode(self.dims, self.state, g["q"], g["k"], g["v"], g["alpha"], g["beta"],
                           self.scale, y)
        ref = self.oracle.decode(self._sub(tok))
        if check:
            got = host(y)[self.seqs][:, self.heads]
            self.compare_out(got, ref, f"step {t}")
        return y, ref

    def fold_decode(self, t, check=True):
        """One step through the fused fold + decode call (Mamba-2 or delta);
        the oracle takes the same step as consolidate(k_next=1) then decode."""
        tok = self.token(t)
        self.last_tok = tok
        g = self._to_dev(tok)
        rows = self.wl.P if self.kind == "mamba2" else self.wl.dv
        y = torch.full((self.wl.batch, self.wl.heads, rows), float("nan"), device=DEV)
        if self.kind == "mamba2":
            api.mamba2_fold_decode(self.dims, self.state, self.dA, self.dD, g["x"], g["B"],
                                   g["C"], g["dt"], y)
        else:
            api.gdn_fold_decode(self.dims, self.state, g["q"], g["k"], g["v"], g["alpha"],
                                g["beta"], self.scale, y)
        fold = self.oracle.consolidate(1)
        ref = self.oracle.decode(self._sub(tok))
        if check:
            got = host(y)[self.seqs][:, self.heads]
            self.compare_out(got, ref, f"fused step {t}")
        return y, ref, fold

    def compare_out(self, got, ref, what):
        ok = ~np.isnan(ref).any(axis=-1)
        assert np.array_equal(np.isnan(got).any(axis=-1), ~ok), f"{what}: refused rows differ"
        if self.read == "f32":
            self.worst = max(self.worst, f32_close(got[ok], ref[ok], what))
        else:
            self.worst = max(self.worst, bf16_close(got[ok], ref[ok], what))

    def verify(self, r, K, check=True):
        wl = self.wl
        if self.kind == "mamba2":
            d = synth.mamba2_draft_inputs(wl.seed, r, wl.batch, K, wl.heads, wl.groups, wl.P,
                                          wl.N, self.dt_bias, wl.in_dtype)
            g = self._to_dev(d)
            o = torch.full((wl.batch, K, wl.heads, wl.P), float("nan"), device=DEV)
            api.mamba2_spec_verify(self.dims, self.state, K, self.dA, self.dD, g["x"], g["B"],
                                   g["C"], g["dt"], o)
            sub = {k: v[self.seqs] if k in ("B", "C") else np.take(v[self.seqs], self.heads, axis=2)
                   for k, v in d.items()}
        else:
            d = synth.spec_draft_inputs(wl.seed, r, wl.batch, K, wl.heads, wl.dk, wl.dv,
                                        self.kind, wl.in_dtype)
            g = self._to_dev(d)
            o = torch.full((wl.batch, K, wl.heads, wl.dv), float("nan"), device=DEV)
            api.spec_verify(self.dims, self.state, K, g["q"], g["k"], g["v"], g["alpha"],
                            g["beta"], self.scale, o)
            sub = {k: np.take(v[self.seqs], self.heads, axis=2) for k, v in d.items()}
        ref = self.oracle.spec_verify(K, sub)
        if check:
            got = host(o)[self.seqs][:, :, self.heads]
            self.compare_out(got, ref, f"verify round {r}")
        return o, ref

    def accept(self, m, K):
        api.accept(self.dims, self.state, dev(m, torch.int32), K)
        self.oracle.accept(np.asarray(m)[self.seqs], K)

    # ----------------------------------------------- every unit of a call
    def snapshot(self):
        """Host copies of what the next decode reads: the checkpoint as the
        kernels read it (the read copy, else the FP32 checkpoint), every ring
        field and the ring pointers, for the whole batch."""
        st = self.state
        S = st.S_read if st.S_read is not None else st.S_ckpt
        return {"S": S.cpu(), "ring": {k: v.cpu() for k, v in st.ring.items()},
                "head": st.ring_head.cpu().numpy().astype(np.int64),
                "len": st.ring_len.cpu().numpy().astype(np.int64)}

    def check_all_units(self, snap, tok, out, what, chunk=16):
        """Every (sequence, head) output of the decode that followed ``snap``,
        against the oracle's replay formula evaluated on the GPU's own
        checkpoint copy and ring, the values the kernels read. This reaches
        every unit of every persistent block, whatever the sampled oracle
        follows. The decode must not have folded (len + 1 <= W everywhere)."""
        wl, W = self.wl, self.wl.window
        head, lens = snap["head"], snap["len"]
        assert (lens + 1 <= W).all(), "a folding step: use a plain one"
        out = host(out)
        for lo in range(0, wl.batch, chunk):
            for n in np.unique(lens[lo:lo + chunk]):
                sel = np.arange(lo, min(lo + chunk, wl.batch))
                sel = sel[lens[sel] == n]
                ent = [self._ring_entry(snap, sel, (head[sel] + j) % W) for j in range(n)]
                cur = {k: np.asarray(v)[sel] for k, v in tok.items()}
                Sc = snap["S"][torch.from_numpy(sel)].double().numpy()
                if self.kind == "mamba2":
                    ent.append({k: cur[k] for k in ("x", "B", "dt")})
                    ref = rep.mamba2_replay_output(Sc, ent, cur["C"], self.A, self.D)
                else:
                    ent.append({k: cur[k] for k in ("k", "v", "alpha", "beta")})
                    ref = rep.delta_replay_output(Sc, ent, cur["q"], self.scale)
                f32_close(out[sel], ref, f"{what}: all units, sequences {sel[0]}..{sel[-1]}")

    def _ring_entry(self, snap, sel, slot):
        """Ring entry at per-sequence slots ``slot`` of sequences ``sel``, in
        the oracle's entry layout (float64)."""
        r, rows, n = snap["ring"], torch.from_numpy(sel), np.arange(len(sel))
        slot = np.asarray(slot, np.int64)
        # per-head fields are [b, H, W(d), ...]: pick slot[i] of sequence sel[i]
        per_head = lambda name: r[name][rows].double().numpy()[n, :, slot]  # noqa: E731
        if self.kind == "mamba2":
            return {"x": per_head("x"), "dt": per_head("dt"),
                    "B": r["B"][rows, torch.from_numpy(slot)].double().numpy()}
        return {"k": per_head("k"), "v": per_head("v"), "alpha": per_head("alpha"),
                "beta": per_head("beta")}

    # ------------------------------------------------------------- checks
    def check_pointers(self, what=""):
        st = self.state
        for name, g, o in (("head", st.ring_head, self.oracle.head),
                           ("len", st.ring_len, self.oracle.len),
                           ("status", st.status, self.oracle.status)):
            got = g.cpu().numpy()[self.seqs]
            assert np.array_equal(got, o), f"{what} {name}: gpu {got} oracle {o}"
        assert int(st.sync.abs().sum()) == 0, "arrival counters not back at zero"

    def ring_as_oracle(self, name):
        """A GPU ring field in the oracle's [b, W, ...] layout (sampled seqs/heads)."""
        g = host(self.state.ring[name])[self.seqs]
        if self.kind == "mamba2" and name in ("B", "C"):
            return g                                    # [b, W, G, N]
        g = np.take(g, self.heads, axis=1)              # [b, Hs, W(d), ...]
        g = g[:, :, :self.wl.window]                    # drop the scalar-row padding
        return np.swapaxes(g, 1, 2)                     # [b, W, Hs, ...]

    def check_ring(self, what=""):
        for name, ref in self.oracle.ring.items():
            g = self.ring_as_oracle(name)
            assert np.array_equal(bits(g), bits(ref)), f"{what} ring field {name} differs"

    def check_checkpoint(self, what=""):
        got = host(self.state.S_ckpt)[self.seqs][:, self.heads]
        f32_close(got, self.oracle.ckpt, f"{what} checkpoint")
        if self.state.S_read is not None:
            rd = self.state.S_read.view(torch.int16)
            want = self.state.S_ckpt.to(torch.bfloat16).view(torch.int16)
            assert torch.equal(rd, want), f"{what} read copy is not bf16_rne(checkpoint)"
