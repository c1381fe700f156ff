"""Ring / pointer model of the ReplaySSM decode method (oracle; tests only).

State per sequence, as described on the pages ("ReplaySSM: o ganho aparece
na carga concorrente…", introduction; "NVIDIA y Princeton aceleran modelos
híbridos…", paragraphs 2 to 4):

* a checkpoint (the recurrence state at position c),
* a ring of the last W token inputs after c (W = 16 on the pages, section
  "O que muda para quem desenvolve"),
* ``head`` (slot of the oldest entry after c) and ``len`` (committed entries).

Semantics restated here (the pages fix the mechanism, not these details; the
readings are listed with their reasons in the design notes):

* append: entry i of a call goes to slot (head + len + i) mod W; a decode
  commits it (len += 1); speculative drafts are written but not committed.
* consolidate(k_next, force): a sequence folds when len + k_next > W, or when
  force is set and len > 0. Folding moves the checkpoint to the committed
  position (head += len mod W, len = 0). Folding only when the buffer would
  overflow follows paragraph 2 of "NVIDIA y Princeton aceleran modelos
  híbridos…".
* accept(m): len += m for 0 <= m <= K and len + m <= W, else a status bit;
  nothing else moves (paragraph 3: rollback by a pointer, no per-draft copy).
* outputs are those of conventional decoding (section "Cuidados e limites"),
  so the oracle carries the exact float64 conventional state alongside.

Status bits: 1 = ring would overflow (decode or verify refused),
2 = accept count out of range. Refused sequences are left untouched.
"""

from __future__ import annotations

import numpy as np

from . import recurrences as rec
from . import replay as rep

RING_FULL = 1
BAD_ACCEPT = 2


def bf16_rne(a: np.ndarray) -> np.ndarray:
    """Round to float32 first, then to the nearest bfloat16 (ties to even); float64 out."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.int64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    return (u & 0xFFFFFFFF).astype(np.uint32).view(np.float32).reshape(f.shape).astype(np.float64)


def _ring_fields(kind: str, heads: int, rows: int, cols: int, groups: int,
                 store_optional: bool):
    """Per-entry shapes of the ring fields (rows = P or d_v, cols = N or d_k)."""
    if kind == "mamba2":
        f = {"x": (heads, rows), "B": (groups, cols), "dt": (heads,)}
        if store_optional:
            f["C"] = (groups, cols)
    else:
        f = {"k": (heads, cols), "v": (heads, rows),
             "alpha": (heads,) if kind == "gdn" else (heads, cols), "beta": (heads,)}
        if store_optional:
            f["q"] = (heads, cols)
    return f


class ReplayOracle:
    """Float64 model of one SSM layer's decode state for a batch of sequences.

    kind: "mamba2", "gdn" or "kda". S0: initial checkpoint [b,H,rows,cols]
    (Mamba-2 h as [b,H,P,N], delta S as [b,H,d_v,d_k]). For Mamba-2 pass A, D
    [H] and the number of B/C groups.
    """

    def __init__(self, kind, S0, window, *, A=None, D=None, groups=1, scale=1.0,
                 store_optional=True):
        if kind not in ("mamba2", "gdn", "kda"):
            raise ValueError(kind)
        self.kind = kind
        self.W = int(window)
        S0 = np.asarray(S0, dtype=np.float64)
        self.batch, self.heads, self.rows, self.cols = S0.shape
        self.A = None if A is None else np.asarray(A, dtype=np.float64)
        self.D = None if D is None else np.asarray(D, dtype=np.float64)
        self.groups = groups
        self.scale = float(scale)
        self.committed = S0.copy()   # exact state after every committed token
        self.ckpt = S0.copy()        # exact state at the checkpoint position c
        b = self.batch
        self.head = np.zeros(b, np.int32)
        self.len = np.zeros(b, np.int32)
        self.status = np.zeros(b, np.int32)
        self.fields = _ring_fields(kind, self.heads, self.rows, self.cols, groups, store_optional)
        self.ring = {k: np.zeros((b, self.W) + s, np.float32) for k, s in self.fields.items()}
        self._drafts = None          # per-draft states of the last verify
        self._verified = None        # sequences whose last verify was accepted

    # ------------------------------------------------------------ helpers
    def _step(self, S, tok):
        if self.kind == "mamba2":
            return rec.mamba2_step(S, tok["x"], tok["B"], tok["C"], tok["dt"], self.A, self.D)
        return rec.delta_step(S, tok["q"], tok["k"], tok["v"], tok["alpha"], tok["beta"],
                              self.scale)

    def _write(self, mask, slot, tok):
        idx = np.nonzero(mask)[0]
        for name in self.fields:
            self.ring[name][idx, slot[idx]] = np.asarray(tok[name], np.float32)[idx]

    def entries(self, seq: int, count: int | None = None):
        """Committed ring entries of one sequence, oldest first (dicts of float64)."""
        n = int(self.len[seq]) if count is None else count
        out = []
        for i in range(n):
            s = (int(self.head[seq]) + i) % self.W
            out.append({k: self.ring[k][seq, s].astype(np.float64) for k in self.fields})
        return out

    def read_copy(self, precision: str = "f32") -> np.ndarray:
        """The checkpoint as read for outputs: exact ("f64"), float32, or bfloat16 (RNE)."""
        if precision == "bf16":
            return bf16_rne(self.ckpt)
        if precision == "f32":
            return self.ckpt.astype(np.float32).astype(np.float64)
        if precision == "f64":
            return self.ckpt.copy()
        raise ValueError(precision)

    def restart(self, seqs, S0) -> None:
        """New sequences take over the slots ``seqs`` (continuous batching).

        Each gets its own checkpoint S0[i] (also its committed state) and the
        initial pointers and status, zero; the ring bytes stay as they are and
        are overwritten as the new sequence appends. S0: [len(seqs),H,rows,cols].
        """
        seqs = np.asarray(seqs, np.int64)
        S0 = np.asarray(S0, dtype=np.float64)
        self.committed[seqs] = S0
        self.ckpt[seqs] = S0
        self.head[seqs] = 0
        self.len[seqs] = 0
        self.status[seqs] = 0

    def copy_sequences(self, src, dst) -> None:
        """Sequence dst[i] becomes a copy of sequence src[i]: checkpoint,
        committed state, ring pointers, status and every ring slot.

        A sequence is fully described by its checkpoint, its ring and its
        pointers ("NVIDIA y Princeton aceleran…", paragraph 2), so a copy
        resumes where its source stands without replaying history (the
        prefix-cache and continuous-batching setting of "NVIDIA présente
        ReplaySSM…", "D'où vient le problème de l'état"). All sources are
        read before any destination is written.
        """
        src = np.asarray(src, np.int64)
        dst = np.asarray(dst, np.int64)
        for arr in (self.committed, self.ckpt, self.head, self.len, self.status,
                    *self.ring.values()):
            arr[dst] = arr[src].copy()

    # ---------------------------------------------------------- the calls
    def consolidate(self, k_next: int = 1, force: bool = False) -> np.ndarray:
        """Fold where len + k_next > W (or force and len > 0); returns the fold mask."""
        fold = (self.len + k_next > self.W) | (bool(force) & (self.len > 0))
        self.ckpt[fold] = self.committed[fold]
        self.head[fold] = (self.head[fold] + self.len[fold]) % self.W
        self.len[fold] = 0
        return fold

    def decode(self, tok) -> np.ndarray:
        """Append one token per sequence and return the conventional output.

        Sequences whose ring is full get status bit RING_FULL, no change, and
        NaN outputs (the kernels leave their outputs untouched).
        """
        ok = self.len + 1 <= self.W
        self.status[~ok] |= RING_FULL
        self._write(ok, (self.head + self.len) % self.W, tok)
        S_new, y = self._step(self.committed, tok)
        self.committed[ok] = S_new[ok]
        self.len[ok] += 1
        y[~ok] = np.nan
        return y

    def replay_output(self, tok, precision: str = "f32") -> np.ndarray:
        """Output of the current (already appended) token by the replay formula.

        Uses the checkpoint read copy at the given precision; this is the
        output the method computes with a low-precision read copy. Call right
        after ``decode`` with the same token.
        """
        Sc = self.read_copy(precision)
        out = np.empty((self.batch, self.heads, self.rows))
        for s in range(self.batch):
            ent = [{k: v[None] for k, v in e.items()} for e in self.entries(s)]
            if self.kind == "mamba2":
                out[s] = rep.mamba2_replay_output(Sc[s:s + 1], ent,
                                                  np.asarray(tok["C"])[s:s + 1],
                                                  self.A, self.D)[0]
            else:
                out[s] = rep.delta_replay_output(Sc[s:s + 1], ent,
                                                 np.asarray(tok["q"])[s:s + 1], self.scale)[0]
        return out

    def spec_verify(self, K: int, drafts) -> np.ndarray:
        """Write K drafts per sequence after the committed entries; outputs [b,K,H,rows].

        Draft i sees the committed entries and drafts 0..i. Nothing is
        committed. Sequences with len + K > W are refused (RING_FULL, NaN).
        Any layer kind: the pointer rollback applies to every SSM layer type
        the pages name ("NVIDIA y Princeton aceleran…", paragraph 3;
        "NVIDIA présente ReplaySSM…", "Pourquoi les hybrides sont devenus la
        norme").
        """
        ok = self.len + K <= self.W
        self.status[~ok] |= RING_FULL
        outs, states = [], []
        S = self.committed
        for i in range(K):
            tok = {k: np.asarray(v)[:, i] for k, v in drafts.items()}
            self._write(ok, (self.head + self.len + i) % self.W, tok)
            S, o = self._step(S, tok)
            outs.append(o)
            states.append(S)
        out = np.stack(outs, axis=1)
        out[~ok] = np.nan
        self._drafts = states
        self._verified = ok
        return out

    def accept(self, m, K: int) -> None:
        """Commit the first m[s] drafts of each sequence by moving its pointer."""
        m = np.asarray(m, np.int64)
        bad = (m < 0) | (m > K) | (self.len + m > self.W)
        self.status[bad] |= BAD_ACCEPT
        good = ~bad
        verified = self._verified if self._verified is not None else np.zeros_like(bad)
        if np.any(good & (m > 0) & ~verified):
            raise ValueError("accept of drafts that were never verified")
        for s in np.nonzero(good & (m > 0))[0]:
            self.committed[s] = self._drafts[m[s] - 1][s]
        self.len[good] += m[good].astype(np.int32)
