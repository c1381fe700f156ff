#!/usr/bin/env python
"""Benchmark of the ReplaySSM SSM-layer decode step on B300.

Default workload: a Mamba-2 layer of hybrid-LLM shape, batch 256, H = 128
heads, P = 64, N = 128 (4 MiB FP32 state per sequence), W = 16, BF16 vector
inputs, FP32 checkpoint plus BF16 read copy. One step = consolidate(k_next = 1)
+ replay decode of one token for every sequence, i.e. the whole hot path for
plain decoding. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload mamba2|gdn|kda|gdn_spec] [--read bf16|f32] [--stagger]
                  [--step fused|split]

A Mamba-2 step is one fused call (replayssm_mamba2_fold_decode: a full ring
is folded while its state rows stream past) unless --step split asks for
the two calls consolidate + decode; the delta kinds always take two calls.
By default every sequence starts at the same ring phase, so all of them fold
on the same step (every W-th). --stagger starts sequence s at phase s mod W,
as sequences that joined a continuous batch at different steps are: then
1/W of the batch folds on every step.

Timing: device time with CUDA events on the launching stream, W untimed
warm-up steps first, a barrier and a synchronize on both sides of the K timed
steps, max over ranks. The state (1.5 GiB) is larger than L2, so no flush is
needed between steps. Under torchrun every rank decodes its own batch of 256
sequences (independent shards, no collective on the data path).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SSM-layer decode tokens/s at batch 256 on 1 B300; achieved HBM GB/s vs ~8 TB/s"
UNIT = "tokens/s"

WORKLOADS = {
    "mamba2": dict(kind="mamba2", batch=256, heads=128, dk=128, dv=64, window=16, groups=1),
    "gdn": dict(kind="gdn", batch=256, heads=32, dk=128, dv=128, window=16, groups=1),
    "kda": dict(kind="kda", batch=256, heads=32, dk=128, dv=128, window=16, groups=1),
    # speculative rounds: consolidate(k_next = K) + verify K drafts + accept m
    "gdn_spec": dict(kind="gdn", batch=512, heads=32, dk=128, dv=128, window=16, groups=1, K=4),
}
POOL = 16  # distinct synthetic tokens, cycled through the timed steps

# DRAM bytes (read + write) of one decode call at batch 64 from single-launch
# ncu captures of the same kernels (Mamba-2: stream + prep kernels; GDN: the
# fused kernel; ring length 8); traffic grows in proportion to the batch, so
# it is scaled by batch / 64. Only for the captured kernels.
TRAFFIC_B64 = {
    ("mamba2", "bf16"): 136.526592e6 + 3.470848e6 + 10.205184e6,
    ("gdn", "bf16"): 77.416192e6 + 1.435392e6,
}
# The same for one fused Mamba-2 fold + decode call (coefficient + step
# stream kernels), averaged over 16 consecutive calls of which one folds
# every sequence: a sixteenth of the batch folds per call on average, in
# lockstep or with staggered ring phases alike. Empty until captured for the
# current kernels.
TRAFFIC_B64_FUSED: dict = {}


def traffic_per_call(wl: dict, read: str, fused: bool):
    """DRAM bytes of one decode call at this batch, from the batch-64 captures
    (None for kernels or shapes without one)."""
    table = TRAFFIC_B64_FUSED if fused else TRAFFIC_B64
    key = (wl["kind"], read)
    if key not in table or wl["heads"] != WORKLOADS[wl["kind"]]["heads"]:
        return None
    return round(table[key] * wl["batch"] / 64)


def parse(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4096)
    p.add_argument("--warmup", type=int, default=64)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="mamba2")
    p.add_argument("--read", choices=["bf16", "f32"], default="bf16")
    p.add_argument("--batch", type=int, default=None, help="override the batch size")
    p.add_argument("--step", choices=["fused", "split"], default="fused",
                   help="Mamba-2: one fused fold + decode call per step, or two calls")
    p.add_argument("--stagger", action="store_true",
                   help="start sequence s at ring phase s mod W (continuous batching)")
    p.add_argument("--no-extras", action="store_true",
                   help="time the main loop only (no A/B, e2e, CPU baseline, clocks)")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="budget of the CPU-oracle baseline sample")
    return p.parse_args(argv)


# ------------------------------------------------------------------ config
def decode_config(wl: dict, read: str, world: int, stagger: bool, fused: bool = False) -> dict:
    k, W = wl["kind"], wl["window"]
    rows, cols = ("p", "n") if k == "mamba2" else ("dv", "dk")
    return {
        "workload": f"{k}_decode_b{wl['batch']}_h{wl['heads']}_{rows}{wl['dv']}_"
                    f"{cols}{wl['dk']}_w{W}" + ("_staggered" if stagger else ""),
        "batch_per_gpu": wl["batch"], "heads": wl["heads"], "dk_or_N": wl["dk"],
        "dv_or_P": wl["dv"], "window": W, "read_copy": read, "inputs": "bf16",
        "checkpoint": "f32",
        "step": ("fold_decode: consolidate(k_next=1) + replay decode fused in one call"
                 if fused else "consolidate(k_next=1) + replay decode"),
        "ring_phases": ("staggered: sequence s starts at phase s mod W" if stagger else
                        "lockstep: every sequence at the same phase"),
        "l2": "state larger than L2 (no flush)", "parallelism": f"replicas x{world}",
    }


def spec_config(wl: dict, read: str, world: int) -> dict:
    k, b, H, dk, W, K = (wl[x] for x in ("kind", "batch", "heads", "dk", "window", "K"))
    return {"workload": f"{k}_spec_b{b}_h{H}_d{dk}_w{W}_k{K}", "batch_per_gpu": b,
            "drafts": K, "read_copy": read, "inputs": "bf16", "checkpoint": "f32",
            "step": "consolidate(k_next=K) + spec_verify(K) + accept(m)",
            "l2": "state larger than L2 (no flush)", "parallelism": f"replicas x{world}"}


SPEC_METRIC = ("speculative rounds: accepted tokens/s per SSM layer (verified K drafts per "
               "sequence from one state read, pointer accept)")
SPEC_UNIT = "accepted tokens/s"


# ------------------------------------------------------------- distributed
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (the job ends when its slowest rank does)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ peaks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            # lowest CPU priority and a 200 ms period: the sampler must not
            # delay the host thread that enqueues the timed launches
            self.proc = subprocess.Popen(
                ["nice", "-n", "19", "nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return self
        # nvidia-smi takes a while to start; its start-up must not overlap
        # the timed region, so wait (at most 5 s) for its first sample
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.file.name) > 0:
                break
            time.sleep(0.05)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            reasons.add("no clock samples")
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ our arm
class Layer:
    """One SSM layer's state, token pool and step functions on one GPU."""

    def __init__(self, wl: dict, read: str, device, seed: int = 2, fused: bool = False):
        import numpy as np
        import torch

        import synth
        from recurrent_state_fp32_b300 import api

        self.api, self.torch, self.np = api, torch, np
        self.wl = wl
        k = wl["kind"]
        b, H, dk, dv, W, G = (wl[x] for x in ("batch", "heads", "dk", "dv", "window", "groups"))
        self.dims = api.LayerDims(k, b, H, dk=dk, dv=dv, window=W, groups=G, in_dtype="bf16")
        self.state = api.LayerState(self.dims, device=device, read_copy=(read == "bf16"))
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        self.state.S_ckpt.normal_(0.0, 0.1, generator=gen)
        if self.state.S_read is not None:
            api.refresh_read_copy(self.dims, self.state)
        self.device = device
        dt = lambda a, ty: torch.from_numpy(np.ascontiguousarray(a)).to(device, ty)  # noqa: E731
        self.host_pool, self.pool = [], []
        if k == "mamba2":
            A, D, bias = synth.mamba2_params(seed, H)
            self.A, self.D = dt(A, torch.float32), dt(D, torch.float32)
            for t in range(POOL):
                tok = synth.mamba2_step_inputs(seed, t, b, H, G, dv, dk, bias, "bf16")
                self.host_pool.append(tok)
            names = ("x", "B", "C", "dt")
        else:
            self.A = None
            for t in range(POOL):
                self.host_pool.append(synth.delta_step_inputs(seed, t, b, H, dk, dv, k, "bf16"))
            names = ("q", "k", "v", "alpha", "beta")
        vec = {"x", "B", "C", "q", "k", "v"}
        for tok in self.host_pool:
            self.pool.append({n: dt(tok[n], torch.bfloat16 if n in vec else torch.float32)
                              for n in names})
        self.out = torch.empty((b, H, dv), device=device)
        self.names = names
        self.vec = vec
        self.fused = fused and k == "mamba2"

    # one decode step on device-resident inputs
    def consolidate(self, stream=None):
        self.api.consolidate(self.dims, self.state, self.A, 1, False, stream)

    def decode(self, tok, stream=None):
        a = self.api
        if self.wl["kind"] == "mamba2":
            a.mamba2_decode(self.dims, self.state, self.A, self.D, tok["x"], tok["B"], tok["C"],
                            tok["dt"], self.out, stream)
        else:
            a.gdn_decode(self.dims, self.state, tok["q"], tok["k"], tok["v"], tok["alpha"],
                         tok["beta"], 1.0, self.out, stream)

    def step(self, tok, stream=None):
        """One whole step: the fused call, or consolidate then decode."""
        if self.fused:
            self.api.mamba2_fold_decode(self.dims, self.state, self.A, self.D, tok["x"], tok["B"],
                                        tok["C"], tok["dt"], self.out, stream)
        else:
            self.consolidate(stream)
            self.decode(tok, stream)

    def conventional(self, S, tok, stream=None):
        a = self.api
        if self.wl["kind"] == "mamba2":
            a.conventional_mamba2_step(self.dims, S, self.A, self.D, tok["x"], tok["B"], tok["C"],
                                       tok["dt"], self.out, stream)
        else:
            a.conventional_gdn_step(self.dims, S, tok["q"], tok["k"], tok["v"], tok["alpha"],
                                    tok["beta"], 1.0, self.out, stream)

    def step_launches(self):
        """Kernels of one step: the fused call's two, or consolidate's one
        plus the decode's (two for Mamba-2, one for the delta kinds)."""
        if self.fused:
            return 2
        return 1 + (2 if self.wl["kind"] == "mamba2" else 1)

    def decode_kernels(self):
        if self.fused:
            return "mamba2_step_coef_kernel + mamba2_step_stream_kernel (one fused call)"
        if self.wl["kind"] == "mamba2":
            return "mamba2_prep_kernel + stream_kernel (one decode call)"
        return "delta_fused_kernel (one decode call)"

    # ------------------------------------------------ algorithmic bytes
    def token_bytes(self):
        """Bytes of one token's inputs for the whole batch (as read, and as ring-written)."""
        return sum(t.numel() * t.element_size() for t in self.pool[0].values())

    def ring_entry_bytes(self):
        """Bytes of one ring entry for the whole batch that the replay reads back."""
        wl, b = self.wl, self.wl["batch"]
        H, dk, dv, G = wl["heads"], wl["dk"], wl["dv"], wl["groups"]
        if wl["kind"] == "mamba2":
            return b * (H * dv * 2 + G * dk * 2 + H * 4)          # x, B, dt
        gate = H * 4 if wl["kind"] == "gdn" else H * dk * 4
        return b * (H * dk * 2 + H * dv * 2 + gate + H * 4)       # k, v, alpha, beta

    def state_elems(self):
        wl = self.wl
        return wl["batch"] * wl["heads"] * wl["dv"] * wl["dk"]

    def decode_bytes(self, n_prior):
        """Algorithmic bytes of one decode launch with n_prior committed entries.

        Read copy (or FP32 checkpoint) once + token inputs read + the token
        written to the ring + the n_prior buffered entries read + the output.
        """
        ts = 2 if self.state.S_read is not None else 4
        out = self.out.numel() * 4
        return self.state_elems() * ts + 2 * self.token_bytes() + n_prior * self.ring_entry_bytes() + out

    def fold_bytes(self, n, frac=1.0):
        """Algorithmic bytes of one consolidate that folds a fraction frac of the
        sequences, n entries each (on average)."""
        rd = 2 if self.state.S_read is not None else 0
        return frac * (self.state_elems() * (4 + 4 + rd) + n * self.ring_entry_bytes())

    def account(self, lens, steps):
        """Algorithmic bytes (decode, consolidate) of `steps` steps of
        consolidate(k_next = 1) + decode from per-sequence ring lengths `lens`.
        Both byte counts are linear in the entries, so batch means suffice."""
        lens = self.np.array(lens, dtype=self.np.int64)
        W, b = self.wl["window"], len(lens)
        ts = 2 if self.state.S_read is not None else 4
        dec = fold = 0.0
        for _ in range(steps):
            f = lens + 1 > W
            if f.any():
                fold += self.fold_bytes(lens[f].mean(), f.sum() / b)
                lens[f] = 0
                if self.fused:  # a folded sequence's output comes from its new rows
                    dec -= f.sum() / b * self.state_elems() * ts
            dec += self.decode_bytes(lens.mean())
            lens += 1
        return dec, fold

    def fold_steps(self, lens, steps):
        """For each of `steps` steps from ring lengths `lens`: whether the
        step's consolidate(k_next = 1) folds any sequence."""
        lens = self.np.array(lens, dtype=self.np.int64)
        W, out = self.wl["window"], []
        for _ in range(steps):
            f = lens + 1 > W
            out.append(bool(f.any()))
            lens[f] = 0
            lens += 1
        return out

    def stagger(self):
        """Puts sequence s at ring phase s mod W: W lockstep steps, before the
        j-th of which the sequences with s mod W == j restart from their
        checkpoint (ring length 0, as a sequence that joins the batch with its
        prefill state does). Afterwards their lengths are W, W - 1, ..., 1."""
        torch = self.torch
        W = self.wl["window"]
        phase = torch.arange(self.wl["batch"], device=self.device) % W
        for j in range(W):
            self.state.ring_len[phase == j] = 0
            self.step(self.pool[j % POOL])

    def conventional_bytes(self):
        return self.state_elems() * 8 + self.token_bytes() + self.out.numel() * 4


def run_ours(args, rank, local_rank, world):
    import torch

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = dict(WORKLOADS[args.workload])
    if args.batch:
        wl["batch"] = args.batch
    W = wl["window"]
    layer = Layer(wl, args.read, device, fused=args.step == "fused")
    stream = torch.cuda.current_stream(device)
    K, Wm = args.steps, args.warmup

    # The clock sampler starts first (its start-up takes the host for a
    # while); the A/B and end-to-end loops then run, and the warm-up steps
    # and the timed steps follow them directly, so the GPU does not idle
    # (and drop its clocks) just before the timed region.
    clocks = ClockSampler(local_rank) if not args.no_extras else None
    if clocks:
        clocks.__enter__()
    extras = {}
    if not args.no_extras:
        extras["ab"] = run_ab(layer, K, Wm, stream, world)
        extras["e2e"] = run_e2e(layer, args, stream, world)

    # warm-up
    for i in range(Wm):
        layer.step(layer.pool[i % POOL])
    if args.stagger:
        layer.stagger()
    torch.cuda.synchronize()
    lens0 = layer.state.ring_len.cpu().numpy()

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    start, end = ev(), ev()
    d0 = [ev() for _ in range(K)]
    d1 = [ev() for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(K):
        # events around the decode call (the fused call also holds the folds)
        if layer.fused:
            d0[i].record(stream)
            layer.step(layer.pool[i % POOL])
        else:
            layer.consolidate()
            d0[i].record(stream)
            layer.decode(layer.pool[i % POOL])
        d1[i].record(stream)
    end.record(stream)
    end.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.__exit__(None, None, None)
    ms = max_over_ranks(start.elapsed_time(end), world)
    dec_ms = [d0[i].elapsed_time(d1[i]) for i in range(K)]
    gaps_us = [1e3 * d1[i].elapsed_time(d0[i + 1]) for i in range(K - 1)]
    bad = int(layer.state.status.ne(0).sum().item())
    if bad:
        print(f"warning: {bad} sequences report device status bits "
              f"{sorted(set(layer.state.status.tolist()))}", file=sys.stderr)

    # algorithmic bytes of the timed region
    dec_bytes, fold_bytes = layer.account(lens0, K)
    peak, peak_kind = measured_peaks()
    dec_s = sum(dec_ms) / 1e3
    call_bytes = dec_bytes + (fold_bytes if layer.fused else 0)
    achieved = call_bytes / dec_s / 1e9
    tokens = wl["batch"] * K * world
    value = tokens / (ms / 1e3)
    step_gbs = (dec_bytes + fold_bytes) / (ms / 1e3) / 1e9

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded; no weights or datasets)",
        "config": decode_config(wl, args.read, world, args.stagger, layer.fused),
        "step_hbm_gbs": round(step_gbs, 1),
        "roofline": {
            "kernel": layer.decode_kernels(), "bound": "hbm", "achieved": round(achieved, 1),
            "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic_per_call(wl, args.read, layer.fused),
            "bytes_per_launch": int(call_bytes / K),
            "avg_launch_us": round(1e3 * sum(dec_ms) / K, 3),
        },
        "gpu_launches": K * layer.step_launches(),
        "device_status_ok": bad == 0,
        "calls": call_stats(dec_ms, gaps_us, layer.fold_steps(lens0, K)),
    }
    if clocks:
        res["clocks"] = clocks.summary()
    res.update(extras)
    if not args.no_extras and rank == 0:
        res["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    return res


def call_stats(dec_ms, gaps_us, folds):
    """Per-call device times of the timed steps: the median of the calls that
    fold nothing, the mean of those that fold, and the median idle gap on the
    device between one call's end and the next call's start (host-bound
    stretches show up there)."""
    plain = [1e3 * t for t, f in zip(dec_ms, folds) if not f]
    fold = [1e3 * t for t, f in zip(dec_ms, folds) if f]
    return {"plain_call_us_median": round(statistics.median(plain), 2) if plain else None,
            "fold_call_us": round(sum(fold) / len(fold), 2) if fold else None,
            "fold_calls": len(fold),
            "host_gap_us_median": round(statistics.median(gaps_us), 2) if gaps_us else None}


def run_ab(layer, K, Wm, stream, world):
    """In-library conventional read-modify-write step on the same workload."""
    import torch

    S = layer.state.S_ckpt.clone()
    for i in range(Wm):
        layer.conventional(S, layer.pool[i % POOL])
    Kc = max(16, K // 4)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for i in range(Kc):
        layer.conventional(S, layer.pool[i % POOL])
    b.record(stream)
    b.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world)
    del S
    torch.cuda.empty_cache()
    tok_s = layer.wl["batch"] * Kc * world / (ms / 1e3)
    return {"conventional_tokens_per_s": round(tok_s, 1),
            "conventional_ms_per_step": round(ms / Kc, 5),
            "conventional_hbm_gbs": round(layer.conventional_bytes() / (ms / Kc / 1e3) / 1e9, 1),
            "conventional_bytes_per_step": layer.conventional_bytes(), "steps": Kc}


def run_e2e(layer, args, stream, world):
    """The same step through the public API with host buffers: every step copies
    its inputs from pinned host memory and reads the output back."""
    import torch

    host = [{n: t.cpu().pin_memory() for n, t in tok.items()} for tok in layer.pool]
    stage = {n: torch.empty_like(t) for n, t in layer.pool[0].items()}
    y_host = torch.empty(layer.out.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host[0].values())
    d2h = y_host.numel() * 4
    K = max(16, args.steps // 4)

    def step(i):
        for n, t in host[i % POOL].items():
            stage[n].copy_(t, non_blocking=True)
        layer.step(stage)
        y_host.copy_(layer.out, non_blocking=True)

    for i in range(8):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(K):
        step(i)
    b.record(stream)
    b.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world)
    return {"value": round(layer.wl["batch"] * K * world / (ms / 1e3), 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K}


# ------------------------------------------------------ speculative rounds
def run_spec(args, rank, local_rank, world):
    """Speculative decoding rounds on a delta layer: consolidate(k_next = K),
    verify K drafts from one read of the state, accept m drafts by moving the
    ring pointer (m drawn U{0..K} per sequence and round). The A/B runs the
    conventional baseline on the same drafts: verify with a state snapshot per
    draft, then accept by copying snapshot m - 1 into the state."""
    import numpy as np
    import torch

    import synth
    from recurrent_state_fp32_b300 import api

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = dict(WORKLOADS[args.workload])
    if args.batch:
        wl["batch"] = args.batch
    b, H, dk, dv, W, K, kind = (wl[x] for x in ("batch", "heads", "dk", "dv", "window", "K", "kind"))
    dims = api.LayerDims(kind, b, H, dk=dk, dv=dv, window=W, in_dtype="bf16")
    state = api.LayerState(dims, device=device, read_copy=(args.read == "bf16"), max_drafts=K)
    gen = torch.Generator(device=device)
    gen.manual_seed(4)
    state.S_ckpt.normal_(0.0, 0.1, generator=gen)
    if state.S_read is not None:
        api.refresh_read_copy(dims, state)
    seed, rounds_pool = 4, 8
    to = lambda a, ty: torch.from_numpy(np.ascontiguousarray(a)).to(device, ty)  # noqa: E731
    drafts, ms, m_tot = [], [], []
    for r in range(rounds_pool):
        dr = synth.spec_draft_inputs(seed, r, b, K, H, dk, dv, kind, "bf16")
        drafts.append({n: to(v, torch.bfloat16 if n in ("q", "k", "v") else torch.float32)
                       for n, v in dr.items()})
        m = synth.accept_counts(seed, r, b, K)
        ms.append(to(m, torch.int32))
        m_tot.append(int(m.sum()))
    o = torch.empty((b, K, H, dv), device=device)

    def round_(i):
        d = drafts[i % rounds_pool]
        api.consolidate(dims, state, None, K, False)
        api.spec_verify(dims, state, K, d["q"], d["k"], d["v"], d["alpha"], d["beta"], 1.0, o)
        api.accept(dims, state, ms[i % rounds_pool], K)

    Kt, Wm = args.steps, args.warmup
    for i in range(Wm):
        round_(i)
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    a0, a1 = ev(), ev()
    clocks = ClockSampler(local_rank) if not args.no_extras else None
    if clocks:
        clocks.__enter__()
    barrier(world)
    torch.cuda.synchronize()
    a0.record()
    for i in range(Kt):
        round_(Wm + i)
    a1.record()
    a1.synchronize()
    barrier(world)
    if clocks:
        clocks.__exit__(None, None, None)
    ms_tot = max_over_ranks(a0.elapsed_time(a1), world)
    accepted = sum(m_tot[(Wm + i) % rounds_pool] for i in range(Kt)) * world
    bad = int(state.status.ne(0).sum().item())
    res = {
        "metric": SPEC_METRIC,
        "value": round(accepted / (ms_tot / 1e3), 1), "unit": SPEC_UNIT,
        "n_gpus": world, "steps": Kt, "warmup": Wm, "ms_per_step": round(ms_tot / Kt, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; no weights or datasets)",
        "config": spec_config(wl, args.read, world),
        "verified_tokens_per_s": round(b * K * Kt * world / (ms_tot / 1e3), 1),
        "gpu_launches": Kt * 3, "device_status_ok": bad == 0,
    }
    if clocks:
        res["clocks"] = clocks.summary()
    if not args.no_extras:
        # the conventional baseline: snapshots per draft, accept by copy
        S = state.S_ckpt.clone()
        snaps = torch.empty((b, K, H, dv, dk), device=device)
        st = torch.zeros(b, dtype=torch.int32, device=device)

        def conv_round(i):
            d = drafts[i % rounds_pool]
            api.conventional_gdn_verify(dims, S, K, d["q"], d["k"], d["v"], d["alpha"],
                                        d["beta"], 1.0, snaps, o)
            api.conventional_accept(dims, S, snaps, ms[i % rounds_pool], K, st)

        for i in range(4):
            conv_round(i)
        Kc = max(8, Kt // 4)
        c0, c1 = ev(), ev()
        torch.cuda.synchronize()
        c0.record()
        for i in range(Kc):
            conv_round(i)
        c1.record()
        c1.synchronize()
        cms = max_over_ranks(c0.elapsed_time(c1), world)
        acc_c = sum(m_tot[i % rounds_pool] for i in range(Kc)) * world
        res["ab"] = {"conventional_accepted_tokens_per_s": round(acc_c / (cms / 1e3), 1),
                     "conventional_ms_per_round": round(cms / Kc, 5), "rounds": Kc,
                     # verify: read S, write K snapshots; accept: copy one snapshot
                     # for every sequence with m > 0
                     "conventional_bytes_per_round":
                         int(b * H * dv * dk * 4 * (1 + K) +
                             np.mean([int((mm > 0).sum().item()) for mm in ms]) * H * dv * dk * 8)}
        del S, snaps
        torch.cuda.empty_cache()
    return res


# --------------------------------------------------------- oracle timing
def oracle_sample(wl: dict, heads: int, seed: int = 2):
    """A one-sequence, `heads`-head slice of the workload for the CPU oracle."""
    import numpy as np

    import synth
    from oracle.method import ReplayOracle

    k, W, dk, dv = wl["kind"], wl["window"], wl["dk"], wl["dv"]
    H = wl["heads"]
    if k == "mamba2":
        A, D, bias = synth.mamba2_params(seed, H)
        S0 = synth.mamba2_initial_state(seed, 1, heads, dv, dk)
        orc = ReplayOracle(k, S0, W, A=A[:heads], D=D[:heads])
        toks = []
        for t in range(POOL):
            tok = synth.mamba2_step_inputs(seed, t, 1, H, 1, dv, dk, bias, "bf16")
            toks.append({"x": tok["x"][:, :heads], "B": tok["B"], "C": tok["C"],
                         "dt": tok["dt"][:, :heads]})
    else:
        S0 = synth.delta_initial_state(seed, 1, heads, dv, dk)
        orc = ReplayOracle(k, S0, W)
        toks = []
        for t in range(POOL):
            tok = synth.delta_step_inputs(seed, t, 1, H, dk, dv, k, "bf16")
            toks.append({n: v[:, :heads] for n, v in tok.items()})
    return orc, toks, np


def _single_thread():
    try:
        from threadpoolctl import threadpool_limits

        return threadpool_limits(limits=1)
    except ImportError:  # pragma: no cover
        import contextlib

        return contextlib.nullcontext()


def cpu_baseline(wl: dict, seconds: float):
    """The oracle as it stands, single-threaded on the host, on a bounded sample
    (one sequence, all heads) of the same workload; scaled to tokens/s."""
    heads = wl["heads"]
    orc, toks, _ = oracle_sample(wl, heads)
    with _single_thread():
        t0 = time.perf_counter()
        n = 0
        while True:
            orc.consolidate(1)
            orc.decode(toks[n % POOL])
            n += 1
            if time.perf_counter() - t0 > seconds and n % wl["window"] == 0:
                break
        dt = time.perf_counter() - t0
    return {"value": round(n / dt, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"1 sequence x {heads} heads, {n} consecutive decode steps "
                      f"(consolidate + decode), float64 numpy, {dt:.1f} s"}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: K timed steps (after W warm-up), each
    a bounded sample of the workload (one sequence, a slice of its heads). For
    a speculative workload a step is one round: consolidate(k_next = K),
    verify K drafts, accept the same m as the GPU arm draws."""
    if rank != 0:
        return None
    wl = dict(WORKLOADS[args.workload])
    if args.batch:
        wl["batch"] = args.batch
    heads = max(1, wl["heads"] // 16)
    frac = heads / wl["heads"]
    spec = "K" in wl
    if spec:
        import synth

        K, seed = wl["K"], 4
        orc, _, np = oracle_sample(wl, heads, seed=seed)
        H, dk, dv, kind = wl["heads"], wl["dk"], wl["dv"], wl["kind"]
        rounds = []
        for r in range(8):
            d = synth.spec_draft_inputs(seed, r, 1, K, H, dk, dv, kind, "bf16")
            m = synth.accept_counts(seed, r, wl["batch"], K)[:1]
            rounds.append(({n: v[:, :, :heads] for n, v in d.items()}, m))

        def step(i):
            d, m = rounds[i % len(rounds)]
            orc.consolidate(K)
            orc.spec_verify(K, d)
            orc.accept(m, K)
            return int(m[0])
    else:
        orc, toks, _ = oracle_sample(wl, heads)

        def step(i):
            orc.consolidate(1)
            orc.decode(toks[i % POOL])
            return 1
    with _single_thread():
        for i in range(args.warmup):
            step(i)
        t0 = time.perf_counter()
        tokens = sum(step(args.warmup + i) for i in range(args.steps))
        dt = time.perf_counter() - t0
    value = tokens * frac / dt
    what = "speculative round" if spec else "step"
    sample = (f"1 sequence x {heads} of {wl['heads']} heads per {what} ({frac:.4f} of a "
              f"layer's work for that sequence), float64 numpy oracle, single thread")
    unit = SPEC_UNIT if spec else UNIT
    return {
        "impl": "reference", "metric": SPEC_METRIC if spec else METRIC,
        "value": round(value, 4), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * dt / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; no weights or datasets)",
        "config": dict(spec_config(wl, args.read, world) if spec else
                       decode_config(wl, args.read, world, args.stagger,
                                     args.step == "fused" and wl["kind"] == "mamba2"),
                       sample=sample),
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse(argv)
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if "K" in WORKLOADS[args.workload]:
        res = run_spec(args, rank, local_rank, world)
    else:
        res = run_ours(args, rank, local_rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
