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

# DRAM bytes (read + write) of one split-step decode call at batch 64 from
# ncu captures of the same kernels (Mamba-2: prep + stream kernels; GDN: the
# decode kernel; ring length 8); traffic grows in proportion to the batch, so
# it is scaled by batch / 64. Only for the captured kernels.
TRAFFIC_B64 = {
    ("mamba2", "bf16"): 136.523008e6 + 0.763136e6 + 10.210816e6,
    ("gdn", "bf16"): 77.419264e6 + 1.037824e6,
}
# The same for one fused fold + decode call (Mamba-2: coefficient + step
# stream kernels; GDN/KDA: decode grid + fold grid), averaged over a 16-call
# cycle in which one call folds every sequence: a plain call (Mamba-2 at ring
# length 5, GDN/KDA at 8) and the folding call, captured at batch 64,
# weighted 15 : 1. A sixteenth of the batch folds per call on
# average, in lockstep or with staggered ring phases alike.
TRAFFIC_B64_FUSED = {
    ("mamba2", "bf16"): (15 * (0.756736e6 + 141.772032e6 + 3.569920e6)
                         + (0.940544e6 + 288.052224e6 + 345.972224e6)) / 16,
    # decode grid + fold grid; plain call at ring length 8, and the folding call
    ("gdn", "bf16"): (15 * (77.420032e6 + 1.021184e6 + 0.052736e6)
                      + (0.068608e6 + 152.920832e6 + 140.507648e6)) / 16,
    ("kda", "bf16"): (15 * (86.726656e6 + 1.957888e6 + 0.051200e6)
                      + (0.070400e6 + 170.641920e6 + 141.317632e6)) / 16,
}


# Captures whose kernels changed afterwards. Their figures are no longer
# reported as the call's traffic; the record carries them beside it, with
# the change, until the kernels are captured again.
_DECODE_CONFIG_CHANGE = ("the decode grid's launch configuration changed after this capture "
                         "(two consumer warps per group and 7 prep warps instead of one and 8); "
                         "the kernel code and the bytes each unit moves did not")
TRAFFIC_STALE = {
    ("mamba2", "bf16", True): ("the step stream kernel's block-end arrivals lost their fence after "
                               "this capture; no memory access of the kernel changed"),
    ("gdn", "bf16", True): _DECODE_CONFIG_CHANGE,
    ("kda", "bf16", True): _DECODE_CONFIG_CHANGE,
    ("gdn", "bf16", False): _DECODE_CONFIG_CHANGE,
}


def traffic_per_call(wl: dict, read: str, fused: bool):
    """DRAM bytes of one decode call at this batch from the batch-64 captures,
    as the roofline record's keys: {"traffic": bytes} for a kernel unchanged
    since its capture; {"traffic": None, "traffic_last_capture": {...}} for
    one changed since; {"traffic": None} without a capture."""
    table = TRAFFIC_B64_FUSED if fused else TRAFFIC_B64
    key = (wl["kind"], read)
    if key not in table or wl["heads"] != WORKLOADS[wl["kind"]]["heads"]:
        return {"traffic": None}
    t = round(table[key] * wl["batch"] / 64)
    stale = TRAFFIC_STALE.get(key + (fused,))
    if stale:
        return {"traffic": None, "traffic_last_capture": {"bytes": t, "changed_since": stale}}
    return {"traffic": t}


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

    def __init__(self, wl: dict, read: str, device, seed: int = 2, fused: bool = False,
                 share: "Layer | None" = None):
        """share: another layer of the same workload whose token pool (and
        Mamba-2 A, D) this one reuses; only the state is new."""
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
        self.fused = fused
        if share is not None:
            for name in ("host_pool", "pool", "A", "D", "out", "names", "vec"):
                setattr(self, name, getattr(share, name, None))
            return
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
        if self.fused and self.wl["kind"] == "mamba2":
            self.api.mamba2_fold_decode(self.dims, self.state, self.A, self.D, tok["x"], tok["B"],
                                        tok["C"], tok["dt"], self.out, stream)
        elif self.fused:
            self.api.gdn_fold_decode(self.dims, self.state, tok["q"], tok["k"], tok["v"],
                                     tok["alpha"], tok["beta"], 1.0, self.out, stream)
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
        if self.fused and self.wl["kind"] == "mamba2":
            return "mamba2_step_coef_kernel + mamba2_step_stream_kernel (one fused call)"
        if self.fused:
            return "delta_fused_kernel + delta_fold_stream_kernel (one fused call)"
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


def time_steps(layer, K, Wm, stream, world, stagger=False):
    """W untimed warm-up steps, then K timed steps bracketed by a barrier and a
    synchronize, with events around every decode call. Returns the step-loop
    milliseconds (max over ranks), per-call milliseconds, the device gaps
    between calls (us), the ring lengths before the timed steps and the
    number of sequences with device status bits."""
    import torch

    for i in range(Wm):
        layer.step(layer.pool[i % POOL])
    if stagger:
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
    ms = max_over_ranks(start.elapsed_time(end), world)
    dec_ms = [d0[i].elapsed_time(d1[i]) for i in range(K)]
    gaps_us = [1e3 * d1[i].elapsed_time(d0[i + 1]) for i in range(K - 1)]
    bad = int(layer.state.status.ne(0).sum().item())
    if bad:
        print(f"warning: {bad} sequences report device status bits "
              f"{sorted(set(layer.state.status.tolist()))}", file=sys.stderr)
    return ms, dec_ms, gaps_us, lens0, bad


def decode_record(layer, read, K, Wm, stream, world, stagger=False):
    """Timed steps of one layer: tokens/s, the decode call's roofline, per-call
    times. Keys of the JSON line (metric header excluded)."""
    wl = layer.wl
    ms, dec_ms, gaps_us, lens0, bad = time_steps(layer, K, Wm, stream, world, stagger)
    # algorithmic bytes of the timed region
    dec_bytes, fold_bytes = layer.account(lens0, K)
    peak, peak_kind = measured_peaks()
    dec_s = sum(dec_ms) / 1e3
    call_bytes = dec_bytes + (fold_bytes if layer.fused else 0)
    achieved = call_bytes / dec_s / 1e9
    tokens = wl["batch"] * K * world
    return {
        "value": round(tokens / (ms / 1e3), 1), "ms_per_step": round(ms / K, 5),
        "config": decode_config(wl, read, world, stagger, layer.fused),
        "step_hbm_gbs": round((dec_bytes + fold_bytes) / (ms / 1e3) / 1e9, 1),
        "roofline": {
            "kernel": layer.decode_kernels(), "bound": "hbm", "achieved": round(achieved, 1),
            "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            **traffic_per_call(wl, read, layer.fused),
            "bytes_per_launch": int(call_bytes / K),
            "avg_launch_us": round(1e3 * sum(dec_ms) / K, 3),
        },
        "gpu_launches": K * layer.step_launches(),
        "device_status_ok": bad == 0,
        "calls": call_stats(dec_ms, gaps_us, layer.fold_steps(lens0, K), wl["window"],
                            wl["batch"] * world),
    }


def run_ours(args, rank, local_rank, world):
    import torch

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = dict(WORKLOADS[args.workload])
    if args.batch:
        wl["batch"] = args.batch
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
    rec = decode_record(layer, args.read, K, Wm, stream, world, args.stagger)
    res = {"metric": METRIC, "value": rec.pop("value"), "unit": UNIT, "n_gpus": world,
           "steps": K, "warmup": Wm, "ms_per_step": rec.pop("ms_per_step"),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f32", "data": "synthetic (seeded; no weights or datasets)"}
    res.update(rec)
    res.update(extras)
    if not args.no_extras and args.workload == "mamba2" and not args.batch:
        del layer
        torch.cuda.empty_cache()
        res["others"] = other_workloads(args, device, stream, world)
        res["kda_sweep"] = kda_sweep(device, stream, world)
    if clocks:
        clocks.__exit__(None, None, None)
        res["clocks"] = clocks.summary()
    if not args.no_extras and rank == 0:
        res["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    return res


def other_workloads(args, device, stream, world):
    """The headline layer with staggered ring phases (a sixteenth of the batch
    folds in every call, as in continuous batching), the GDN and KDA layers
    (b256) and the GDN speculative rounds (b512, K = 4), measured the same way
    as the headline (the delta layers and the rounds with their conventional
    A/B), so the line carries every workload: {name: record}."""
    import torch

    out = {}
    K, Wm = args.steps, args.warmup
    layer = Layer(dict(WORKLOADS["mamba2"]), args.read, device, fused=args.step == "fused")
    rec = decode_record(layer, args.read, K, Wm, stream, world, stagger=True)
    rec["unit"] = UNIT
    out["mamba2_staggered"] = rec
    del layer
    torch.cuda.empty_cache()
    for name in ("gdn", "kda"):
        layer = Layer(dict(WORKLOADS[name]), args.read, device, fused=args.step == "fused")
        rec = {"ab": run_ab(layer, K, Wm, stream, world)}
        rec.update(decode_record(layer, args.read, K, Wm, stream, world))
        rec["unit"] = UNIT
        out[name] = rec
        del layer
        torch.cuda.empty_cache()
    spec_args = argparse.Namespace(**dict(vars(args), workload="gdn_spec", batch=None))
    rec = spec_rounds(spec_args, device, world)
    out["gdn_spec"] = rec
    torch.cuda.empty_cache()
    return out


def kda_sweep(device, stream, world, steps=256, warm=16):
    """The KDA layer (H32, d_k = d_v = 128, W16) at batch 1, 8, 64, 256 and 512:
    replay with the BF16 read copy and with the FP32 read path, against the
    conventional read-modify-write step, 256 steps each (16 folds). Below
    batch 256 a step goes to the next of L layer instances in turn, L chosen
    so that the instances' state exceeds four times the L2 cache; a row whose
    working set still fits that bound (L capped at 256) says "hot_l2": true.
    Tokens/s count the whole step loop; frac is its algorithmic bytes per
    second against the measured peak."""
    import math

    import torch

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    peak, _ = measured_peaks()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    rows = []
    for b in (1, 8, 64, 256, 512):
        wl = dict(WORKLOADS["kda"], batch=b)
        row = {"batch": b}
        base = None
        for read in ("bf16", "f32"):
            first = Layer(wl, read, device, seed=5, share=base)
            base = base or first
            per = layer_bytes(first)
            n_inst = 1 if per >= 4 * l2 else min(256, math.ceil(4 * l2 / per))
            layers = [first] + [Layer(wl, read, device, seed=5 + i, share=first)
                                for i in range(1, n_inst)]
            for i in range(warm):
                layers[i % n_inst].step(first.pool[i % POOL])
            torch.cuda.synchronize()
            lens0 = [lay.state.ring_len.cpu().numpy() for lay in layers]
            a, e = ev(), ev()
            a.record(stream)
            for i in range(steps):
                layers[i % n_inst].step(first.pool[i % POOL])
            e.record(stream)
            e.synchronize()
            ms = max_over_ranks(a.elapsed_time(e), world)
            nbytes = 0.0
            for j, lay in enumerate(layers):  # steps j, j + L, ... went to instance j
                n_j = len(range(j, steps, n_inst))
                dec, fold = lay.account(lens0[j], n_j)
                nbytes += dec + fold
            row[f"replay_{read}"] = {
                "tokens_per_s": round(b * steps * world / (ms / 1e3), 1),
                "us_per_step": round(1e3 * ms / steps, 2),
                "frac": round(nbytes / (ms / 1e3) / 1e9 / peak, 4),
                "instances": n_inst, "hot_l2": n_inst * per < 4 * l2}
            del layers, first
            torch.cuda.empty_cache()
        # conventional read-modify-write on the same rotation of states
        conv = Layer(wl, "f32", device, seed=5, share=base)
        per = conv.state_elems() * 4
        n_inst = 1 if per >= 4 * l2 else min(256, math.ceil(4 * l2 / per))
        states = [conv.state.S_ckpt] + [conv.state.S_ckpt.clone() for _ in range(1, n_inst)]
        for i in range(warm):
            conv.conventional(states[i % n_inst], base.pool[i % POOL])
        torch.cuda.synchronize()
        a, e = ev(), ev()
        a.record(stream)
        for i in range(steps):
            conv.conventional(states[i % n_inst], base.pool[i % POOL])
        e.record(stream)
        e.synchronize()
        ms = max_over_ranks(a.elapsed_time(e), world)
        row["conventional"] = {
            "tokens_per_s": round(b * steps * world / (ms / 1e3), 1),
            "us_per_step": round(1e3 * ms / steps, 2),
            "frac": round(conv.conventional_bytes() * steps / (ms / 1e3) / 1e9 / peak, 4),
            "instances": n_inst, "hot_l2": n_inst * per < 4 * l2}
        row["replay_bf16_vs_conventional"] = round(
            row["replay_bf16"]["tokens_per_s"] / row["conventional"]["tokens_per_s"], 3)
        rows.append(row)
        del conv, states, base
        torch.cuda.empty_cache()
    return {"workload": "kda_h32_d128_w16 batch sweep", "steps": steps, "warmup": warm,
            "l2_bytes": l2, "rows": rows}


def layer_bytes(layer):
    """Device bytes of one layer instance's state: checkpoint, read copy, ring."""
    st = layer.state
    n = st.S_ckpt.numel() * 4 + (st.S_read.numel() * 2 if st.S_read is not None else 0)
    return n + sum(t.numel() * t.element_size() for t in st.ring.values())


def call_stats(dec_ms, gaps_us, folds, window=None, tokens_per_call=None):
    """Per-call device times of the timed steps: the median of the calls that
    fold nothing, the mean of those that fold, and the median idle gap on the
    device between one call's end and the next call's start (host-bound
    stretches show up there).

    With both kinds of call present (lockstep ring phases), also the steady
    state of one fold cycle, which does not depend on how many folds the
    timed window happens to hold: window - 1 plain calls and one folding
    call per cycle, each followed by the median gap."""
    plain = [1e3 * t for t, f in zip(dec_ms, folds) if not f]
    fold = [1e3 * t for t, f in zip(dec_ms, folds) if f]
    gap = statistics.median(gaps_us) if gaps_us else None
    out = {"plain_call_us_median": round(statistics.median(plain), 2) if plain else None,
           "fold_call_us": round(sum(fold) / len(fold), 2) if fold else None,
           "fold_calls": len(fold),
           "host_gap_us_median": round(gap, 2) if gap is not None else None}
    if plain and fold and window and tokens_per_call:
        cycle = ((window - 1) * statistics.median(plain) + sum(fold) / len(fold)) / window
        out["cycle_call_us"] = round(cycle, 2)
        out["cycle_tokens_per_s"] = round(tokens_per_call / ((cycle + (gap or 0.0)) * 1e-6), 1)
    return out


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
    its inputs from pinned host memory and reads the output back. The copies
    run on two copy streams, one per direction, with three staging sets: step
    i + 1's inputs go up while step i computes and step i - 1's output comes
    down, as a serving loop that overlaps transfers with compute does. The
    record adds each direction's copy rate alone and the token rate they
    bound, and the host's enqueue time per step."""
    import torch

    # A step's inputs travel as one pinned buffer (one copy per step); the
    # tensors the call takes are views of its device twin, 256-byte aligned.
    names = list(layer.pool[0])
    offs, o = {}, 0
    for n in names:
        offs[n] = o
        o += -(-layer.pool[0][n].numel() * layer.pool[0][n].element_size() // 256) * 256
    h2d = o

    def views(buf):
        return {n: buf[offs[n]:offs[n] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for n, t in layer.pool[0].items()}

    host = []
    for tok in layer.pool:
        hb = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        for n, t in views(hb).items():
            t.copy_(tok[n].cpu())
        host.append(hb)
    NB = 3  # staging sets: step i + 1 goes up and step i - 1 comes down while step i runs
    dev_bufs = [torch.empty(h2d, dtype=torch.uint8, device=layer.device) for _ in range(NB)]
    stages = [views(b) for b in dev_bufs]
    outs = [layer.out] + [torch.empty_like(layer.out) for _ in range(NB - 1)]
    y_host = [torch.empty(layer.out.shape, dtype=torch.float32).pin_memory() for _ in range(NB)]
    d2h = y_host[0].numel() * 4
    K = max(64, args.steps // 4)
    up, down = torch.cuda.Stream(layer.device), torch.cuda.Stream(layer.device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    landed, done, read = [ev() for _ in range(NB)], [ev() for _ in range(NB)], [ev() for _ in range(NB)]
    started = [False] * NB

    def step(i):
        k = i % NB
        with torch.cuda.stream(up):  # inputs of step i, once step i - NB has used the set
            if started[k]:
                up.wait_event(done[k])
            dev_bufs[k].copy_(host[i % POOL], non_blocking=True)
            landed[k].record(up)
        stream.wait_event(landed[k])
        if started[k]:
            stream.wait_event(read[k])  # step i - NB's output has been read back
        layer.out = outs[k]
        layer.step(stages[k])
        done[k].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(done[k])
            y_host[k].copy_(outs[k], non_blocking=True)
            read[k].record(down)
        started[k] = True

    for i in range(8):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    up.wait_event(a)
    t0 = time.perf_counter()
    for i in range(K):
        step(i)
    host_us = (time.perf_counter() - t0) * 1e6 / K
    stream.wait_event(read[(K - 1) % NB])
    b.record(stream)
    b.synchronize()
    layer.out = outs[0]
    ms = max_over_ranks(a.elapsed_time(b), world)
    # the same copies alone, each direction on its stream: the bound the
    # transfers set on this loop (the directions overlap each other)
    t = {}
    for name, strm in (("up", up), ("down", down)):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        c0.record(strm)
        with torch.cuda.stream(strm):
            for i in range(K):
                if name == "up":
                    dev_bufs[i % NB].copy_(host[i % POOL], non_blocking=True)
                else:
                    y_host[i % NB].copy_(outs[i % NB], non_blocking=True)
        c1.record(strm)
        c1.synchronize()
        t[name] = max_over_ranks(c0.elapsed_time(c1), world) / K
    bound = layer.wl["batch"] * world / (max(t["up"], t["down"]) / 1e3)
    return {"value": round(layer.wl["batch"] * K * world / (ms / 1e3), 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "copies": "one pinned input buffer and the output per step; one copy stream per direction, three staging sets",
            "host_enqueue_us_per_step": round(host_us, 2),
            "h2d_gbs": round(h2d / (t["up"] / 1e3) / 1e9, 1),
            "d2h_gbs": round(d2h / (t["down"] / 1e3) / 1e9, 1),
            "copy_bound_tokens_per_s": round(bound, 1)}


def run_spec(args, rank, local_rank, world):
    """Speculative decoding rounds as the JSON line's workload."""
    import torch

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    clocks = ClockSampler(local_rank) if not args.no_extras else None
    if clocks:
        clocks.__enter__()
    res = spec_rounds(args, device, world)
    if clocks:
        clocks.__exit__(None, None, None)
        res["clocks"] = clocks.summary()
    return res


def spec_rounds(args, device, world):
    """Speculative decoding rounds on a delta layer: consolidate(k_next = K),
    verify K drafts from one read of the state, accept m drafts by moving the
    ring pointer (m drawn U{0..K} per sequence and round). The A/B runs the
    conventional baseline on the same drafts first: verify with a state
    snapshot per draft, then accept by copying snapshot m - 1 into the state."""
    import numpy as np
    import torch

    import synth
    from recurrent_state_fp32_b300 import api

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
    drafts, ms, m_host, m_tot = [], [], [], []
    for r in range(rounds_pool):
        dr = synth.spec_draft_inputs(seed, r, b, K, H, dk, dv, kind, "bf16")
        drafts.append({n: to(v, torch.bfloat16 if n in ("q", "k", "v") else torch.float32)
                       for n, v in dr.items()})
        m = synth.accept_counts(seed, r, b, K)
        ms.append(to(m, torch.int32))
        m_host.append(np.asarray(m, np.int64))
        m_tot.append(int(m.sum()))
    o = torch.empty((b, K, H, dv), device=device)
    stream = torch.cuda.current_stream(device)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    Kt, Wm = args.steps, args.warmup
    extras = {}
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
        extras["ab"] = {"conventional_accepted_tokens_per_s": round(acc_c / (cms / 1e3), 1),
                        "conventional_ms_per_round": round(cms / Kc, 5), "rounds": Kc,
                        # verify: read S, write K snapshots; accept: copy one snapshot
                        # for every sequence with m > 0
                        "conventional_bytes_per_round":
                            int(b * H * dv * dk * 4 * (1 + K) +
                                np.mean([int((mm > 0).sum().item()) for mm in ms]) * H * dv * dk * 8)}
        del S, snaps
        torch.cuda.empty_cache()

    v0 = [ev() for _ in range(Kt)]
    v1 = [ev() for _ in range(Kt)]

    def round_(i, timed=None):
        d = drafts[i % rounds_pool]
        api.consolidate(dims, state, None, K, False)
        if timed is not None:
            v0[timed].record(stream)
        api.spec_verify(dims, state, K, d["q"], d["k"], d["v"], d["alpha"], d["beta"], 1.0, o)
        if timed is not None:
            v1[timed].record(stream)
        api.accept(dims, state, ms[i % rounds_pool], K)

    for i in range(Wm):
        round_(i)
    torch.cuda.synchronize()
    lens0 = state.ring_len.cpu().numpy().astype(np.int64)
    a0, a1 = ev(), ev()
    barrier(world)
    torch.cuda.synchronize()
    a0.record(stream)
    for i in range(Kt):
        round_(Wm + i, timed=i)
    a1.record(stream)
    a1.synchronize()
    barrier(world)
    ms_tot = max_over_ranks(a0.elapsed_time(a1), world)
    ver_ms = sum(v0[i].elapsed_time(v1[i]) for i in range(Kt))
    accepted = sum(m_tot[(Wm + i) % rounds_pool] for i in range(Kt)) * world
    bad = int(state.status.ne(0).sum().item())
    ver_bytes, fold_bytes = spec_account(dims, state, lens0, [m_host[(Wm + i) % rounds_pool]
                                                                for i in range(Kt)], K)
    peak, peak_kind = measured_peaks()
    res = {
        "metric": SPEC_METRIC,
        "value": round(accepted / (ms_tot / 1e3), 1), "unit": SPEC_UNIT,
        "n_gpus": world, "steps": Kt, "warmup": Wm, "ms_per_step": round(ms_tot / Kt, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; no weights or datasets)",
        "config": spec_config(wl, args.read, world),
        "verified_tokens_per_s": round(b * K * Kt * world / (ms_tot / 1e3), 1),
        "step_hbm_gbs": round((ver_bytes + fold_bytes) / (ms_tot / 1e3) / 1e9, 1),
        "roofline": {
            "kernel": "delta_fused_kernel<K=4> (one verify call)", "bound": "hbm",
            "achieved": round(ver_bytes / (ver_ms / 1e3) / 1e9, 1), "peak": peak,
            "peak_source": peak_kind, "unit": "GB/s",
            "frac": round(ver_bytes / (ver_ms / 1e3) / 1e9 / peak, 4), "traffic": None,
            "bytes_per_launch": int(ver_bytes / Kt), "avg_launch_us": round(1e3 * ver_ms / Kt, 3)},
        "gpu_launches": Kt * 3, "device_status_ok": bad == 0,
    }
    res.update(extras)
    return res


def spec_account(dims, state, lens0, m_rounds, K):
    """Algorithmic bytes of speculative rounds (verify, consolidate) from the
    ring lengths before them and each round's accept counts. Verify: the
    state read once (read copy, else FP32), the committed entries' k, v, gate
    and beta, the K drafts read and written to the ring, the K outputs.
    Consolidate(k_next = K): for each sequence with len + K > W, FP32 read and
    write (and the read copy written) plus its entries."""
    import numpy as np

    b, H, dk, dv, W = dims.batch, dims.heads, dims.dk, dims.dv, dims.window
    elems = H * dv * dk
    ts = 2 if state.S_read is not None else 4
    gate = H * 4 if dims.kind == "gdn" else H * dk * 4
    entry = H * dk * 2 + H * dv * 2 + gate + H * 4        # k, v, alpha, beta of one entry
    draft = H * dk * 2 * 2 + H * dv * 2 + gate + H * 4    # q, k, v, alpha, beta
    lens = np.array(lens0, np.int64)
    ver = fold = 0.0
    for m in m_rounds:
        f = lens + K > W
        fold += f.sum() * (elems * (8 + (2 if ts == 2 else 0))) + lens[f].sum() * entry
        lens[f] = 0
        ver += b * elems * ts + lens.sum() * entry + b * K * (2 * draft) + b * K * H * dv * 4
        lens += np.asarray(m, np.int64)
    return ver, fold


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


def _oracle_steps(job):
    """One host process or thread of the CPU baseline: the oracle on one
    sequence (all heads) of the workload for about `seconds`, single-threaded.
    Returns (steps, seconds)."""
    wl, seconds, seed = job
    with _single_thread():
        orc, toks, _ = oracle_sample(wl, wl["heads"], seed=seed)
        t0 = time.perf_counter()
        n = 0
        while True:
            orc.consolidate(1)
            orc.decode(toks[n % POOL])
            n += 1
            if time.perf_counter() - t0 > seconds and n % wl["window"] == 0:
                break
        return n, time.perf_counter() - t0


def cpu_baseline(wl: dict, seconds: float):
    """The oracle as it stands on the host's cores, on a bounded sample of the
    same workload: one single-threaded process per host core, each decoding
    its own sequence (all heads) for about `seconds`; tokens/s summed over the
    processes. The single-threaded rate of one such process is reported too.
    The pool is spawned (never forked) so no child inherits a CUDA context."""
    import multiprocessing as mp

    host_cores = os.cpu_count() or 1
    n1, t1 = _oracle_steps((wl, seconds, 2))
    single = round(n1 / t1, 3)
    procs = host_cores
    with mp.get_context("spawn").Pool(procs) as pool:
        runs = pool.map(_oracle_steps, [(wl, seconds, 100 + i) for i in range(procs)])
    value = sum(n / t for n, t in runs)
    return {"value": round(value, 3), "unit": UNIT, "cores": procs, "host_cores": host_cores,
            "kind": "oracle",
            "sample": f"{procs} processes x 1 sequence x {wl['heads']} heads, each about "
                      f"{seconds:.0f} s of consecutive decode steps (consolidate + decode), "
                      f"float64 numpy, one thread each",
            "single_thread": {"value": single, "unit": UNIT, "cores": 1,
                              "sample": f"1 sequence x {wl['heads']} heads, {n1} steps, "
                                        f"{t1:.1f} s"}}


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
        # ms_per_step is per sampled step (one sequence, a slice of its heads);
        # a whole step or round of the workload is batch / frac of them
        "ms_per_workload_step": round(1e3 * dt / args.steps * wl["batch"] / frac, 1),
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
