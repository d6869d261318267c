#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300: one step = forward +
backward (fa_fwd, then fa_bwd's three kernels) over one batch of synthetic
bf16 inputs of the long-context causal shape (B=1, Hq=Hkv=16, N=32768,
d=128), the largest causal configuration; the standard causal (B4 H16 N2048),
grouped-query causal (B2 Hq32 Hkv8 N8192), stressed non-causal d=64 and tiny
workloads are timed the same way in the same run and reported under
`per_config`.

Prints ONE JSON line (rank 0).  `value` is TFLOPS under the convention
fwd = 4*B*Hq*N^2*d (halved when causal), bwd = 2.5 x fwd, over the device time
of the K timed steps (CUDA events around each step on the launching stream;
between steps, outside the events, L2 is flushed by a 256 MiB write and then
a 256 MiB read of another buffer, so each step starts from a cold and clean
L2 instead of writing back the flush's dirty lines itself).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-per-config] [--no-cpu-baseline]
  python bench.py --next     # the widened paths: decode (Nq << Nk) and window

--next prints one JSON line per widened-path case (not the contract line):
decode-shaped grouped attention (few query rows against a long key/value
history, key splits + merge) against the HBM roofline, and sliding-window
causal attention (forward and backward) in TFLOPS over the visible pairs.

--impl reference times the CPU oracle (fp64 NumPy) on the host cores: each
step is a bounded sample of the same workload (one block of query rows of one
head, forward + backward), reported in the same unit.
Multi-GPU (torchrun): every rank runs an independent replica of the workload
on its own GPU (weak scaling, no collective on the data path); the time is
the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_io_aware_flashattention_gb300.inputs import BENCH_WORKLOAD, WORKLOADS, make_workload_inputs  # noqa: E402

L2_FLUSH_BYTES = 256 * 2 ** 20
L2_FLUSH_DESC = ("flushed between steps: 256 MiB write, then a 256 MiB read of another buffer so the write's "
                 "dirty lines are written back before the step (all outside the timed events)")


class L2Flush:
    """Between timed steps: write a buffer larger than L2 (nothing of the
    previous step stays resident), then read a second one, so that the lines
    the write left dirty are written back here and not inside the next timed
    step: the step starts from a cold and clean L2, the state ncu profiles
    from."""

    def __init__(self, torch, dev):
        self.wr = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)   # sums without a cast

    def __call__(self):
        self.wr.fill_(1)
        self.rd.sum()
FALLBACK_BF16_TFLOPS = 1900.0
DOMINANT_KERNEL = "fa_bwd_dkdv_kernel"
METRIC = "attention fwd/bwd TFLOPS (bf16, causal) and % of GB300 dense-bf16 peak, 1 GPU"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank float over the default process group (identity if none)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(step_flops: float, world: int, total_ms_max: float, steps: int) -> float:
    """Whole-job TFLOPS: the work of every rank over the slowest rank's time."""
    return step_flops * world * steps / (total_ms_max * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# measured peaks, kernel source hash, ncu traffic record
# ---------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s, earlier GB300 measurement)"


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16 burst, earlier GB300 measurement)"


def bf16_peak_sustained():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["bf16_tflops_sustained"]), "measured (MEASURED_PEAKS.json bf16_tflops_sustained)"
    except Exception:
        return 1700.0, "fallback (1.7 PFLOP/s bf16 sustained, earlier GB300 measurement)"


# Source files each timed kernel is compiled from; a committed ncu figure is
# used only while these files are unchanged.
KERNEL_SOURCES = {
    "fa_fwd_kernel": ("fa_fwd.cu", "fa_internal.h", "sm103a.cuh"),
    "fa_bwd_dkdv_kernel": ("fa_bwd.cu", "fa_internal.h", "sm103a.cuh"),
    "fa_bwd_dq_kernel": ("fa_bwd_dq.cu", "fa_internal.h", "sm103a.cuh"),
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_io_aware_flashattention_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    if there is none for this workload or the kernel's sources changed since."""
    src_hash = kernel_source_hash(kernel)
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
        e = rec[kernel][workload]
        if e.get("source_hash") != src_hash:
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(os.devnull, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=self.out, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            text, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            text, _ = self.proc.communicate()
        rows = [[c.strip() for c in l.split(",")] for l in text.strip().splitlines() if l.count(",") >= 9]
        if self.bus_id:
            mine = [r for r in rows if r[1].lower().endswith(self.bus_id[-12:])]
            rows = mine or rows
        if rows and not self.bus_id:
            first = rows[0][0]
            rows = [r for r in rows if r[0] == first]
        sm = [float(r[2].split()[0]) for r in rows if r[2].split()[0].replace(".", "").isdigit()]
        mx = [float(r[3].split()[0]) for r in rows if r[3].split()[0].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle sample (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def oracle_sample_plan(w, rows_per_sample=128):
    """Row blocks (b, h, r0, r1) of the workload, spread over the sequence."""
    import numpy as np
    rng = np.random.default_rng(12345)
    nblk = w.N // rows_per_sample if w.N >= rows_per_sample else 1
    while True:
        b = int(rng.integers(w.B))
        h = int(rng.integers(w.Hq))
        blk = int(rng.integers(nblk))
        r0 = blk * rows_per_sample
        yield b, h, r0, min(w.N, r0 + rows_per_sample)


def sample_flops(w, r0, r1):
    """Convention FLOPs (fwd + bwd) of query rows r0..r1-1 of one head."""
    if w.causal:
        pairs = sum(i + 1 for i in range(r0, r1))
    else:
        pairs = (r1 - r0) * w.N
    return 4.0 * w.d * pairs * 3.5


def run_oracle_sample(w, tensors, b, h, r0, r1):
    from oracle import ref
    q, k, v, do = tensors
    g = h // (w.Hq // w.Hkv)
    sub = (q[b:b + 1, h:h + 1], k[b:b + 1, g:g + 1], v[b:b + 1, g:g + 1])
    ref.attention_forward(*sub, w.causal, w.scale, row_range=(r0, r1))
    ref.attention_backward(*sub, do[b:b + 1, h:h + 1], w.causal, w.scale, row_range=(r0, r1))


def f64_tensors(w):
    q, k, v, do = make_workload_inputs(w)
    return tuple(t.to(__import__("torch").float64).numpy() for t in (q, k, v, do))


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(w, tensors, budget_s=12.0):
    plan = oracle_sample_plan(w)
    flops = 0.0
    n = 0
    t0 = time.perf_counter()
    while True:
        b, h, r0, r1 = next(plan)
        run_oracle_sample(w, tensors, b, h, r0, r1)
        flops += sample_flops(w, r0, r1)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} blocks of 128 query rows (one head each, fwd+bwd, fp64 NumPy), {dt:.1f} s"}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    tensors = f64_tensors(w)
    plan = oracle_sample_plan(w)
    for _ in range(args.warmup):
        run_oracle_sample(w, tensors, *next(plan))
    flops = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        b, h, r0, r1 = next(plan)
        run_oracle_sample(w, tensors, b, h, r0, r1)
        flops += sample_flops(w, r0, r1)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"each step: one block of 128 query rows of one head, forward + backward, "
                                   f"fp64 NumPy oracle; {args.steps} steps"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d, "causal": w.causal,
            "scale": w.scale, "global_batch": w.B, "seq_len": w.N,
            "l2": L2_FLUSH_DESC,
            "parallelism": "replicas (one independent workload per GPU)"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class Problem:
    """Device buffers of one workload and one contract step over them: fa_fwd,
    then fa_bwd's three kernels (preprocess, dK/dV, dQ conversion) through the
    C ABI on one stream."""

    def __init__(self, fa, torch, w, dev, stream):
        self.fa, self.w, self.stream = fa, w, stream
        self.host = make_workload_inputs(w)
        self.q, self.k, self.v, self.do = (t.to(dev) for t in self.host)
        B, Hq, Hkv, N, d = w.B, w.Hq, w.Hkv, w.N, w.d
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = torch.empty_like(self.q), torch.empty_like(self.k), torch.empty_like(self.v)
        self.ws_bytes = fa.fa_bwd_workspace_bytes(B, Hq, Hkv, N, d)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)

    def device_mib(self):
        """Device memory the step needs: inputs, outputs and the backward's
        workspace (the library allocates nothing itself), MiB; and the same as
        a multiple of the O(N d) inputs."""
        ts = (self.q, self.k, self.v, self.do, self.o, self.lse, self.dq, self.dk, self.dv, self.ws)
        total = sum(t.numel() * t.element_size() for t in ts)
        inputs = sum(t.numel() * t.element_size() for t in (self.q, self.k, self.v, self.do))
        return {"step_buffers_mib": round(total / 2**20, 1), "x_inputs": round(total / inputs, 2)}

    def _call(self, status, what):
        if status != 0:
            raise self.fa.FAError(status, what)

    def step(self, ev=None):
        fa, w, sh = self.fa, self.w, self.stream.cuda_stream
        B, Hq, Hkv, N, d = w.B, w.Hq, w.Hkv, w.N, w.d
        p = lambda t: t.data_ptr()  # noqa: E731
        if ev:
            ev[0].record(self.stream)
        self._call(fa.fa_fwd(p(self.q), p(self.k), p(self.v), p(self.o), p(self.lse), B, Hq, Hkv, N, d, w.causal,
                             w.scale, sh), "fwd")
        if ev:
            ev[1].record(self.stream)
        self._call(fa.fa_bwd_preprocess(p(self.o), p(self.do), p(self.lse), B, Hq, Hkv, N, d, p(self.ws),
                                        self.ws_bytes, sh), "bwd_preprocess")
        if ev:
            ev[2].record(self.stream)
        self._call(fa.fa_bwd_dkdv(p(self.q), p(self.k), p(self.v), p(self.do), p(self.dk), p(self.dv), B, Hq, Hkv,
                                  N, d, w.causal, w.scale, p(self.ws), self.ws_bytes, sh), "bwd_dkdv")
        if ev:
            ev[3].record(self.stream)
        self._call(fa.fa_bwd_dq_convert(p(self.dq), B, Hq, Hkv, N, d, w.scale, p(self.ws), self.ws_bytes, sh),
                   "bwd_dq_convert")
        if ev:
            ev[4].record(self.stream)

    def time(self, torch, steps, warmup, flush):
        """Per-kernel mean device ms over `steps` steps (L2 flushed before each,
        outside the events): dict fwd, pre, dkdv, conv, step, plus the step total."""
        for _ in range(max(3, warmup)):
            flush()
            self.step()
        torch.cuda.synchronize()
        self.fa.check_device_status()
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        for i in range(steps):
            flush()
            self.step(events[i])
        torch.cuda.synchronize()
        self.fa.check_device_status()
        ms = {"fwd": [e[0].elapsed_time(e[1]) for e in events], "pre": [e[1].elapsed_time(e[2]) for e in events],
              "dkdv": [e[2].elapsed_time(e[3]) for e in events], "conv": [e[3].elapsed_time(e[4]) for e in events],
              "step": [e[0].elapsed_time(e[4]) for e in events]}
        out = {k: statistics.mean(v) for k, v in ms.items()}
        out["step_total"] = sum(ms["step"])
        return out


def kernel_figures(w, t, peak):
    """fwd / bwd TFLOPS and fractions of `peak` from Problem.time's means."""
    bwd_ms = t["pre"] + t["dkdv"] + t["conv"]
    fwd_tf = w.fwd_flops / (t["fwd"] * 1e-3) / 1e12
    bwd_tf = w.bwd_flops / (bwd_ms * 1e-3) / 1e12
    dkdv_tf = w.bwd_flops / (t["dkdv"] * 1e-3) / 1e12
    return {
        "fwd": {"tflops": fwd_tf, "ms": t["fwd"], "frac_of_peak": fwd_tf / peak},
        "bwd": {"tflops": bwd_tf, "ms": bwd_ms, "frac_of_peak": bwd_tf / peak, "ms_preprocess": t["pre"],
                "ms_dkdv": t["dkdv"], "ms_dq_convert": t["conv"], "dkdv_tflops": dkdv_tf,
                "dkdv_frac_of_peak": dkdv_tf / peak},
        "step": {"ms": t["step"], "tflops": (w.fwd_flops + w.bwd_flops) / (t["step"] * 1e-3) / 1e12},
    }


# The other workloads of the path, timed in the same run as the headline (one
# line, `per_config`): the tiny and stressed ones are reported, the causal ones
# carry the same targets as the headline.
PER_CONFIG = ("tiny_b1_h1_n128_d64", "causal_b4_h16_n2048_d128", "gqa_causal_b2_hq32_hkv8_n8192_d128",
              "stressed_b8_h32_n4096_d64")


def run_ours(args, w):
    import torch
    import exact_io_aware_flashattention_gb300 as fa
    from exact_io_aware_flashattention_gb300 import _build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device() if world == 1 else local)
    if rank == 0 or world > 1:
        _build.build()
    if world > 1:
        dist.barrier()
    fa.load_library()

    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(torch, dev)
    prob = Problem(fa, torch, w, dev, stream)
    q_h, k_h, v_h, do_h = prob.host
    B, Hq, N = w.B, w.Hq, w.N
    peak, peak_src = bf16_peak()
    peak_sus, peak_sus_src = bf16_peak_sustained()

    for _ in range(max(3, args.warmup)):
        flush()
        prob.step()
    torch.cuda.synchronize(dev)
    fa.check_device_status()

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    sampler = ClockSampler(getattr(torch.cuda.get_device_properties(dev), "pci_bus_id", None))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.25)  # let the sampler attach before the timed region
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush()
        prob.step(events[i])
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    fa.check_device_status()

    t = {"fwd": statistics.mean(e[0].elapsed_time(e[1]) for e in events),
         "pre": statistics.mean(e[1].elapsed_time(e[2]) for e in events),
         "dkdv": statistics.mean(e[2].elapsed_time(e[3]) for e in events),
         "conv": statistics.mean(e[3].elapsed_time(e[4]) for e in events),
         "step": statistics.mean(e[0].elapsed_time(e[4]) for e in events)}
    total_ms = max_over_ranks(sum(e[0].elapsed_time(e[4]) for e in events), dev)
    ms_per_step = total_ms / args.steps
    step_flops = w.fwd_flops + w.bwd_flops
    value = aggregate_tflops(step_flops, world, total_ms, args.steps)
    figs = kernel_figures(w, t, peak)
    if t["dkdv"] >= t["fwd"]:
        dom, dom_flops, dom_ms = "fa_bwd_dkdv_kernel", w.bwd_flops, t["dkdv"]
    else:
        dom, dom_flops, dom_ms = "fa_fwd_kernel", w.fwd_flops, t["fwd"]
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    src_hash = {k: kernel_source_hash(k) for k in KERNEL_SOURCES}

    # ---------------- e2e through host buffers (pinned), copies inside the timed region
    e2e = None
    if rank == 0 or world > 1:
        pin = lambda t_: t_.pin_memory()  # noqa: E731
        hq, hk, hv, hdo = pin(q_h), pin(k_h), pin(v_h), pin(do_h)
        ho, hlse = pin(torch.empty_like(q_h)), pin(torch.empty((B, Hq, N), dtype=torch.float32))
        hdq, hdk, hdv = pin(torch.empty_like(q_h)), pin(torch.empty_like(k_h)), pin(torch.empty_like(v_h))
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdo))
        d2h = sum(x.numel() * x.element_size() for x in (ho, hlse, hdq, hdk, hdv))

        # Steps are pipelined the way a training loop prefetches: step i's
        # inputs are copied in on one stream while step i-1 computes, and its
        # outputs are copied out on another while step i+1 computes.  Two
        # device buffer sets alternate; each step still moves all of its
        # inputs in and all of its outputs (O, LSE, dQ, dK, dV) out inside
        # the timed region.
        sets = [dict(q=prob.q, k=prob.k, v=prob.v, do=prob.do, o=prob.o, lse=prob.lse, dq=prob.dq, dk=prob.dk,
                     dv=prob.dv, ws=prob.ws)]
        sets.append({name: torch.empty_like(x) for name, x in sets[0].items()})
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_c = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_run(n_steps):
            for i in range(n_steps):
                x, S = i % 2, sets[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_c[x])       # compute i-2 has read this set's inputs
                    S["q"].copy_(hq, non_blocking=True)
                    S["k"].copy_(hk, non_blocking=True)
                    S["v"].copy_(hv, non_blocking=True)
                    S["do"].copy_(hdo, non_blocking=True)
                    ev_in[x].record(s_in)
                stream.wait_event(ev_in[x])
                if i >= 2:
                    stream.wait_event(ev_out[x])       # outputs of step i-2 copied out
                fa.forward(S["q"], S["k"], S["v"], causal=w.causal, scale=w.scale, out=S["o"], lse=S["lse"],
                           stream=stream)
                fa.backward(S["q"], S["k"], S["v"], S["o"], S["lse"], S["do"], causal=w.causal, scale=w.scale,
                            workspace=S["ws"], dq=S["dq"], dk=S["dk"], dv=S["dv"], stream=stream)
                ev_c[x].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_c[x])
                    ho.copy_(S["o"], non_blocking=True)
                    hlse.copy_(S["lse"], non_blocking=True)
                    hdq.copy_(S["dq"], non_blocking=True)
                    hdk.copy_(S["dk"], non_blocking=True)
                    hdv.copy_(S["dv"], non_blocking=True)
                    ev_out[x].record(s_out)

        e2e_run(3)
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(args.steps, 50))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        e2e_run(n_e2e)
        e1.record(s_out)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        fa.check_device_status()
        e2e = {"value": step_flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": n_e2e, "path": "pinned host -> fa.forward/fa.backward (C ABI) -> pinned host, "
               "copies on their own streams, overlapping the neighbouring steps' compute"}
        del sets, hq, hk, hv, hdo, ho, hlse, hdq, hdk, hdv

    # ---------------- the other workloads, same run, same step, same timing
    per_config = None
    if rank == 0 and not args.no_per_config:
        per_config = {}
        pc_sampler = ClockSampler(getattr(torch.cuda.get_device_properties(dev), "pci_bus_id", None))
        pc_sampler.start()
        for name in PER_CONFIG:
            if name == w.name:
                continue
            pw = WORKLOADS[name]
            pp = Problem(fa, torch, pw, dev, stream)
            pt = pp.time(torch, args.per_config_steps, 3, flush)
            per_config[name] = kernel_figures(pw, pt, peak)
            per_config[name]["device_memory"] = pp.device_mib()
            del pp
            torch.cuda.empty_cache()
        per_config["clocks"] = pc_sampler.stop()
        per_config["steps"] = args.per_config_steps

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, f64_tensors(w))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w),
            "fwd": figs["fwd"],
            "bwd": figs["bwd"],
            "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_src,
                         "frac_of_sustained": achieved / peak_sus, "sustained_peak": peak_sus,
                         "sustained_peak_source": peak_sus_src,
                         "traffic": ncu_traffic(dom, w.name),
                         "algorithmic_flops_per_launch": dom_flops},
            "device_memory": prob.device_mib(),
            "per_config": per_config,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks,
            "gpu_launches": 4 * args.steps,
            "wall_s_timed_region": wall,
            "kernel_source_hash": src_hash,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile(args, w):
    """A short launch sequence for profilers: `warmup` + `steps` contract steps
    of the workload, no L2 flush, no timing, no host copies.  `--heads H`
    scales the workload down to H query heads (and Hkv in proportion) so a
    full counter capture stays small; traffic then scales with the heads."""
    import dataclasses
    import torch
    import exact_io_aware_flashattention_gb300 as fa
    from exact_io_aware_flashattention_gb300 import _build
    _build.build()
    fa.load_library()
    if args.heads:
        g = w.Hq // w.Hkv
        if args.heads % g:
            raise SystemExit(f"--heads must be a multiple of {g}")
        w = dataclasses.replace(w, name=f"{w.name}@hq{args.heads}", Hq=args.heads, Hkv=args.heads // g)
    dev = torch.device("cuda", 0)
    prob = Problem(fa, torch, w, dev, torch.cuda.current_stream(dev))
    for _ in range(args.warmup + args.steps):
        prob.step()
    torch.cuda.synchronize(dev)
    fa.check_device_status()
    print(json.dumps({"profile": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
                      "launches": 4 * (args.warmup + args.steps)}), flush=True)
    return 0


def _time_events(fn, steps, warmup, flush, stream):
    """Mean device ms of fn over `steps` runs (CUDA events on `stream`), with an
    L2 flush before each run outside the events."""
    import torch
    for _ in range(warmup):
        fn()
    total = 0.0
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        total += a.elapsed_time(b)
    return total / steps


def run_next(args):
    """Measure the widened paths; one JSON line per case."""
    import torch
    import exact_io_aware_flashattention_gb300 as fa
    from exact_io_aware_flashattention_gb300 import _build
    _build.build()
    fa.load_library()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(torch, dev)
    steps, warmup = max(args.steps, 20), max(args.warmup, 3)
    hbm, hbm_src = hbm_peak()
    peak, peak_src = bf16_peak()

    def gen(shape, seed):
        g = torch.Generator().manual_seed(seed)
        return torch.randn(shape, generator=g).to(torch.bfloat16).to(dev)

    # Decode: B=8, Hq=32, Hkv=8 (4 query heads per kv head), one new query row.
    for Nk in (8192, 32768):
        B, Hq, Hkv, Nq, d = 8, 32, 8, 1, 128
        q, k, v = gen((B, Hq, Nq, d), 1), gen((B, Hkv, Nk, d), 2), gen((B, Hkv, Nk, d), 3)
        splits = fa.fa_fwd_ex_default_splits(B, Hq, Hkv, Nq, Nk, d, 1, 0)
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
        ws = torch.empty(max(1, fa.fa_fwd_ex_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, splits)), dtype=torch.uint8,
                         device=dev)

        def fn():
            st = fa.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Nq,
                              Nk, d, 1, 0, splits, d ** -0.5, ws.data_ptr(), ws.numel(), stream.cuda_stream)
            if st != 0:
                raise fa.FAError(st, "fa_fwd_ex")
        ms = _time_events(fn, steps, warmup, flush, stream)
        fa.check_device_status()
        # Algorithmic bytes: K and V once (each kv head read once for its 4
        # query heads), Q, O and LSE.
        nbytes = 2 * B * Hkv * Nk * d * 2 + 2 * B * Hq * Nq * d * 2 + B * Hq * Nq * 4
        gbs = nbytes / (ms * 1e-3) / 1e9
        print(json.dumps({"case": "decode", "metric": "decode attention HBM throughput", "value": gbs,
                          "unit": "GB/s", "us": ms * 1e3, "dtype": "bf16", "data": "synthetic",
                          "config": {"B": B, "Hq": Hq, "Hkv": Hkv, "Nq": Nq, "Nk": Nk, "d": d, "causal": True,
                                     "num_splits": splits, "l2": L2_FLUSH_DESC},
                          "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                       "frac": gbs / hbm, "peak_source": hbm_src,
                                       "algorithmic_bytes": nbytes}}), flush=True)

    # Sliding window: B=2, H=16, N=8192, d=128, causal, window 1024.
    B, Hq, Hkv, N, d, win = 2, 16, 16, 8192, 128, 1024
    q, k, v, do = gen((B, Hq, N, d), 4), gen((B, Hkv, N, d), 5), gen((B, Hkv, N, d), 6), gen((B, Hq, N, d), 7)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8, device=dev)
    sh = stream.cuda_stream

    def fwd():
        st = fa.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, N, N, d,
                          1, win, 1, d ** -0.5, None, 0, sh)
        if st != 0:
            raise fa.FAError(st, "fa_fwd_ex")

    def bwd():
        st = fa.fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, d, 1, win, 0, d ** -0.5,
                          ws.data_ptr(), ws.numel(), sh)
        if st != 0:
            raise fa.FAError(st, "fa_bwd_ex")
    fwd()
    ms_f = _time_events(fwd, steps, warmup, flush, stream)
    ms_b = _time_events(bwd, steps, warmup, flush, stream)
    fa.check_device_status()
    pairs = sum(min(i + 1, win) for i in range(N))       # visible (query, key) pairs per head
    ff = 4.0 * B * Hq * d * pairs
    tf_f, tf_b = ff / (ms_f * 1e-3) / 1e12, 2.5 * ff / (ms_b * 1e-3) / 1e12
    print(json.dumps({"case": "window", "metric": "sliding-window attention TFLOPS over visible pairs",
                      "value": {"fwd": tf_f, "bwd": tf_b}, "unit": "TFLOPS",
                      "ms": {"fwd": ms_f, "bwd": ms_b}, "dtype": "bf16", "data": "synthetic",
                      "config": {"B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "causal": True, "window": win,
                                 "l2": L2_FLUSH_DESC},
                      "frac_of_peak": {"fwd": tf_f / peak, "bwd": tf_b / peak}, "peak_source": peak_src}),
          flush=True)

    # Deterministic backward (separate dQ kernel) on the standard causal
    # workload, against the reduce-add backward.
    w = WORKLOADS["causal_b4_h16_n2048_d128"]
    B, Hq, Hkv, N, d = w.B, w.Hq, w.Hkv, w.N, w.d
    q, k, v, do = (t.to(dev) for t in make_workload_inputs(w))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8, device=dev)
    res = {}
    for det in (0, 1):
        def bwd_det():
            st = fa.fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                              dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, d, 1, 0, det, w.scale,
                              ws.data_ptr(), ws.numel(), sh)
            if st != 0:
                raise fa.FAError(st, "fa_bwd_ex")
        res[det] = _time_events(bwd_det, steps, warmup, flush, stream)
    fa.check_device_status()
    bf = 2.5 * 4.0 * B * Hq * N * N * d / 2
    print(json.dumps({"case": "deterministic_backward", "metric": "backward TFLOPS (convention 2.5 x causal fwd)",
                      "value": {"deterministic": bf / (res[1] * 1e-3) / 1e12,
                                "reduce_add": bf / (res[0] * 1e-3) / 1e12},
                      "unit": "TFLOPS", "ms": {"deterministic": res[1], "reduce_add": res[0]}, "dtype": "bf16",
                      "data": "synthetic", "config": {"workload": w.name, "l2": L2_FLUSH_DESC}}),
          flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=BENCH_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="time the headline workload only")
    ap.add_argument("--per-config-steps", type=int, default=20)
    ap.add_argument("--next", action="store_true", help="measure the widened paths (decode, window) instead")
    ap.add_argument("--profile", action="store_true",
                    help="only run warmup + steps contract steps (for ncu); prints a short line, not the contract line")
    ap.add_argument("--heads", type=int, default=0, help="with --profile: scale the workload to this many query heads")
    args = ap.parse_args()
    if args.next:
        return run_next(args)
    if args.profile:
        return run_profile(args, WORKLOADS[args.workload])
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
