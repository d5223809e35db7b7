#!/usr/bin/env python
"""Benchmark of the gated delta-rule scan on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one library call over one batch of the named synthetic workload
(default: the packed varlen bf16 prefill, 8 sequences of U[512, 8192] tokens,
H=16, d_k=d_v=128, the largest of the prefill workloads), inputs resident in
HBM, L2 flushed (256 MiB write) before every step and outside its timing.
The same line also carries the other full-size workloads (the 4096-token bf16
prefill, the GQA f16 prefill and the B=256 decode step), each timed the same
way, under "configs".
Each GPU (torchrun rank) runs its own full copy of the workload: the units
(sequence, head) are independent, so there is no collective on the data path
and scaling is weak.  `--impl reference` times the CPU oracle on host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "gated-delta-rule tokens/s (prefill) & state GB/s (decode), % of roofline"
DEFAULT_WORKLOAD = "varlen_bf16_prefill"
# Full-size workloads timed after the main one and reported beside it.
EXTRA_WORKLOADS = ("bf16_prefill_t4096", "gqa_f16_prefill", "bf16_decode_b256")
CHUNK = 64                         # tokens per chunk of the tensor-core prefill
FLUSH_BYTES = 256 << 20            # > 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=workloads.ALL_WORKLOADS)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-extra-configs", action="store_true",
                   help="time only the named workload (no 'configs' entry)")
    return p.parse_args()


# ---------------------------------------------------------------- accounting

def io_bytes(inp) -> dict:
    s = inp.spec
    es = 4 if s.io == "f32" else 2
    T = inp.total_tokens
    n = inp.n_seq
    st = n * s.h_v * s.d_k * s.d_v * 4
    per = s.h_v * (s.d_k if s.decay_per_key else 1)   # decay gates per token
    decay = getattr(s, "rule", "gated_delta") in ("gated_delta", "gated")
    delta = getattr(s, "rule", "gated_delta") in ("gated_delta", "delta")
    return {
        "q": T * s.h_qk * s.d_k * es, "k": T * s.h_qk * s.d_k * es, "v": T * s.h_v * s.d_v * es,
        "a": T * per * es if decay else 0, "b": T * (1 if s.beta_shared else s.h_v) * es if delta else 0,
        "params": 2 * per * 4 if decay else 0,
        "state_in": st if (inp.state_in is not None or inp.pool is not None) else 0,
        "o": T * s.h_v * s.d_v * es, "state_out": st * (s.window if s.window else 1),
        "slots": 4 * n if inp.pool is not None else 0,
    }


def bandwidth_metric(spec) -> bool:
    """Decode-like steps (one token, or a short verify window of per-step states) are
    measured in state GB/s on the token-sequential kernel; prefill in tokens/s."""
    return bool(spec.decode or spec.window)


def algorithmic_bytes(inp) -> int:
    """Minimum HBM traffic of one call: every input read once, every output written once."""
    return int(sum(io_bytes(inp).values()))


def algorithmic_flops(inp) -> float:
    """Chunked prefill, C = 64, per (token, value head): 10*C*d + 6*d^2, with the
    q.k and k.k chunk products (4*C*d) counted once per q/k head.  Decode: 8*d_k*d_v."""
    s = inp.spec
    T = inp.total_tokens
    if bandwidth_metric(s):
        return 8.0 * T * s.h_v * s.d_k * s.d_v
    d = s.d_k
    return T * s.h_v * (6.0 * CHUNK * d + 6.0 * d * s.d_v) + T * s.h_qk * 4.0 * CHUNK * d


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return {k: float(m[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# Sources of the kernels each workload's traffic figure belongs to.
KERNEL_SOURCES = {"decode": ("scan_simt.cu",), "prefill": ("prefill_tc.cu", "tc_ptx.cuh"),
                  "neighbours": ("neighbours.cu",), "layer": ("layer_decode.cu",)}


def source_digest(kind: str = "prefill") -> str:
    """Hash of the kernel sources behind `kind` ("decode" or "prefill")."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "recurrent_state_scan_gb300", "csrc")
    for fn in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kind: str):
    """DRAM bytes of one call from the committed ncu summary, or None when there is none
    or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256") != source_digest(kind):
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
                for name, val in zip(names, r[3:7]):
                    if val.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- distributed

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- CPU oracle timing

def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(inp, budget_s: float, min_reps: int = 1):
    """Run the oracle over the whole workload repeatedly for about budget_s seconds."""
    import oracle
    threads = cpu_threads()
    oracle.build()
    reps, t0 = 0, time.perf_counter()
    while True:
        if inp.pool is not None:
            oracle.slot_scan_inputs(inp, threads=threads)
        elif inp.spec.window:
            oracle.window_scan_inputs(inp, threads=threads)
        else:
            oracle.scan_inputs(inp, threads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if reps >= min_reps and el >= budget_s:
            break
        if el > 0 and reps >= min_reps and el / reps * (reps + 1) > 3 * budget_s:
            break
    return el / reps, reps, threads


def units_per_step(inp):
    return inp.total_tokens


def cpu_baseline_line(inp, budget_s=10.0):
    per, reps, threads = time_oracle(inp, budget_s)
    s = inp.spec
    if bandwidth_metric(s):
        val, unit = algorithmic_bytes(inp) / per / 1e9, "GB/s"
    else:
        val, unit = units_per_step(inp) / per, "tokens/s"
    return {"value": val, "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"the whole {s.name} workload x{reps} through the float64 C oracle "
                      f"({threads} threads over (sequence, head) units), {per * reps:.1f} s"}


# ---------------------------------------------------------------- neighbouring ops
#
# The causal convolution and the gated RMS norm are single HBM-bound kernels: a step is
# one call over the whole workload, measured in GB/s of algorithmic bytes (every input
# read once, every output written once).

def neighbour_io_bytes(inp) -> dict:
    if isinstance(inp, workloads.ConvInputs):
        s = inp.spec
        es = inp.x.element_size()
        n = inp.x.numel()
        carry = (s.kernel - 1) * s.dilation
        one = s.batch * carry * s.channels * es
        win = max(s.state_window, 1)
        return {"x": n * es, "y": n * es, "weight": inp.w.numel() * es,
                "bias": 0 if inp.bias is None else inp.bias.numel() * es,
                "state_in": one if (inp.state_in is not None or inp.pool is not None) else 0,
                "state_out": one * win, "slots": 0 if inp.slots is None else 4 * s.batch}
    es = inp.x.element_size()
    n = inp.x.numel()
    return {"x": n * es, "gate": n * es, "y": n * es, "scale": inp.scale.numel() * es}


def neighbour_oracle(inp):
    import oracle
    f = inp.f64
    if isinstance(inp, workloads.ConvInputs):
        s = inp.spec
        if inp.pool is not None:
            return oracle.conv_slots(f["x"], f["w"], f["pool"], inp.slots.numpy(), f["bias"],
                                     dilation=s.dilation, silu=s.silu)
        return oracle.causal_conv(f["x"], f["w"], f["bias"], f["state_in"], dilation=s.dilation,
                                  channels_last=s.channels_last, silu=s.silu,
                                  state_window=s.state_window)
    return oracle.gated_rmsnorm(f["x"], f["scale"], f["gate"], inp.spec.eps, inp.spec.activation)


def neighbour_sample(inp):
    """A bounded sample of a convolution workload for the CPU oracle: its first 512
    channels when the whole would take the oracle more than a second or so (the oracle
    walks each channel's tokens, a strided pass over x).  Returns (inputs, description)."""
    if not isinstance(inp, workloads.ConvInputs) or inp.x.numel() <= (1 << 24):
        return inp, f"the whole {inp.spec.name} workload"
    s = inp.spec
    c = min(512, s.channels)
    cut = lambda t: None if t is None else np.ascontiguousarray(t[..., :c])
    f = {n: cut(v) for n, v in inp.f64.items() if n != "w" and n != "bias"}
    f["w"] = inp.f64["w"][:c]
    f["bias"] = None if inp.f64["bias"] is None else inp.f64["bias"][:c]
    small = workloads.ConvInputs(
        spec=dataclasses.replace(s, channels=c),
        x=inp.x[..., :c].contiguous(), w=inp.w[:c].contiguous(),
        bias=None if inp.bias is None else inp.bias[:c].contiguous(),
        state_in=None if inp.state_in is None else inp.state_in[..., :c].contiguous(),
        pool=None if inp.pool is None else inp.pool[..., :c].contiguous(),
        slots=inp.slots, f64=f)
    return small, f"the first {c} of {s.channels} channels of {s.name} (all rows and tokens)"


def time_neighbour_oracle(inp, budget_s: float, min_reps: int = 1):
    import oracle
    oracle.build()
    reps, t0 = 0, time.perf_counter()
    while True:
        neighbour_oracle(inp)
        reps += 1
        el = time.perf_counter() - t0
        if reps >= min_reps and el >= budget_s:
            break
    return el / reps, reps, 1


def neighbour_config(inp, world):
    s = inp.spec
    c = {"workload": s.name, "io_dtype": s.io, "l2": "flushed before every step (256 MiB write, untimed)",
         "parallelism": f"replicas: the full workload on each of {world} GPU(s), no collective"}
    if isinstance(inp, workloads.ConvInputs):
        c.update({"op": "causal depthwise conv with carried state", "batch": s.batch,
                  "seq_len": s.seqlen, "channels": s.channels, "kernel": s.kernel,
                  "dilation": s.dilation, "activation": "silu" if s.silu else "none",
                  "layout": "channels last" if s.channels_last else "channels first",
                  "past_state": "N(0,%g)" % s.state_std if s.state_std else "zero",
                  "state_update": "in place" if s.decode else "separate present state"})
    else:
        c.update({"op": "gated RMS norm", "shape": list(s.shape), "eps": s.eps,
                  "activation": s.activation})
    return c


def main_neighbour(args, rank, world, local):
    inp = workloads.any_workload(args.workload)
    nbytes = int(sum(neighbour_io_bytes(inp).values()))
    conv = isinstance(inp, workloads.ConvInputs)
    s = inp.spec
    if args.impl == "reference":
        if rank != 0:
            return
        sample, what = neighbour_sample(inp)
        sbytes = int(sum(neighbour_io_bytes(sample).values()))
        for _ in range(args.warmup):
            time_neighbour_oracle(sample, 0.0)
        per, reps, threads = time_neighbour_oracle(sample, 0.0, min_reps=args.steps)
        value = sbytes / per / 1e9
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": neighbour_config(inp, world),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{what} per step, {reps} steps"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return

    from recurrent_state_scan_gb300 import (gdn_causal_conv, gdn_causal_conv_slots,
                                            gdn_gated_rmsnorm, load)
    load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    if conv:
        names = [("x", inp.x), ("w", inp.w), ("bias", inp.bias), ("state", inp.state_in),
                 ("pool", inp.pool), ("slots", inp.slots)]
    else:
        names = [("x", inp.x), ("scale", inp.scale), ("gate", inp.gate)]
    t = {n: v.to(dev) for n, v in names if v is not None}
    y = torch.empty_like(t["x"])
    act = ("silu" if s.silu else "none") if conv else s.activation
    st_out = None
    if conv and inp.pool is None and not s.decode:
        from recurrent_state_scan_gb300 import gdn
        st_out = torch.empty(gdn.conv_state_shape(s.batch, s.channels, s.kernel, s.dilation,
                                                  s.channels_last, s.state_window),
                             dtype=t["x"].dtype, device=dev)

    def call(d):
        if not conv:
            gdn_gated_rmsnorm(d["x"], d["scale"], d["gate"], s.eps, act, y=y, stream=stream)
        elif "pool" in d:
            gdn_causal_conv_slots(d["x"], d["w"], d["pool"], d["slots"], d.get("bias"),
                                  dilation=s.dilation, activation=act, y=y, stream=stream)
        else:
            gdn_causal_conv(d["x"], d["w"], d.get("bias"), d.get("state"), dilation=s.dilation,
                            channels_last=s.channels_last, activation=act,
                            state_window=s.state_window, y=y,
                            state_out=d.get("state") if s.decode else st_out, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        call(t)
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        call(t)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in zip(starts, ends)])), world)

    e2e = None
    if not args.no_e2e:
        # Pinned host inputs -> device -> call -> y (and the state, unless it lives in a
        # resident pool) back to the host.
        host = {n: v.pin_memory() for n, v in names if v is not None and n != "pool"}
        dbuf = {n: torch.empty_like(v, device=dev) for n, v in host.items()}
        if "pool" in t:
            dbuf["pool"] = t["pool"]
        y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        st_dev = (dbuf.get("state") if s.decode else st_out) if conv and "pool" not in t else None
        st_host = None if st_dev is None else torch.empty(st_dev.shape, dtype=st_dev.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = y_host.numel() * y_host.element_size() + \
            (0 if st_host is None else st_host.numel() * st_host.element_size())

        def e2e_step():
            for n, v in host.items():
                dbuf[n].copy_(v, non_blocking=True)
            call(dbuf)
            if st_host is not None:
                st_host.copy_(dbuf.get("state") if s.decode else st_out, non_blocking=True)
            y_host.copy_(y, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize(dev)
        es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier(world)
        for i in range(args.steps):
            flush.zero_()
            es[i].record(stream)
            e2e_step()
            ee[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        ems = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in zip(es, ee)])), world)
        e2e = {"value": world * nbytes / (ems / 1e3) / 1e9, "unit": "GB/s", "ms_per_step": ems,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    pk, pk_kind = peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    if conv:   # the kernel that takes the workload's shape (16-bit, channels last)
        kernel = ("gdn::causal_conv_decode_stream_kernel" if inp.spec.decode
                  else "gdn::causal_conv_tma_kernel")
    else:
        kernel = "gdn::gated_rmsnorm_rows_kernel"
    line = {
        "metric": METRIC, "value": world * gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": neighbour_config(inp, world),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"],
                     "traffic": profiled_traffic(args.workload, "neighbours"),
                     "peak_source": f"{pk_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                     if pk_kind == "measured" else "fallback 6.8 TB/s",
                     "kernels": kernel},
        "gpu_launches": args.steps,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if clocks is not None:
        line["clocks"] = clocks
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample, what = neighbour_sample(inp)
        per, reps, threads = time_neighbour_oracle(sample, 10.0)
        line["cpu_baseline"] = {
            "value": sum(neighbour_io_bytes(sample).values()) / per / 1e9, "unit": "GB/s",
            "cores": threads, "kind": "oracle",
            "sample": f"{what} x{reps} through the float64 C oracle (one thread), "
                      f"{per * reps:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- the fused layer step
#
# One decode token of the whole layer (conv -> step -> gated norm) in one call.  A step is
# one gdn_decode_layer call; its bytes are every input read once and every output written
# once, the recurrent state both ways.

def layer_io_bytes(inp) -> dict:
    s = inp.spec
    es = inp.x.element_size()
    B, C, K = s.batch, inp.x.shape[2], s.kernel
    return {"x": B * C * es, "conv_weight": C * K * es, "conv_bias": 0 if inp.bias is None else C * es,
            "conv_state_in": B * (K - 1) * C * es, "conv_state_out": B * (K - 1) * C * es,
            "a": B * s.h_v * es, "b": B * s.h_v * es, "A_log": 4 * s.h_v, "dt_bias": 4 * s.h_v,
            "state": 2 * B * s.h_v * 128 * s.d_v * 4, "norm_scale": s.d_v * es,
            "gate": B * s.h_v * s.d_v * es, "y": B * s.h_v * s.d_v * es}


def layer_oracle(inp, rows: int):
    """The float64 oracle chain on the first `rows` sequences: conv -> step -> gated norm."""
    import oracle
    s, f = inp.spec, inp.f64
    B, dqk = rows, s.h_qk * 128
    yc, _ = oracle.causal_conv(f["x"][:B], f["w"], f["bias"], f["conv_state"][:B], silu=True)
    q = yc[:, 0, :dqk].reshape(B, s.h_qk, 128)
    k = yc[:, 0, dqk:2 * dqk].reshape(B, s.h_qk, 128)
    v = yc[:, 0, 2 * dqk:].reshape(B, s.h_v, s.d_v)
    o, _ = oracle.scan(np.arange(B + 1), s.h_qk, s.h_v, 128, s.d_v, q, k, v,
                       a=f["a"][:B].reshape(B, s.h_v), b=f["b"][:B].reshape(B, s.h_v),
                       A_log=f["A_log"], dt_bias=f["dt_bias"], state_in=f["state"][:B],
                       threads=cpu_threads())
    oracle.gated_rmsnorm(o.reshape(B, 1, s.h_v, s.d_v), f["norm_scale"], f["gate"][:B], eps=s.eps)


def time_layer_oracle(inp, budget_s: float, min_reps: int = 1):
    rows = max(1, inp.spec.batch // 8)
    reps, t0 = 0, time.perf_counter()
    while reps < min_reps or time.perf_counter() - t0 < budget_s:
        layer_oracle(inp, rows)
        reps += 1
    return (time.perf_counter() - t0) / reps, reps, rows


def layer_config(inp, world):
    s = inp.spec
    return {"workload": s.name, "io_dtype": s.io, "op": "decode token of the layer: causal conv "
            "(silu) over [q | k | v] channels -> gated delta-rule step -> gated RMS norm (silu)",
            "batch": s.batch, "h_qk": s.h_qk, "h_v": s.h_v, "d_k": 128, "d_v": s.d_v,
            "conv_kernel": s.kernel, "state": "fp32, in place", "conv_state": "two buffers, alternating",
            "l2": "flushed before every step (256 MiB write, untimed)",
            "parallelism": f"replicas: the full workload on each of {world} GPU(s), no collective"}


def main_layer(args, rank, world, local):
    inp = workloads.any_workload(args.workload)
    s = inp.spec
    nbytes = int(sum(layer_io_bytes(inp).values()))
    if args.impl == "reference":
        if rank != 0:
            return
        for _ in range(args.warmup):
            time_layer_oracle(inp, 0.0)
        per, reps, rows = time_layer_oracle(inp, 0.0, min_reps=args.steps)
        value = nbytes * rows / s.batch / per / 1e9
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": layer_config(inp, world),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": f"the first {rows} of {s.batch} sequences per step, {reps} steps"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return

    from recurrent_state_scan_gb300 import (gdn_causal_conv, gdn_decode_layer, gdn_decode_step,
                                            gdn_gated_rmsnorm, load)
    load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    names = ("x", "w", "bias", "conv_state", "a", "b", "A_log", "dt_bias", "state", "norm_scale", "gate")
    t = {n: getattr(inp, n).to(dev) for n in names if getattr(inp, n) is not None}
    cs = [t["conv_state"], torch.empty_like(t["conv_state"])]
    y = torch.empty((s.batch, 1, s.h_v, s.d_v), dtype=t["x"].dtype, device=dev)
    step_no = [0]

    def call(d):
        i = step_no[0] % 2
        step_no[0] += 1
        gdn_decode_layer(d["x"], d["w"], d.get("bias"), cs[i], cs[1 - i], d["a"], d["b"], d["A_log"],
                         d["dt_bias"], d["state"], d["norm_scale"], d["gate"], h_qk=s.h_qk, h_v=s.h_v,
                         eps=s.eps, y=y, stream=stream)

    dqk = s.h_qk * 128

    def separate(d):
        # The same token through the separate calls: conv, the q / k / v cut, step, norm.
        i = step_no[0] % 2
        step_no[0] += 1
        yc, _ = gdn_causal_conv(d["x"], d["w"], d.get("bias"), cs[i], activation="silu",
                                state_out=cs[1 - i], stream=stream)
        q = yc[:, :, :dqk].reshape(s.batch, 1, s.h_qk, 128).contiguous()
        k = yc[:, :, dqk:2 * dqk].reshape(s.batch, 1, s.h_qk, 128).contiguous()
        v = yc[:, :, 2 * dqk:].reshape(s.batch, 1, s.h_v, s.d_v).contiguous()
        o = gdn_decode_step(q, k, v, d["a"], d["b"], d["A_log"], d["dt_bias"], d["state"], stream=stream)
        gdn_gated_rmsnorm(o, d["norm_scale"], d["gate"], s.eps, y=y, stream=stream)

    def timed(fn, d):
        for _ in range(args.warmup):
            flush.zero_()
            fn(d)
        torch.cuda.synchronize(dev)
        st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.zero_()
            st[i].record(stream)
            fn(d)
            en[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in zip(st, en)])), world)

    sampler = ClockSampler(local) if rank == 0 else None
    ms = timed(call, t)
    clocks = sampler.stop() if sampler else None
    ms_sep = timed(separate, t)

    e2e = None
    if not args.no_e2e:
        # Pinned host inputs of the token (x, a, b, gate) in, y out; the recurrent state,
        # the conv states and the weights stay resident.
        host = {n: getattr(inp, n).pin_memory() for n in ("x", "a", "b", "gate")}
        dbuf = dict(t)
        for n, v in host.items():
            dbuf[n] = torch.empty_like(v, device=dev)
        y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = y_host.numel() * y_host.element_size()

        def e2e_step(d):
            for n, v in host.items():
                d[n].copy_(v, non_blocking=True)
            call(d)
            y_host.copy_(y, non_blocking=True)

        ems = timed(e2e_step, dbuf)
        e2e = {"value": world * nbytes / (ems / 1e3) / 1e9, "unit": "GB/s", "ms_per_step": ems,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    pk, pk_kind = peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": world * gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": layer_config(inp, world),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "traffic": profiled_traffic(args.workload, "layer"),
                     "peak_source": f"{pk_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                     if pk_kind == "measured" else "fallback 6.8 TB/s",
                     "kernels": "gdn::decode_layer_kernel"},
        "separate_calls": {"ms_per_step": ms_sep, "launches": 6,
                           "calls": "gdn_causal_conv, three q/k/v slice copies, gdn_decode_step, "
                                    "gdn_gated_rmsnorm"},
        "gpu_launches": args.steps,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if clocks is not None:
        line["clocks"] = clocks
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        per, reps, rows = time_layer_oracle(inp, 10.0)
        line["cpu_baseline"] = {"value": nbytes * rows / s.batch / per / 1e9, "unit": "GB/s",
                                "cores": cpu_threads(), "kind": "oracle",
                                "sample": f"the first {rows} of {s.batch} sequences x{reps} through the "
                                          f"float64 C oracle chain, {per * reps:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- prefill + gated norm

def prefill_norm_io_bytes(inp) -> dict:
    """The prefill's bytes with o replaced by y, plus the gate and the norm scale."""
    p = inp.prefill
    b = io_bytes(p)
    es = p.v.element_size()
    y = b.pop("o")
    return dict(b, gate=y, y=y, norm_scale=p.spec.d_v * es)


def prefill_norm_oracle(inp, tokens: int):
    """The float64 oracle chain over the first sequences that hold `tokens` tokens: the
    scan, o rounded to the I/O type, the gated RMS norm.  Returns the tokens covered."""
    import oracle
    p, s = inp.prefill, inp.prefill.spec
    cu = [int(c) for c in p.cu_seqlens]
    n = 1
    while n < p.n_seq and cu[n] < tokens:
        n += 1
    T = int(cu[n])
    f = {k: v for k, v in ((k, getattr(p, k)) for k in ("q", "k", "v", "a", "b"))}
    q = f["q"].reshape(-1, s.h_qk, s.d_k)[:T].double().numpy()
    k = f["k"].reshape(-1, s.h_qk, s.d_k)[:T].double().numpy()
    v = f["v"].reshape(-1, s.h_v, s.d_v)[:T].double().numpy()
    a = f["a"].reshape(-1, s.h_v)[:T].double().numpy()
    b = f["b"].reshape(-1, s.h_v)[:T].double().numpy()
    st = None if p.state_in is None else p.state_in[:n].double().numpy()
    o, _ = oracle.scan(np.asarray(cu[:n + 1]), s.h_qk, s.h_v, s.d_k, s.d_v, q, k, v, a=a, b=b,
                       A_log=p.A_log.double().numpy(), dt_bias=p.dt_bias.double().numpy(),
                       state_in=st, scale=p.scale, threads=cpu_threads())
    o_io = torch.from_numpy(np.ascontiguousarray(o)).to(p.v.dtype).double().numpy()
    g = inp.gate.reshape(-1, s.h_v, s.d_v)[:T].double().numpy()
    oracle.gated_rmsnorm(o_io.reshape(-1, s.d_v), inp.norm_scale.double().numpy(),
                         g.reshape(-1, s.d_v), inp.spec.eps, inp.spec.activation)
    return T


def time_prefill_norm_oracle(inp, budget_s: float, min_reps: int = 1, tokens: int = 4096):
    reps, t0, done = 0, time.perf_counter(), 0
    while reps < min_reps or time.perf_counter() - t0 < budget_s:
        done = prefill_norm_oracle(inp, tokens)
        reps += 1
    return (time.perf_counter() - t0) / reps, reps, done


def main_prefill_norm(args, rank, world, local):
    inp = workloads.any_workload(args.workload)
    p, s = inp.prefill, inp.prefill.spec
    nbytes = int(sum(prefill_norm_io_bytes(inp).values()))
    config = dict(config_of(p, world), workload=inp.spec.name,
                  op="packed prefill, then the gated RMS norm (silu gate) of each head's "
                     "output row: gdn_prefill_norm (the norm in place on y)",
                  norm={"eps": inp.spec.eps, "activation": inp.spec.activation})
    if args.impl == "reference":
        if rank != 0:
            return
        for _ in range(args.warmup):
            time_prefill_norm_oracle(inp, 0.0)
        per, reps, done = time_prefill_norm_oracle(inp, 0.0, min_reps=args.steps)
        value = done / per
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(),
                             "kind": "oracle",
                             "sample": f"the first {done} of {p.total_tokens} tokens per step "
                                       f"(whole sequences), {reps} steps"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return

    from recurrent_state_scan_gb300 import (gdn, gdn_gated_rmsnorm, gdn_prefill, gdn_prefill_norm,
                                            load)
    load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    t = {n: getattr(p, n).to(dev) for n in ("q", "k", "v", "a", "b", "A_log", "dt_bias")}
    t["gate"], t["norm_scale"] = inp.gate.to(dev), inp.norm_scale.to(dev)
    state0 = None if p.state_in is None else p.state_in.to(dev)
    cu = torch.tensor(p.cu_seqlens, dtype=torch.int32, device=dev) if p.varlen else None
    y = torch.empty(t["v"].shape, dtype=t["v"].dtype, device=dev)
    o = torch.empty_like(y)
    state_out = torch.empty((p.n_seq, s.h_v, s.d_k, s.d_v), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, gdn.gdn_prefill_workspace_bytes(gdn.shape_of_spec(s, p.n_seq,
                                                                               p.total_tokens))),
                     dtype=torch.uint8, device=dev)
    eps, act = inp.spec.eps, inp.spec.activation

    def call(d, fuse=False):
        gdn_prefill_norm(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], state0,
                         cu, p.scale, norm_scale=d["norm_scale"], gate=d["gate"], eps=eps,
                         activation=act, fuse=fuse, y=y, state_out=state_out, workspace=ws,
                         stream=stream)

    def fused(d):
        call(d, fuse=True)

    def separate(d):
        gdn_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], state0, cu,
                    p.scale, o=o, state_out=state_out, workspace=ws, stream=stream)
        gdn_gated_rmsnorm(o, d["norm_scale"], d["gate"], eps, act, y=y, stream=stream)

    def timed(fn, d):
        for _ in range(args.warmup):
            flush.zero_()
            fn(d)
        torch.cuda.synchronize(dev)
        st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.zero_()
            st[i].record(stream)
            fn(d)
            en[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in zip(st, en)])), world)

    sampler = ClockSampler(local) if rank == 0 else None
    ms = timed(call, t)
    clocks = sampler.stop() if sampler else None
    ms_sep = timed(separate, t)
    ms_fused = timed(fused, t)

    e2e = None
    if not args.no_e2e:
        # Pinned host inputs (q, k, v, a, b, the gate) in, y and the state out.
        host = {n: getattr(p, n).pin_memory() for n in ("q", "k", "v", "a", "b")}
        host["gate"] = inp.gate.pin_memory()
        dbuf = dict(t)
        for n, v in host.items():
            dbuf[n] = torch.empty_like(v, device=dev)
        y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        s_host = torch.empty(state_out.shape, dtype=torch.float32).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = y_host.numel() * y_host.element_size() + s_host.numel() * 4

        def e2e_step(d):
            for n, v in host.items():
                d[n].copy_(v, non_blocking=True)
            call(d)
            y_host.copy_(y, non_blocking=True)
            s_host.copy_(state_out, non_blocking=True)

        ems = timed(e2e_step, dbuf)
        e2e = {"value": world * p.total_tokens / (ems / 1e3), "unit": "tokens/s",
               "ms_per_step": ems, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    pk, pk_kind = peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": world * p.total_tokens / (ms / 1e3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(p),
        "data": "synthetic", "config": config,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"],
                     "traffic": profiled_traffic(args.workload, "prefill"),
                     "peak_source": f"{pk_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                     if pk_kind == "measured" else "fallback 6.8 TB/s",
                     "kernels": "gdn_chunk_prep + gdn_chunk_scan + gated_rmsnorm_rows_kernel, one call"},
        "separate_calls": {"ms_per_step": ms_sep, "launches": 3,
                           "calls": "gdn_prefill (prep, scan), gdn_gated_rmsnorm"},
        "fused_readout": {"ms_per_step": ms_fused, "launches": 2,
                          "kernels": "gdn_chunk_prep + gdn_chunk_scan with the norm (cluster pairs)"},
        "gpu_launches": args.steps * 3,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if clocks is not None:
        line["clocks"] = clocks
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        per, reps, done = time_prefill_norm_oracle(inp, 10.0)
        line["cpu_baseline"] = {"value": done / per, "unit": "tokens/s", "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": f"the first {done} of {p.total_tokens} tokens (whole "
                                          f"sequences) x{reps} through the float64 C oracle "
                                          f"chain, {per * reps:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def prefill_layer_io_bytes(inp) -> dict:
    """One layer prefill: x, the conv's weight, bias and states, a, b, the gate parameters,
    the recurrent states, the norm's scale and gate, and y, each once."""
    s = inp.spec
    es = inp.x.element_size()
    T, N, K = inp.total_tokens, inp.n_seq, s.kernel
    C = inp.x.shape[-1]
    st = N * s.h_v * 128 * 128 * 4
    y = T * s.h_v * 128 * es
    return {"x": T * C * es, "conv_weight": C * K * es, "conv_bias": C * es if inp.bias is not None else 0,
            "conv_state_in": N * (K - 1) * C * es, "conv_state_out": N * (K - 1) * C * es,
            "a": T * s.h_v * es, "b": T * s.h_v * es, "params": 2 * s.h_v * 4,
            "state_in": st if inp.state_in is not None else 0, "state_out": st,
            "norm_scale": 128 * es, "gate": y, "y": y}


def prefill_layer_oracle(inp, tokens: int):
    """The float64 oracle chain over the first sequences that hold `tokens` tokens: the
    convolution per sequence, its output rounded to the I/O type, the scan, o rounded, the
    gated RMS norm.  Returns the tokens covered."""
    import oracle
    s, cu = inp.spec, [int(c) for c in inp.cu_seqlens]
    n = 1
    while n < inp.n_seq and cu[n] < tokens:
        n += 1
    T = cu[n]
    C = inp.x.shape[-1]
    x = inp.x.reshape(-1, C)[:T].double().numpy()
    w = inp.w.double().numpy()
    bias = None if inp.bias is None else inp.bias.double().numpy()
    cs = inp.conv_state.double().numpy()
    yc = np.zeros_like(x)
    for i in range(n):
        if cu[i + 1] > cu[i]:
            yc[cu[i]:cu[i + 1]] = oracle.causal_conv(x[cu[i]:cu[i + 1]][None], w, bias, cs[i][None],
                                                     silu=s.silu)[0][0]
    yc = torch.from_numpy(yc).to(inp.x.dtype).double().numpy()
    hk = s.h_qk * 128
    st = None if inp.state_in is None else inp.state_in[:n].double().numpy()
    o, _ = oracle.scan(np.asarray(cu[:n + 1]), s.h_qk, s.h_v, 128, 128, yc[:, :hk], yc[:, hk:2 * hk],
                       yc[:, 2 * hk:], a=inp.a.reshape(-1, s.h_v)[:T].double().numpy(),
                       b=inp.b.reshape(-1, s.h_v)[:T].double().numpy(), A_log=inp.A_log.double().numpy(),
                       dt_bias=inp.dt_bias.double().numpy(), state_in=st, scale=inp.scale,
                       threads=cpu_threads())
    o_io = torch.from_numpy(np.ascontiguousarray(o)).to(inp.x.dtype).double().numpy()
    g = inp.gate.reshape(-1, 128)[:T * s.h_v].double().numpy()
    oracle.gated_rmsnorm(o_io.reshape(-1, 128), inp.norm_scale.double().numpy(), g, s.eps, s.activation)
    return T


def time_prefill_layer_oracle(inp, budget_s: float, min_reps: int = 1, tokens: int = 4096):
    reps, t0, done = 0, time.perf_counter(), 0
    while reps < min_reps or time.perf_counter() - t0 < budget_s:
        done = prefill_layer_oracle(inp, tokens)
        reps += 1
    return (time.perf_counter() - t0) / reps, reps, done


def main_prefill_layer(args, rank, world, local):
    inp = workloads.any_workload(args.workload)
    s = inp.spec
    nbytes = int(sum(prefill_layer_io_bytes(inp).values()))
    C = inp.x.shape[-1]
    config = {"workload": s.name, "io_dtype": s.io, "num_seqs": inp.n_seq, "total_tokens": inp.total_tokens,
              "h_qk": s.h_qk, "h_v": s.h_v, "d_k": 128, "d_v": 128, "channels": C,
              "conv": {"kernel": s.kernel, "bias": inp.bias is not None, "activation": "silu" if s.silu else "none"},
              "norm": {"eps": s.eps, "activation": s.activation},
              "l2": "flushed before every step (256 MiB write, untimed)",
              "parallelism": f"replicas: the full workload on each of {world} GPU(s), no collective",
              "op": "layer prefill: causal conv of the mixed input (a streaming pass), the gated "
                    "delta-rule prefill, the gated RMS norm of o: gdn_prefill_layer"}
    if args.impl == "reference":
        if rank != 0:
            return
        for _ in range(args.warmup):
            time_prefill_layer_oracle(inp, 0.0)
        per, reps, done = time_prefill_layer_oracle(inp, 0.0, min_reps=args.steps)
        value = done / per
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": f"the first {done} of {inp.total_tokens} tokens per step "
                                       f"(whole sequences), {reps} steps"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return

    from recurrent_state_scan_gb300 import (gdn, gdn_causal_conv, gdn_gated_rmsnorm, gdn_prefill,
                                            gdn_prefill_layer, load)
    load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    names = ("x", "w", "bias", "conv_state", "a", "b", "A_log", "dt_bias", "norm_scale", "gate")
    t = {n: (None if getattr(inp, n) is None else getattr(inp, n).to(dev)) for n in names}
    state0 = None if inp.state_in is None else inp.state_in.to(dev)
    cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device=dev) if inp.varlen else None
    T, N = inp.total_tokens, inp.n_seq
    y = torch.empty(tuple(inp.x.shape[:2]) + (s.h_v, 128), dtype=inp.x.dtype, device=dev)
    state_out = torch.empty((N, s.h_v, 128, 128), dtype=torch.float32, device=dev)
    cs_out = torch.empty((N, s.kernel - 1, C), dtype=inp.x.dtype, device=dev)
    shape = gdn.make_shape(gdn._DTYPE_CODE[inp.x.dtype], 1 if inp.varlen else inp.x.shape[0],
                           T if inp.varlen else inp.x.shape[1], N, s.h_qk, s.h_v, 128, 128)
    ws = torch.empty(max(1, gdn.gdn_prefill_layer_workspace_bytes(shape)), dtype=torch.uint8, device=dev)
    act = "silu" if s.silu else "none"

    def call(d, fuse=False):
        gdn_prefill_layer(d["x"], d["w"], d["bias"], d["conv_state"], d["a"], d["b"], d["A_log"],
                          d["dt_bias"], state0, cu, d["norm_scale"], d["gate"], h_qk=s.h_qk, h_v=s.h_v,
                          scale=inp.scale, conv_activation=act, norm_activation=s.activation, eps=s.eps,
                          fuse=fuse, y=y, state_out=state_out, conv_state_out=cs_out, workspace=ws,
                          stream=stream)

    def fused(d):
        call(d, fuse=True)

    # The separate calls: the conv per sequence (its kernel has no packed form) into q, k,
    # v buffers, the prefill, then the norm.
    hk = s.h_qk * 128
    qkv = torch.empty((T, C), dtype=inp.x.dtype, device=dev)
    q, k, v = (torch.empty((1, T, h, 128), dtype=inp.x.dtype, device=dev) for h in (s.h_qk, s.h_qk, s.h_v))
    o = torch.empty_like(y)
    ws2 = torch.empty(max(1, gdn.gdn_prefill_workspace_bytes(shape)), dtype=torch.uint8, device=dev)
    cuh = [int(c) for c in inp.cu_seqlens]

    def separate(d):
        x2 = d["x"].reshape(-1, C)
        for i in range(N):
            if cuh[i + 1] > cuh[i]:
                gdn_causal_conv(x2[cuh[i]:cuh[i + 1]][None], d["w"], d["bias"], d["conv_state"][i:i + 1],
                                activation=act, y=qkv[cuh[i]:cuh[i + 1]][None],
                                state_out=cs_out[i:i + 1], stream=stream)
        q.view(T, hk).copy_(qkv[:, :hk])
        k.view(T, hk).copy_(qkv[:, hk:2 * hk])
        v.view(T, -1).copy_(qkv[:, 2 * hk:])
        gdn_prefill(q, k, v, d["a"], d["b"], d["A_log"], d["dt_bias"], state0, cu, inp.scale, o=o,
                    state_out=state_out, workspace=ws2, stream=stream)
        gdn_gated_rmsnorm(o, d["norm_scale"], d["gate"], s.eps, s.activation, y=y, stream=stream)

    def timed(fn, d):
        for _ in range(args.warmup):
            flush.zero_()
            fn(d)
        torch.cuda.synchronize(dev)
        st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.zero_()
            st[i].record(stream)
            fn(d)
            en[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in zip(st, en)])), world)

    sampler = ClockSampler(local) if rank == 0 else None
    ms = timed(call, t)
    clocks = sampler.stop() if sampler else None
    ms_sep = timed(separate, t)
    ms_fused = timed(fused, t)

    e2e = None
    if not args.no_e2e:
        # Pinned host inputs (x, a, b, the gate) in; y, the state and the conv state out.
        host = {n: getattr(inp, n).pin_memory() for n in ("x", "a", "b", "gate")}
        dbuf = dict(t)
        for n, hv in host.items():
            dbuf[n] = torch.empty_like(hv, device=dev)
        y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        s_host = torch.empty(state_out.shape, dtype=torch.float32).pin_memory()
        c_host = torch.empty(cs_out.shape, dtype=cs_out.dtype).pin_memory()
        h2d = sum(hv.numel() * hv.element_size() for hv in host.values())
        d2h = sum(h.numel() * h.element_size() for h in (y_host, s_host, c_host))

        def e2e_step(d):
            for n, hv in host.items():
                d[n].copy_(hv, non_blocking=True)
            call(d)
            y_host.copy_(y, non_blocking=True)
            s_host.copy_(state_out, non_blocking=True)
            c_host.copy_(cs_out, non_blocking=True)

        ems = timed(e2e_step, dbuf)
        e2e = {"value": world * T / (ems / 1e3), "unit": "tokens/s", "ms_per_step": ems,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    pk, pk_kind = peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    launches = 4 + (1 if inp.varlen and s.kernel > 1 else 0)
    line = {
        "metric": METRIC, "value": world * T / (ms / 1e3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": s.io,
        "data": "synthetic", "config": config,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "traffic": profiled_traffic(args.workload, "prefill"),
                     "peak_source": f"{pk_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                     if pk_kind == "measured" else "fallback 6.8 TB/s",
                     "kernels": "conv_pass + gdn_chunk_prep + gdn_chunk_scan + conv_state_empty "
                                "+ gated_rmsnorm_rows_kernel, one call"},
        "conv_in_prep": {"ms_per_step": ms_fused, "launches": launches - 1,
                         "kernels": "gdn_chunk_prep (convolution form) + gdn_chunk_scan + conv_state_empty "
                                    "+ gated_rmsnorm_rows_kernel (fuse = 1)"},
        "separate_calls": {"ms_per_step": ms_sep,
                           "calls": f"gdn_causal_conv per sequence ({N}), q/k/v copies, gdn_prefill "
                                    "(prep, scan), gdn_gated_rmsnorm"},
        "gpu_launches": args.steps * launches,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if clocks is not None:
        line["clocks"] = clocks
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        per, reps, done = time_prefill_layer_oracle(inp, 10.0)
        line["cpu_baseline"] = {"value": done / per, "unit": "tokens/s", "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": f"the first {done} of {T} tokens (whole sequences) x{reps} "
                                          f"through the float64 C oracle chain, {per * reps:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local, name=None, with_e2e=True):
    from recurrent_state_scan_gb300 import (gdn_decode_step, gdn_decode_step_slots, gdn_prefill,
                                            gdn_prefill_variant, gdn_scan_variant, gdn_scan_window,
                                            load)
    load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = workloads.workload(name or args.workload)
    s = inp.spec
    t = {n: getattr(inp, n).to(dev) for n in ("q", "k", "v", "a", "b", "A_log", "dt_bias")}
    state0 = None if inp.state_in is None else inp.state_in.to(dev)
    cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device=dev) if inp.varlen else None
    o = torch.empty(t["v"].shape, dtype=t["v"].dtype, device=dev)
    n_state = (inp.n_seq, s.h_v, s.d_k, s.d_v)
    state_out = torch.empty(n_state, dtype=torch.float32, device=dev)
    work_state = None if state0 is None else state0.clone()
    # A state pool stays resident on the device, as a serving pool would.
    pool = None if inp.pool is None else inp.pool.to(dev)
    slots = None if inp.slots is None else inp.slots.to(dev)
    from recurrent_state_scan_gb300 import gdn
    window = None
    if s.window:
        window = torch.empty((s.window,) + n_state, dtype=torch.float32, device=dev)
    ws_need = 0 if (s.decode or s.window) else gdn.gdn_prefill_variant_workspace_bytes(
        gdn.shape_of_spec(s, inp.n_seq, inp.total_tokens), s.rule, s.decay_per_key, s.beta_shared)
    ws = torch.empty(ws_need, dtype=torch.uint8, device=dev) if ws_need else None
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    variant = s.decay_per_key or s.beta_shared or s.rule != "gated_delta"

    def step():
        if variant and not s.decode:
            # Prefill variants take gdn_prefill's path (per-key decay with its larger workspace).
            gdn_prefill_variant(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"],
                                state0, cu, inp.scale, rule=s.rule, decay_per_key=s.decay_per_key,
                                beta_shared=s.beta_shared, o=o, state_out=state_out, workspace=ws,
                                stream=stream)
        elif variant:
            # Decode steps update the state in place; prefill writes state_out.
            gdn_scan_variant(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"],
                             work_state if s.decode else state0, cu, inp.scale,
                             decay_per_key=s.decay_per_key, beta_shared=s.beta_shared, o=o,
                             state_out=work_state if s.decode else state_out, stream=stream)
        elif window is not None:
            gdn_scan_window(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"],
                            state0, inp.scale, window_len=s.window, o=o, window=window,
                            stream=stream)
        elif pool is not None:
            gdn_decode_step_slots(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"],
                                  t["dt_bias"], pool, slots, inp.scale, o=o, stream=stream)
        elif s.decode:
            gdn_decode_step(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"],
                            work_state, inp.scale, o=o, stream=stream)
        else:
            gdn_prefill(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"],
                        state0, cu, inp.scale, o=o, state_out=state_out, workspace=ws,
                        stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop() if sampler else None
    times_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = max_over_ranks(float(np.mean(times_ms)), world)

    # End to end through the public API: pinned host inputs -> device -> call -> host.
    e2e = None
    if with_e2e and not args.no_e2e:
        host = {n: v.pin_memory() for n, v in
                [("q", inp.q), ("k", inp.k), ("v", inp.v), ("a", inp.a), ("b", inp.b),
                 ("A_log", inp.A_log), ("dt_bias", inp.dt_bias)] +
                ([("state", inp.state_in)] if inp.state_in is not None else []) +
                ([("slots", inp.slots)] if inp.slots is not None else [])}
        o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        s_host = torch.empty(((s.window,) if s.window else ()) + n_state,
                             dtype=torch.float32).pin_memory()
        dbuf = {n: torch.empty_like(v, device=dev) for n, v in host.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        # With a resident pool only o comes back; otherwise o and the state.
        d2h = o_host.numel() * o_host.element_size() + (0 if pool is not None else s_host.numel() * 4)

        def e2e_step():
            for n, v in host.items():
                dbuf[n].copy_(v, non_blocking=True)
            if variant and not s.decode:
                gdn_prefill_variant(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["a"], dbuf["b"],
                                    dbuf["A_log"], dbuf["dt_bias"], dbuf.get("state"), cu, inp.scale,
                                    rule=s.rule, decay_per_key=s.decay_per_key,
                                    beta_shared=s.beta_shared, o=o, state_out=state_out,
                                    workspace=ws, stream=stream)
                s_host.copy_(state_out, non_blocking=True)
            elif variant:
                st_out = dbuf["state"] if s.decode else state_out
                gdn_scan_variant(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["a"], dbuf["b"],
                                 dbuf["A_log"], dbuf["dt_bias"], dbuf.get("state"), cu, inp.scale,
                                 decay_per_key=s.decay_per_key, beta_shared=s.beta_shared, o=o,
                                 state_out=st_out, stream=stream)
                s_host.copy_(st_out, non_blocking=True)
            elif window is not None:
                gdn_scan_window(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["a"], dbuf["b"],
                                dbuf["A_log"], dbuf["dt_bias"], dbuf.get("state"), inp.scale,
                                window_len=s.window, o=o, window=window, stream=stream)
                s_host.copy_(window, non_blocking=True)
            elif pool is not None:
                gdn_decode_step_slots(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["a"], dbuf["b"],
                                      dbuf["A_log"], dbuf["dt_bias"], pool, dbuf["slots"],
                                      inp.scale, o=o, stream=stream)
            elif s.decode:
                gdn_decode_step(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["a"], dbuf["b"],
                                dbuf["A_log"], dbuf["dt_bias"], dbuf["state"], inp.scale, o=o,
                                stream=stream)
                s_host.copy_(dbuf["state"], non_blocking=True)
            else:
                gdn_prefill(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["a"], dbuf["b"], dbuf["A_log"],
                            dbuf["dt_bias"], dbuf.get("state"), cu, inp.scale, o=o,
                            state_out=state_out, workspace=ws, stream=stream)
                s_host.copy_(state_out, non_blocking=True)
            o_host.copy_(o, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize(dev)
        es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier(world)
        for i in range(args.steps):
            flush.zero_()
            es[i].record(stream)
            e2e_step()
            ee[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        ems = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in zip(es, ee)])), world)
        e2e = {"ms_per_step": ems, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    return inp, ms, times_ms, clocks, e2e


def main():
    args = parse_args()
    rank, world, local = dist_init()
    inp_name = args.workload
    if inp_name in workloads.LAYER_WORKLOADS:
        return main_layer(args, rank, world, local)
    if inp_name in workloads.PREFILL_NORM_WORKLOADS:
        return main_prefill_norm(args, rank, world, local)
    if inp_name in workloads.PREFILL_LAYER_WORKLOADS:
        return main_prefill_layer(args, rank, world, local)
    if inp_name not in workloads.WORKLOADS:
        return main_neighbour(args, rank, world, local)
    if args.impl == "reference":
        # The reference arm is the CPU oracle, timed as it stands, on rank 0 only.
        if rank != 0:
            return
        inp = workloads.workload(inp_name)
        s = inp.spec
        for _ in range(args.warmup):
            time_oracle(inp, 0.0)
        per, reps, threads = time_oracle(inp, 0.0, min_reps=args.steps)
        if bandwidth_metric(s):
            value, unit = algorithmic_bytes(inp) / per / 1e9, "GB/s"
        else:
            value, unit = inp.total_tokens / per, "tokens/s"
        line = {
            "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(inp, world),
            "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                             "sample": f"the whole {s.name} workload per step, {reps} steps"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return

    inp, ms, times_ms, clocks, e2e = run_ours(args, rank, world, local)
    s = inp.spec
    nbytes = algorithmic_bytes(inp)
    value, unit = throughput(inp, ms, world)
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype_of(inp), "data": "synthetic",
        "config": config_of(inp, world), "roofline": roofline_entry(inp, ms),
        "gpu_launches": args.steps * launches_per_call(inp),
    }
    if e2e is not None:
        esec = e2e["ms_per_step"] / 1e3
        ev = world * (nbytes / esec / 1e9 if bandwidth_metric(s) else inp.total_tokens / esec)
        line["e2e"] = {"value": ev, "unit": unit, "ms_per_step": e2e["ms_per_step"],
                       "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                       "d2h_bytes_per_step": e2e["d2h_bytes_per_step"]}
    if clocks is not None:
        line["clocks"] = clocks
    if not args.no_extra_configs and inp_name == DEFAULT_WORKLOAD:
        # The other full-size workloads, each timed like the main one (no e2e leg).
        extra = {}
        for name in EXTRA_WORKLOADS:
            if name == inp_name:
                continue
            x_inp, x_ms, _, x_clocks, _ = run_ours(args, rank, world, local, name=name,
                                                   with_e2e=False)
            x_val, x_unit = throughput(x_inp, x_ms, world)
            extra[name] = {"value": x_val, "unit": x_unit, "ms_per_step": x_ms,
                           "dtype": dtype_of(x_inp), "config": config_of(x_inp, world),
                           "roofline": roofline_entry(x_inp, x_ms),
                           "gpu_launches": args.steps * launches_per_call(x_inp)}
            if x_clocks is not None:
                extra[name]["clocks"] = x_clocks
        line["configs"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_line(inp)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def throughput(inp, ms, world):
    """(value, unit) of one step: state GB/s for decode-like steps, tokens/s for prefill,
    summed over the ranks (each runs its own copy of the workload)."""
    sec = ms / 1e3
    if bandwidth_metric(inp.spec):
        return world * algorithmic_bytes(inp) / sec / 1e9, "GB/s"
    return world * inp.total_tokens / sec, "tokens/s"


def roofline_entry(inp, ms):
    """Roofline of one call on one GPU: algorithmic bytes (and, for prefill, FLOPs) over
    the call's device time, against the measured peaks."""
    s = inp.spec
    pk, pk_kind = peaks()
    nbytes = algorithmic_bytes(inp)
    flops = algorithmic_flops(inp)
    sec = ms / 1e3
    gbs = nbytes / sec / 1e9
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    roof = {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / pk["hbm_gbs"],
            "traffic": profiled_traffic(s.name, "decode" if bandwidth_metric(s) else "prefill"),
            "peak_source": f"{pk_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)"
            if pk_kind == "measured" else "fallback 6.8 TB/s",
            "kernels": prefill_kernels(inp)}
    if not bandwidth_metric(s):
        tfs = flops / sec / 1e12
        roof["tensor_tflops"] = tfs
        roof["tensor_frac_of_bf16_peak"] = tfs / pk["bf16_tflops"]
        roof["roofline_time_us"] = max(t_hbm, t_tc) * 1e6
        roof["frac_of_roofline"] = max(t_hbm, t_tc) / sec
    return roof


def prefill_kernels(inp) -> str:
    """The kernels one call runs, named for the roofline entry."""
    from recurrent_state_scan_gb300 import gdn
    if bandwidth_metric(inp.spec):
        if inp.spec.window:
            return "scan_simt_kernel, one call"
        return "decode_stream_kernel (persistent, prefetching), one call"
    s = inp.spec
    prep = "gdn_chunk_prep_pk (per-key-dim decay)" if s.decay_per_key else "gdn_chunk_prep"
    path, _ = gdn.gdn_prefill_variant_plan(gdn.shape_of_spec(s, inp.n_seq, inp.total_tokens),
                                           s.rule, s.decay_per_key, s.beta_shared)
    if path == gdn.PATH_TC_TP:
        return (f"{prep} + gdn_chunk_scan (time-parallel segments) + gdn_tp_combine "
                "+ gdn_tp_correct, one call")
    if path == gdn.PATH_TC:
        return f"{prep} + gdn_chunk_scan, one call"
    return "scan_simt, one call"


def dtype_of(inp) -> str:
    from recurrent_state_scan_gb300 import gdn
    return gdn.path_dtype(inp.spec, inp.n_seq, inp.total_tokens)


def launches_per_call(inp) -> int:
    from recurrent_state_scan_gb300 import gdn
    return gdn.launches_per_call(inp.spec, inp.n_seq, inp.total_tokens)


def config_of(inp, world):
    s = inp.spec
    c = {"workload": s.name, "io_dtype": s.io, "state_dtype": "f32", "num_seqs": inp.n_seq,
         "total_tokens": inp.total_tokens, "h_qk": s.h_qk, "h_v": s.h_v, "d_k": s.d_k,
         "d_v": s.d_v, "initial_state": "N(0,%g)" % s.state_std if s.state_std else "zero",
         "l2": "flushed before every step (256 MiB write, untimed)",
         "parallelism": f"replicas: the full workload on each of {world} GPU(s), no collective"}
    if inp.varlen:
        c["lengths"] = [int(x) for x in inp.lengths()]
    else:
        c["batch"], c["seq_len"] = s.batch, s.seqlen
    if s.decay_per_key or s.beta_shared or s.rule != "gated_delta":
        c["gates"] = {"decay": "per key dimension" if s.decay_per_key else "per head",
                      "beta": "shared by all heads" if s.beta_shared else "per head",
                      "rule": s.rule}
    if inp.pool is not None:
        c["initial_state"] = "pool of %d states, N(0,%g)" % (s.pool_size, s.pool_std)
        c["state_pool"] = {"entries": s.pool_size, "slots": "distinct, seeded permutation",
                           "resident": "on the device; e2e moves the step's q, k, v, a, b and "
                                       "slots in and o out"}
    return c


if __name__ == "__main__":
    main()
