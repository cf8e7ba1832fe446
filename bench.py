#!/usr/bin/env python
"""Benchmark of the EFLA token mixer on GB300.

Headline: chunked forward (efla_fwd) on the 340M-layer-shaped workload
B8 H8 L2048 dk=dv=128 chunk 64, bf16 q/k/v/o, fp32 beta and state, zero S0.
A step is one efla_fwd call over that batch; `value` is tokens (B*L) per second
summed over ranks.  The same line carries the decode-step bandwidth
(B256 H16 d128 fp32 state, 1024 steps) and the backward pass (B4 H16 L4096).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

--impl reference times the fp64 CPU oracle (the only other implementation of
the method available here) on the host cores, on a bounded sample of the same
workload, and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import efla_workloads as wl  # noqa: E402

METRIC = "EFLA chunked fwd tokens/s & TFLOP/s (B8 H8 L2048 d128) vs roofline; decode GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def _source_sha1(source: str) -> str:
    """SHA-1 over a kernel's source file and every header of the package that it includes,
    directly or through other headers (so that a change in shared device code, e.g. the
    chunk preparation that the fused forward inlines, invalidates the record too)."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "exact_flow_recurrence_gb300", "csrc")
    h, seen, todo = hashlib.sha1(), set(), [source]
    while todo:
        name = todo.pop(0)
        if name in seen or not os.path.exists(os.path.join(csrc, name)):
            continue
        seen.add(name)
        with open(os.path.join(csrc, name), "rb") as f:
            text = f.read()
        h.update(name.encode() + b"\0" + text)
        todo.extend(m.decode() for m in re.findall(rb'^\s*#include\s+"([^"]+)"', text, re.M))
    return h.hexdigest()


def measured_traffic(key: str):
    """DRAM bytes (read + write) per launch of one kernel on one workload, from the ncu
    capture recorded in profiles/dram_traffic.json under `key` (see record_traffic), or
    None when there is none or the kernel's source has changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            ent = json.load(f)["entries"][key]
        if _source_sha1(ent["source"]) != ent["source_sha1"]:
            return None
        return int(ent["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def record_traffic(csv_path: str, key: str, kernel_regex: str, source: str, command: str):
    """Write one entry of profiles/dram_traffic.json from an ncu CSV capture taken with
    --metrics dram__bytes_read.sum,dram__bytes_write.sum --print-units base --csv: the
    mean of read + write bytes over the captured launches whose name matches."""
    import csv
    import re
    per_launch = {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(f) if r]
    hdr_i = next(i for i, r in enumerate(rows) if "Metric Name" in r)
    hdr = rows[hdr_i]
    ci, ck, cm, cv = (hdr.index(c) for c in ("ID", "Kernel Name", "Metric Name", "Metric Value"))
    for r in rows[hdr_i + 1:]:
        if len(r) <= cv or not re.search(kernel_regex, r[ck]):
            continue
        if r[cm] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            per_launch[r[ci]] = per_launch.get(r[ci], 0.0) + float(r[cv].replace(",", ""))
    if not per_launch:
        raise SystemExit(f"no dram__bytes rows for /{kernel_regex}/ in {csv_path}")
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    except OSError:
        data = {"about": "DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch, "
                         "from ncu captures; an entry counts only while its source file and "
                         "the package headers it includes are unchanged (SHA-1)", "entries": {}}
    data["entries"][key] = {"source": source, "source_sha1": _source_sha1(source),
                            "dram_bytes_per_launch": int(round(sum(per_launch.values()) / len(per_launch))),
                            "launches_captured": len(per_launch), "command": command}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(data["entries"][key]))


def fwd_flops_per_token_head(dk, dv, C):
    # dense UT contractions: 6 dk dv + 2C(3 dk + 2 dv)
    return 6 * dk * dv + 2 * C * (3 * dk + 2 * dv)


def bwd_flops_per_token_head(dk, dv, C):
    return 16 * dk * dv + 2 * C * (10 * dk + 5 * dv) + 4 * C * C


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the GPU works."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        return self.summary()

    def summary(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in self.rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in self.rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        loaded = [s for s, p in zip(sm, pw) if p is not None and p > 250] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows),
                "power_w_max": max(pw) if pw else None}


# --------------------------------------------------------------- utilities
def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "gb300" and torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def profile_begin(lib):
    lib.efla_profile_begin()


def profile_end(lib):
    import ctypes
    cap = 32
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_float * cap)()
    cnt = (ctypes.c_int * cap)()
    lib.efla_profile_end.restype = ctypes.c_int
    lib.efla_profile_end.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                                     ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]
    n = lib.efla_profile_end(cap, names, ms, cnt)
    if n < 0:
        raise RuntimeError("efla_profile_end failed")
    return {names[i].decode(): {"total_ms": ms[i], "launches": cnt[i]} for i in range(n)}


def timed(fn, n, stream, flush=None):
    """Device time (ms) of each of n calls of fn, bracketed by CUDA events on `stream`
    (the stream the library launches on); L2 is flushed before each call when `flush`
    (a buffer larger than L2) is given.  No per-kernel instrumentation is on."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i, (a, b) in enumerate(evs):
        if flush is not None:
            flush.fill_(float(i))
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def kernel_split(lib, fn, n, stream, flush=None):
    """Per kernel: mean launch time (ms, from the library's own events on its stream) and
    launches per call, taken in a pass of its own so that the timed pass runs without
    this instrumentation."""
    profile_begin(lib)
    timed(fn, n, stream, flush)
    kern = profile_end(lib)
    return {k: {"ms": d["total_ms"] / d["launches"], "per_call": d["launches"] / n} for k, d in kern.items()}


def call_ms(split):
    return sum(d["ms"] * d["per_call"] for d in split.values())


def roofline_timing(split, share=0.9):
    """The kernel time a roofline is computed over: the dominant kernel's own launches when
    they carry at least `share` of the call's kernel time, else every kernel of the call.
    Returns (dominant kernel, time used in ms, whole call's kernel time in ms)."""
    path_ms = call_ms(split)
    dom = max(split, key=lambda n: split[n]["ms"] * split[n]["per_call"])
    dom_ms = split[dom]["ms"] * split[dom]["per_call"]
    return dom, (dom_ms if dom_ms >= share * path_ms else path_ms), path_ms


# ------------------------------------------------- the multi-rank pieces (CPU-testable)
def rank_seed(w, rank: int) -> int:
    """Every rank draws its own batch of the same workload (weak scaling)."""
    return w.index + rank


def headline_config(w, ws: int) -> dict:
    return {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "dk": w.dk, "dv": w.dv,
            "chunk": w.chunk, "global_batch": w.B * ws, "seq_len": w.L,
            "parallelism": "replicas" if ws == 1 else f"batch shards x{ws}, no collective",
            "io": "q,k,v,o bf16; beta, state fp32; S0 = 0",
            "l2": "flushed (256 MB write) before every timed step"}


def headline_value(ws: int, tokens_per_rank: int, step_ms_mean: float, device):
    """(ms per step, tokens/s): the slowest rank's mean step time; every rank's tokens."""
    ms = max_over_ranks(step_ms_mean, ws, device)
    return ms, ws * tokens_per_rank / (ms * 1e-3)


def bench_exact_vs_euler(efla, lib, x, o, Sf, wsp, C, flush, stream, tokens, rounds=3, steps=20):
    """The exact update against the delta rule (Euler mode, alpha := beta: DeltaNet's
    update) through the same kernels, buffers and timing, alternated `rounds` times: the
    pages' claim that the exact update costs what the delta rule costs, on this machine."""
    def fn(mode):
        return lambda: efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], None, chunk=C, o=o, S_final=Sf,
                                     workspace=wsp, mode=mode)
    ex, eu = fn(efla.EXACT), fn(efla.EULER)
    for f in (ex, eu, ex, eu, ex, eu):
        f()
    torch.cuda.synchronize()
    res = {"exact": [], "euler": []}
    for _ in range(rounds):
        res["exact"].append(statistics.mean(timed(ex, steps, stream, flush)))
        res["euler"].append(statistics.mean(timed(eu, steps, stream, flush)))
    kex, keu = kernel_split(lib, ex, 10, stream, flush), kernel_split(lib, eu, 10, stream, flush)
    mex, meu = statistics.mean(res["exact"]), statistics.mean(res["euler"])
    return {"workload": "the headline's, exact update vs Euler mode (delta rule), alternated",
            "rounds": rounds, "steps_per_round": steps,
            "exact_ms_per_step": [round(t, 4) for t in res["exact"]],
            "euler_ms_per_step": [round(t, 4) for t in res["euler"]],
            "exact_kernel_ms": round(call_ms(kex), 4), "euler_kernel_ms": round(call_ms(keu), 4),
            "euler_tokens_per_s": round(tokens / (meu * 1e-3), 1),
            "exact_over_euler_time": round(mex / meu, 4)}


def bench_stiff_long(efla, lib, dev, stream, pk, iters=5):
    """Few long sequences (B1 H16 L65536, the stiff law): the forward takes its
    segment-parallel form there; per-call time and the kernels it ran."""
    w = wl.STIFF_LONG
    B, H, L, dk, dv, C = w.B, w.H, w.L, w.dk, w.dv, w.chunk
    x = wl.fwd_inputs_device(w, dev)
    shape = efla.make_shape(B, H, L, dk, dv, C, torch.bfloat16, torch.bfloat16)
    wsp = torch.empty(efla.efla_fwd_workspace_size(shape), dtype=torch.uint8, device=dev)
    o = torch.empty((B, H, L, dv), dtype=torch.bfloat16, device=dev)
    Sf = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)

    def run():
        efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], None, chunk=C, o=o, S_final=Sf, workspace=wsp)
    for _ in range(3):
        run()
    torch.cuda.synchronize(dev)
    ms = statistics.mean(timed(run, iters, stream))   # inputs (268 MB per tensor) exceed the 129 MB L2
    split = kernel_split(lib, run, 2, stream)
    efla.efla_get_status()
    alg = B * H * L * (2 * dk + 2 * dk + 2 * dv + 4 + 2 * dv) + B * H * dk * dv * 4
    return {"workload": w.name, "ms": round(ms, 4), "tokens_per_s": round(B * L / (ms * 1e-3), 1),
            "form": "segment-parallel" if "efla_seg_combine" in split else "plain",
            "hbm_frac": round(alg / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "kernel_ms": {n: round(d["ms"], 4) for n, d in split.items()}}


# ----------------------------------------------------------- gb300 arm
def run_gb300(args, ws, rank, local):
    import exact_flow_recurrence_gb300 as efla
    from exact_flow_recurrence_gb300 import build as efla_build
    if not efla_build.up_to_date():
        efla_build.build()
    lib = efla.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk, pk_kind = peaks()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # > 129 MB L2
    if args.only_bwd:   # the backward leg alone (profiling its kernels); no headline line
        return {"bwd": bench_bwd(efla, lib, dev, stream, pk, pk_kind, flush, iters=max(args.steps, 1))}
    if args.only_decode:   # the decode leg alone; no headline line
        return {"decode": bench_decode(efla, lib, dev, stream, pk, pk_kind)}
    if args.only_stiff:   # the stiff long-context forward alone; no headline line
        return {"stiff_long_fwd": bench_stiff_long(efla, lib, dev, stream, pk, iters=max(args.steps, 1))}
    if args.only_mixer:   # the token mixer's projections alone; no headline line
        return {"mixer": bench_mixer(efla, lib, dev, stream, pk, flush, iters=max(args.steps, 1))}

    w = wl.LM340M_FWD
    B, H, L, dk, dv, C = w.B, w.H, w.L, w.dk, w.dv, w.chunk
    x = wl.fwd_inputs_device(w, dev, seed=rank_seed(w, rank))
    q, k, v, beta = x["q"], x["k"], x["v"], x["beta"]
    o = torch.empty((B, H, L, dv), dtype=torch.bfloat16, device=dev)
    Sf = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    shape = efla.make_shape(B, H, L, dk, dv, C, torch.bfloat16, torch.bfloat16)
    wsz = efla.efla_fwd_workspace_size(shape)
    wsp = torch.empty(wsz, dtype=torch.uint8, device=dev)

    def step():
        efla.efla_fwd(q, k, v, beta, None, chunk=C, o=o, S_final=Sf, workspace=wsp)

    clocks = ClockSampler(local)
    clocks.start()
    # warm-up, then a short soak so clocks settle before timing
    for _ in range(args.warmup + 20):
        step()
    torch.cuda.synchronize(dev)

    barrier(ws)
    torch.cuda.synchronize(dev)
    step_ms = timed(step, args.steps, stream, flush)
    barrier(ws)
    ms, value = headline_value(ws, B * L, statistics.mean(step_ms), dev)
    split = kernel_split(lib, step, min(args.steps, 20), stream, flush)
    efla.efla_get_status()
    launches = int(round(sum(d["per_call"] for d in split.values()) * args.steps))

    flops = fwd_flops_per_token_head(dk, dv, C) * B * H * L
    tflops = flops / (ms * 1e-3) / 1e12
    alg_bytes = (3 * B * H * L * dk * 2) + (B * H * L * dv * 2) + B * H * L * 4 + B * H * dk * dv * 4
    # (the flag clearing before the fused forward is a few microseconds of the call)
    dom, kern_ms, path_ms = roofline_timing(split)
    hbm = pk["hbm_gbs"]
    achieved = alg_bytes / (kern_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4),
                "traffic": measured_traffic(f"k_fwd_tc@{w.name}") if dom == "efla_tc_fused" else None,
                "kernel": dom if kern_ms < path_ms else "+".join(split),
                "kernel_ms": {n: round(d["ms"], 4) for n, d in split.items()},
                "path_kernel_ms": round(path_ms, 4), "timed_ms": round(kern_ms, 4),
                "dominant": dom,
                "alg_bytes_per_launch": alg_bytes,
                "peak_kind": f"{pk_kind} (copy bandwidth)",
                "tensor_frac": round(flops / (kern_ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                "timing": "kernel time from a separate instrumented pass; ms_per_step from an "
                          "uninstrumented one"}

    e2e = None if args.skip_e2e else bench_e2e(efla, x, o, Sf, wsp, C, stream, dev, ws, B * L, args.steps)

    extras = {}
    if not args.skip_extras:
        extras["euler_fwd"] = bench_exact_vs_euler(efla, lib, x, o, Sf, wsp, C, flush, stream, B * L)
        extras["decode"] = bench_decode(efla, lib, dev, stream, pk, pk_kind)
        extras["bwd"] = bench_bwd(efla, lib, dev, stream, pk, pk_kind, flush)
        extras["stiff_long_fwd"] = bench_stiff_long(efla, lib, dev, stream, pk)
        extras["mixer"] = bench_mixer(efla, lib, dev, stream, pk, flush)
    clk = clocks.stop()

    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded device RNG; 340M-layer shapes and distributions)",
            "config": headline_config(w, ws),
            "tflops": round(tflops, 3), "roofline": roofline, "e2e": e2e,
            "gpu_launches": launches, "clocks": clk}
    line.update(extras)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_fwd()
    return line


def bench_e2e(efla, x, o, Sf, wsp, C, stream, dev, ws, tokens, steps):
    """End to end through host buffers (pinned), copies inside the timed region.  Steps
    are pipelined over two buffer sets: step i's inputs go in (copy stream) while step
    i-1 computes and step i-2's output comes out (a second copy stream); the timed region
    runs from the first input copy to the last output copy."""
    q, k, v, beta = x["q"], x["k"], x["v"], x["beta"]
    hq, hk, hv, hb = (t.cpu().pin_memory() for t in (q, k, v, beta))
    hos = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    din = [tuple(torch.empty_like(t) for t in (q, k, v, beta)) for _ in range(2)]
    dout = [torch.empty_like(o) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()   # noqa: E731
    free = [ev(), ev()]           # buffer set b may be overwritten (its output has left)
    loaded = [ev(), ev()]
    done = [ev(), ev()]
    for b_ in range(2):
        free[b_].record(s_out)

    def e2e_step(i):
        b_ = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(free[b_])
            for dst, src in zip(din[b_], (hq, hk, hv, hb)):
                dst.copy_(src, non_blocking=True)
            loaded[b_].record(s_in)
        stream.wait_event(loaded[b_])
        dq_, dk_, dv_, db_ = din[b_]
        efla.efla_fwd(dq_, dk_, dv_, db_, None, chunk=C, o=dout[b_], S_final=Sf, workspace=wsp)
        done[b_].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b_])
            hos[b_].copy_(dout[b_], non_blocking=True)
            free[b_].record(s_out)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / steps, ws, dev)
    return {"value": round(ws * tokens / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(e2e_ms, 4),
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (hq, hk, hv, hb)),
            "d2h_bytes_per_step": hos[0].numel() * hos[0].element_size(),
            "pipelined": "input copy of step i || compute of step i-1 || output copy of step i-2"}


def bench_decode(efla, lib, dev, stream, pk, pk_kind):
    w = wl.DECODE
    B, H, dk, dv, steps = w.B, w.H, w.dk, w.dv, w.steps
    x = wl.decode_inputs_device(w, steps, dev)
    S = torch.zeros((B, H, dk, dv), dtype=torch.float32, device=dev)
    o = torch.empty((B, H, dv), dtype=torch.bfloat16, device=dev)
    for t in range(3):   # warm-up on the same state
        efla.efla_step(x["q"][t], x["k"][t], x["v"][t], x["beta"][t], S, o=o)
    torch.cuda.synchronize(dev)

    def run_all():
        for t in range(steps):
            efla.efla_step(x["q"][t], x["k"][t], x["v"][t], x["beta"][t], S, o=o)
    S.zero_()
    ms = timed(run_all, 1, stream)[0] / steps
    S.zero_()
    split = kernel_split(lib, run_all, 1, stream)
    efla.efla_get_status()
    kms = split["efla_decode_step"]["ms"]
    sbytes = B * H * dk * dv * 4
    alg = 2 * sbytes + B * H * (2 * dk + dv) * 2 + B * H * 4 + B * H * dv * 2
    gbs = alg / (kms * 1e-3) / 1e9
    return {"workload": w.name, "value": round(alg / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "tokens_per_s": round(B / (ms * 1e-3), 1),
            "steps": steps,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                         "traffic": measured_traffic(f"k_step@{w.name}"),
                         "kernel": "efla_decode_step", "kernel_ms": round(kms, 5),
                         "alg_bytes_per_launch": alg,
                         "peak_kind": f"{pk_kind} (copy bandwidth)"},
            "l2": "state 268 MB > 129 MB L2; no flush"}


def bench_bwd(efla, lib, dev, stream, pk, pk_kind, flush, iters=5):
    w = wl.LM1P3B_FWDBWD
    B, H, L, dk, dv, C = w.B, w.H, w.L, w.dk, w.dv, w.chunk
    x = wl.fwd_inputs_device(w, dev)
    shape = efla.make_shape(B, H, L, dk, dv, C, torch.bfloat16, torch.bfloat16)
    wsp = torch.empty(efla.efla_bwd_workspace_size(shape), dtype=torch.uint8, device=dev)

    def run():
        return efla.efla_bwd(x["q"], x["k"], x["v"], x["beta"], x["dO"], x["S0"], None, chunk=C,
                             workspace=wsp)
    for _ in range(2):
        run()
    torch.cuda.synchronize(dev)
    ms = statistics.mean(timed(run, iters, stream, flush))
    split = kernel_split(lib, run, 2, stream, flush)
    efla.efla_get_status()
    flops = bwd_flops_per_token_head(dk, dv, C) * B * H * L
    alg = (4 * B * H * L * dk * 2) + B * H * L * 4 + 2 * B * H * dk * dv * 4 + \
        (3 * B * H * L * dk * 2) + B * H * L * 4
    res = {"workload": w.name, "ms": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 3),
           "tokens_per_s": round(B * L / (ms * 1e-3), 1),
           "hbm_frac": round(alg / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
           "kernel_ms": {n: round(d["ms"], 4) for n, d in split.items()}}

    # the same training step with a recorded forward: efla_fwd_save keeps every chunk's
    # entering state, efla_bwd_saved skips the state scan (chosen when the record fits)
    o = torch.empty((B, H, L, dv), dtype=torch.bfloat16, device=dev)
    Sf = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    rec = torch.empty(efla.efla_fwd_states_size(shape) // 4, dtype=torch.float32, device=dev)
    fws = torch.empty(efla.efla_fwd_workspace_size(shape), dtype=torch.uint8, device=dev)
    sws = torch.empty(efla.efla_bwd_saved_workspace_size(shape), dtype=torch.uint8, device=dev)

    def fwd_plain():
        efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"], chunk=C, o=o, S_final=Sf, workspace=fws)

    def fwd_save():
        efla.efla_fwd_save(x["q"], x["k"], x["v"], x["beta"], x["S0"], chunk=C, o=o, S_final=Sf, states=rec,
                           workspace=fws)

    def bwd_saved():
        efla.efla_bwd_saved(x["q"], x["k"], x["v"], x["beta"], x["dO"], rec, None, chunk=C, workspace=sws)
    for f in (fwd_plain, fwd_save, bwd_saved):
        f()
    torch.cuda.synchronize(dev)
    t_fp = statistics.mean(timed(fwd_plain, iters, stream, flush))
    t_fs = statistics.mean(timed(fwd_save, iters, stream, flush))
    t_bs = statistics.mean(timed(bwd_saved, iters, stream, flush))
    split_s = kernel_split(lib, bwd_saved, 2, stream, flush)
    efla.efla_get_status()
    res["recorded"] = {
        "record_bytes": rec.numel() * 4,
        "plan_at_record_plus_workspace": efla.efla_bwd_plan(shape, rec.numel() * 4 + sws.numel()),
        "fwd_ms": round(t_fp, 4), "fwd_save_ms": round(t_fs, 4), "bwd_saved_ms": round(t_bs, 4),
        "step_ms_recompute": round(t_fp + ms, 4), "step_ms_recorded": round(t_fs + t_bs, 4),
        "faster_step": "recompute" if t_fp + ms < t_fs + t_bs else "recorded",
        "bwd_saved_kernel_ms": {n: round(d["ms"], 4) for n, d in split_s.items()}}
    return res


def bench_mixer(efla, lib, dev, stream, pk, flush, iters=10):
    """The token mixer's input projections (one tcgen05 GEMM, x [B L, D] -> q, k, v, beta)
    at the 340M and 1.3B layer widths, alone and followed by the EFLA forward."""
    out = {}
    for w in (wl.MIXER_340M, wl.MIXER_1P3B):
        x = wl.mixer_inputs(w, device=dev)
        xd, wd = x["x"], x["w"]
        q = torch.empty((w.B, w.H, w.L, w.dk), dtype=torch.bfloat16, device=dev)
        k, v = torch.empty_like(q), torch.empty_like(q)
        beta = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=dev)
        o = torch.empty_like(q)
        shape = efla.make_shape(w.B, w.H, w.L, w.dk, w.dk, 64, torch.bfloat16, torch.bfloat16)
        fws = torch.empty(efla.efla_fwd_workspace_size(shape), dtype=torch.uint8, device=dev)

        def proj():
            efla.efla_mixer_proj(xd, wd, w.H, q=q, k=k, v=v, beta=beta)

        def layer():
            proj()
            efla.efla_fwd(q, k, v, beta, None, o=o, workspace=fws, want_state=False)
        for f in (proj, layer, proj):
            f()
        torch.cuda.synchronize(dev)
        t_p = statistics.median(timed(proj, iters, stream, flush))
        t_l = statistics.median(timed(layer, iters, stream, flush))
        split = kernel_split(lib, proj, 3, stream, flush)
        efla.efla_get_status()
        N = 3 * w.H * w.dk + w.H
        flops = 2.0 * w.B * w.L * w.D * N
        kms = split["efla_mixer_proj"]["ms"]
        ach = flops / (kms * 1e-3) / 1e12
        out[w.name] = {"proj_ms": round(t_p, 4), "proj_kernel_ms": round(kms, 4),
                       "proj_tflops": round(ach, 1),
                       "roofline": {"bound": "tensor", "achieved": round(ach, 1), "peak": pk["bf16_tflops"],
                                    "unit": "TFLOP/s", "frac": round(ach / pk["bf16_tflops"], 4),
                                    "flops_per_launch": flops},
                       "layer_fwd_ms": round(t_l, 4),
                       "layer_tokens_per_s": round(w.B * w.L / (t_l * 1e-3), 1)}
    return out


# ------------------------------------------------------- CPU oracle legs
def cpu_baseline_fwd(heads=None):
    """The fp64 oracle, as it stands, on the 340M-layer workload (CPU-generated inputs)."""
    import oracle
    w = wl.LM340M_FWD
    x = wl.make_inputs(w)
    q, k, v, beta = x["q"], x["k"], x["v"], x["beta"]
    if heads is not None:
        q, k, v, beta = (t.reshape(w.B * w.H, *t.shape[2:])[:heads].unsqueeze(0)
                         for t in (q, k, v, beta))
    nh = q.shape[0] * q.shape[1]
    q64, k64, v64, b64 = (oracle._f64(t) for t in (q, k, v, beta))
    t0 = time.perf_counter()
    oracle.fwd(q64, k64, v64, b64)
    dt = time.perf_counter() - t0
    tokens = nh * w.L / w.H          # token-heads / heads per token
    return {"value": round(tokens / dt, 1), "unit": "tokens/s", "cores": oracle.max_threads(),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"{nh} of {w.B * w.H} sequences x L={w.L} of {w.name} (fp64, OpenMP over sequences)"}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    w = wl.LM340M_FWD
    heads = 16   # bounded sample per step: 16 of the 64 sequences
    for _ in range(args.warmup):
        cpu_baseline_fwd(heads)
    times = []
    last = None
    for _ in range(args.steps):
        last = cpu_baseline_fwd(heads)
        times.append(last["seconds"])
    ms = 1e3 * statistics.mean(times)
    tokens = heads * w.L / w.H
    value = tokens / (ms * 1e-3)
    cb = dict(last)
    cb["value"] = round(value, 1)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded CPU RNG; 340M-layer shapes and distributions)",
            "config": headline_config(w, ws),
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--skip-extras", action="store_true", help="skip the decode and bwd sections")
    ap.add_argument("--skip-e2e", action="store_true", help="skip the end-to-end (host buffer) leg")
    ap.add_argument("--only-mixer", action="store_true",
                    help="time only the token mixer's projections (340M and 1.3B widths) and print their entry")
    ap.add_argument("--record-traffic", nargs=5, metavar=("CSV", "KEY", "KERNEL_REGEX", "SOURCE", "COMMAND"),
                    help="write the DRAM bytes of an ncu CSV capture into profiles/dram_traffic.json and exit")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-bwd", action="store_true",
                    help="time only the backward leg (1.3B-layer workload) and print its entry")
    ap.add_argument("--only-decode", action="store_true",
                    help="time only the decode leg (B256 H16 d128, 1024 steps) and print its entry")
    ap.add_argument("--only-stiff", action="store_true",
                    help="time only the stiff long-context forward (B1 H16 L65536) and print its entry")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(*args.record_traffic)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
    else:
        line = run_gb300(args, ws, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
