#!/usr/bin/env python
"""Benchmark of the sharded-state step on GB300: params/s and achieved HBM GB/s.

One step = one pass of the whole hot path over one synthetic batch of gradients:
FULL_SHARD = two all-gathers (fsdp_unshard, forward and backward) + the fused
reduce-scatter + AdamW + bf16 recast (fsdp_reduce_scatter_adamw) over all units.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mlp128m]
  python bench.py --impl reference      # the CPU oracle on a bounded sample

Prints ONE JSON line (rank 0).  `value` is whole-job params/s with inputs resident
in HBM; `e2e` is the same metric through the public API with host buffers (the
gradient replicas copied host->device and the updated parameter shards
device->host inside every timed step); `roofline` is the dominant kernel's
algorithmic bytes per launch over its CUDA-event duration against the measured
HBM copy peak; `cpu_baseline` is the oracle timed on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sharded-step params/sec and achieved HBM GB/s (% of GB300 peak) at 1 GPU"
PEAK_FALLBACK_GBS = 6800.0
KERNEL_SRC = {k: [os.path.join(ROOT, "fsdp_sharded_state_gb300", "csrc", f) for f in srcs + ("device_ops.cuh", "common.cuh")]
              for k, srcs in (("k_rs_adamw", ("kernels.cu",)), ("k_rs_adamw_staged", ("staged.cu", "pipeline.cuh")))}


# ---------------------------------------------------------------------------
# helpers that need no GPU (tested on CPU)
# ---------------------------------------------------------------------------
def algorithmic_bytes(N, P, S, F, mode, grad_bytes, param_bytes, grad_out=False):
    """Algorithmic HBM bytes per launch of each kernel, whole layout.
    rs_adamw: N replicas x P logical gradient elements read; fp32 master, exp_avg,
    exp_avg_sq read + written for the N*S shard elements (24 B); the bf16 copy
    written (2 B) when the parameter dtype is bf16; the fp32 reduced gradient
    (4 B) when requested.  Padding is skipped by the kernel, so the shard terms
    count logical elements (N*S - pad = P).
    unshard: the shard elements read and the full-layout elements written
    (FLAT: N*S each -- the padded flat parameter; DIM0: P each)."""
    logical_shard = P
    rs = N * P * grad_bytes + 24 * logical_shard + (2 * logical_shard if param_bytes == 2 else 0)
    if grad_out:
        rs += 4 * N * S
    gathered = N * S if mode == 0 else P
    unshard = 2 * gathered * param_bytes
    return {"rs_adamw": rs, "unshard": unshard}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return PEAK_FALLBACK_GBS, "fallback"


def code_only(src: str) -> str:
    """C/C++/CUDA source without comments and with whitespace collapsed: what the
    compiler sees, so that an edit to a comment does not void a recorded capture."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_src_hash(kernel="k_rs_adamw"):
    """Hash of the code (comments aside) of the sources a core kernel compiles from."""
    h = hashlib.sha256()
    for p in KERNEL_SRC[kernel]:
        with open(p, encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload, with_source=False):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or the kernel source changed since.  A
    summary taken on a smaller case of the same layout class carries `scaled_from`:
    its bytes were scaled to this workload by the ratio of logical parameters.
    with_source=True also returns where the figure comes from."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")
    d = None
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get("kernel_src_sha256_16") != kernel_src_hash(kernel):
            d = None
    v = d.get("dram_bytes_per_launch") if d else None
    if not with_source:
        return v
    src = None
    if d is not None:
        sf = d.get("scaled_from")
        src = (f"ncu on {sf['workload']}, scaled x{d['scale']:.4f} by logical parameters" if sf
               else f"ncu on {workload}")
    return v, src


def launch_stats(ms):
    """Median, 95th percentile and coefficient of variation of per-launch times (ms);
    cv_flag when the spread exceeds 5 %."""
    xs = sorted(ms)
    med = statistics.median(xs)
    p95 = xs[min(len(xs) - 1, int(round(0.95 * (len(xs) - 1))))]
    cv = statistics.pstdev(xs) / statistics.mean(xs) if len(xs) > 1 and statistics.mean(xs) > 0 else 0.0
    return {"median_ms": med, "p95_ms": p95, "cv": cv, "cv_flag": cv > 0.05, "n": len(xs)}


def aggregate_max(value, world, dist=None):
    """Max of a float over ranks (a no-op for one rank)."""
    if world <= 1 or dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def parse_clocks(csv_text):
    """Median SM MHz under load, max SM MHz and the throttle reasons seen."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in csv_text.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9 or not parts[1].split()[0].isdigit():
            continue
        sm.append(float(parts[1].split()[0]))
        smax.append(float(parts[2].split()[0]))
        for nm, flag in zip(names, parts[5:9]):
            if flag.lower().startswith("active"):
                reasons.add(nm)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    load = [x for x in sm if x > 0.5 * max(sm)] or sm
    return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm)}


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.out = ""
        self.dev = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def _normal_block(rng, n, std, block=1 << 22):
    """n fp32 values N(0, std): one seeded block of up to 4M draws, repeated (the oracle's
    speed does not depend on the values, and drawing hundreds of millions of normals
    would take the host longer than the steps it times)."""
    import numpy as np
    x = rng.standard_normal(min(n, block), dtype=np.float32) * np.float32(std)
    return np.resize(x, n)


def oracle_sample_setup(w, target_s=1.0, unit=0):
    """Host inputs for a bounded sample of workload w: the units [unit, u_end) whose
    oracle step takes about target_s seconds (at least one unit)."""
    import numpy as np

    import oracle
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    O = oracle.layout(sh, w.N, w.mode)
    stride = O["S"]
    rng = np.random.default_rng(unit)
    u_end = unit + 1
    numel = int(O["u_numel"][unit])
    # about 2.5e7 elements per second of single-core oracle work at N=4 (measured order)
    budget = int(2.5e7 * target_s * 4 / max(w.N, 1))
    while u_end < O["U"] and numel + int(O["u_numel"][u_end]) <= budget:
        numel += int(O["u_numel"][u_end])
        u_end += 1
    lo = int(O["u_full_off"][unit])
    hi = int(O["u_full_off"][u_end - 1] + (w.N * O["u_S"][u_end - 1] if w.mode == 0 else O["u_numel"][u_end - 1]))
    full = np.zeros(O["F"], np.float32)
    full[lo:hi] = _normal_block(rng, hi - lo, 0.02)
    gdt = np.uint16 if str(w.grad_dtype).endswith("bfloat16") else np.float32
    grads = []
    for _ in range(w.N):
        g = np.zeros(O["F"], gdt)
        x = _normal_block(rng, hi - lo, w.grad_std)
        g[lo:hi] = oracle.bf16_rne(x) if gdt == np.uint16 else x
        grads.append(g)
    bf16 = gdt == np.uint16 or str(w.param_dtype).endswith("bfloat16")
    master, param = oracle.reshard(sh, w.N, w.mode, full, stride, True, bf16)
    st = {"sh": sh, "O": O, "stride": stride, "grads": grads, "master": master, "param": param,
          "m": np.full_like(master, 0.0), "v": np.full_like(master, 0.0), "u_end": u_end, "numel": numel,
          "out": np.zeros(O["F"], np.uint16 if bf16 else np.float32)}
    return st


def oracle_step(w, st, t, strategy, ub=0):
    import oracle
    src = st["param"] if st["param"] is not None else st["master"]
    for _ in range(2 if strategy == "full_shard" else 1):
        oracle.unshard(st["sh"], w.N, w.mode, src, st["stride"], st["O"]["F"], ub, st["u_end"], out=st["out"])
    oracle.rs_adamw(st["sh"], w.N, w.mode, st["grads"], st["stride"], st["master"], st["m"], st["v"],
                    param=st["param"], hp=w.hp, step=t, ub=ub, ue=st["u_end"])


def host_cpu():
    """The host's CPU model (lscpu) and logical core count, recorded beside the oracle's timing."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"model": model, "nproc": os.cpu_count()}


def cpu_baseline(w, strategy, min_seconds=10.0):
    """The oracle on one host core: the step on a prefix of the workload's units."""
    st = oracle_sample_setup(w, target_s=1.0)
    t0 = time.perf_counter()
    steps = 0
    while True:
        steps += 1
        oracle_step(w, st, steps, strategy)
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    return {"value": st["numel"] * steps / el, "unit": "params/s", "cores": 1, "kind": "oracle",
            "sample": f"units [0,{st['u_end']}) of {w.name} ({st['numel']} params), {steps} oracle steps "
                      f"({strategy}), single thread, {el:.1f} s", "host": host_cpu()}


def unit_workload(w, unit):
    """The tensors of one unit of w as a workload of its own (one unit, the same N, mode,
    dtypes and hyper-parameters): a FLAT unit's layout, and so the oracle's arithmetic on
    it, does not depend on the other units, and its buffers are the unit's size."""
    import copy
    idx = [t for t, u in enumerate(w.unit_ids) if u == unit]
    ws = copy.copy(w)
    ws.shapes = [w.shapes[t] for t in idx]
    ws.unit_ids = [0] * len(idx)
    ws.ones = [k for k, t in enumerate(idx) if t in set(w.ones)]
    return ws


def _oracle_proc(name, strategy, unit, warmup, steps, min_seconds, barrier, out):
    """One process of the host-wide oracle run: the unmodified single-threaded oracle
    step on one unit of its own copy of the workload.  After set-up and `warmup` steps
    every process waits at the barrier, so the timed steps of all processes overlap;
    then `steps` steps (or, with steps = 0, as many as fill min_seconds)."""
    try:
        import oracle
        from fsdp_sharded_state_gb300 import synth
        w = unit_workload(synth.workload(name), unit)
        st = oracle_sample_setup(w, target_s=0.0)
        for k in range(warmup):
            oracle_step(w, st, k + 1, strategy)
        barrier.wait(timeout=1800)
        t0 = time.perf_counter()
        k = 0
        while True:
            k += 1
            oracle_step(w, st, warmup + k, strategy)
            el = time.perf_counter() - t0
            if (steps and k >= steps) or (not steps and el >= min_seconds):
                break
        out.put((unit, st["numel"], k, el, None))
    except Exception as e:          # reported by the parent
        try:
            barrier.abort()
        except Exception:
            pass
        out.put((unit, 0, 0, 0.0, repr(e)))


def oracle_host_run(w, strategy, procs=None, warmup=1, steps=0, min_seconds=10.0):
    """The oracle on every host core: `procs` processes (default: the core count,
    capped by host memory), each running the unmodified single-threaded oracle step
    on one unit of its own copy of the workload (process i takes unit i mod U, so
    the processes cover the units in turn; each builds only that unit's tensors).  The
    processes start with `spawn` (a fresh interpreter: nothing of this process's CUDA
    state is inherited) and time their steps together; the aggregate is the parameters
    all processes stepped over the slowest process's time."""
    import multiprocessing as mpr

    import oracle
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    O = oracle.layout(sh, w.N, w.mode)
    U = O["U"]
    n = int(O["u_numel"].max())
    gb = 2 if str(w.grad_dtype).endswith("bfloat16") else 4
    # host bytes of one process (its unit's full-layout buffers): the fp32 full parameters,
    # N gradient replicas, master/m/v and the bf16 copy, the gathered output
    per_proc = 0
    for u in range(U):
        ws = unit_workload(w, u)
        Ou = oracle.layout(oracle.Shapes(ws.shapes, ws.unit_ids), ws.N, ws.mode)
        F, NS = int(Ou["F"]), w.N * int(Ou["S"])
        per_proc = max(per_proc, 4 * F + w.N * gb * F + 14 * NS + 4 * F)
    try:
        host_mem = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    except (ValueError, OSError, AttributeError):
        host_mem = 16 << 30
    ncpu = os.cpu_count() or 1
    if procs is None:
        procs = max(1, min(ncpu, int(0.55 * host_mem // max(per_proc, 1))))
    ctx = mpr.get_context("spawn")
    barrier = ctx.Barrier(procs)
    out = ctx.Queue()
    ps = [ctx.Process(target=_oracle_proc, args=(w.name, strategy, i % U, warmup, steps, min_seconds, barrier, out))
          for i in range(procs)]
    for p in ps:
        p.start()
    import queue
    res, t_give_up = [], time.time() + 3600
    while len(res) < len(ps):
        try:
            res.append(out.get(timeout=1.0))
        except queue.Empty:
            dead = [p.exitcode for p in ps if p.exitcode not in (None, 0)]
            if dead or time.time() > t_give_up:      # a process died before reporting
                for p in ps:
                    if p.is_alive():
                        p.terminate()
                raise RuntimeError(f"oracle processes failed (exit codes {dead})")
    for p in ps:
        p.join(timeout=60)
    errs = [r[4] for r in res if r[4]]
    if errs:
        raise RuntimeError(f"oracle process failed: {errs[0]}")
    params = sum(r[1] * r[2] for r in res)
    el = max(r[3] for r in res)
    return {"value": params / el, "unit": "params/s", "cores": procs, "kind": "oracle",
            "sample": f"{procs} processes, process i one unit (i mod {U}) of its own copy of {w.name} "
                      f"({n} params per unit; inputs N(0, sigma) from a repeated block of 4M seeded draws), "
                      f"{min(r[2] for r in res)}-{max(r[2] for r in res)} oracle steps "
                      f"({strategy}) each, single-threaded oracle in every process, {el:.1f} s",
            "host": host_cpu(), "elapsed_s": el}


def oracle_one_run(w, strategy, warmup=1, steps=0, min_seconds=10.0):
    """The single-process form of oracle_host_run: this process, one core, one unit."""
    ws = unit_workload(w, 0)
    st = oracle_sample_setup(ws, target_s=0.0)
    for k in range(warmup):
        oracle_step(ws, st, k + 1, strategy)
    t0 = time.perf_counter()
    k = 0
    while True:
        k += 1
        oracle_step(ws, st, warmup + k, strategy)
        el = time.perf_counter() - t0
        if (steps and k >= steps) or (not steps and el >= min_seconds):
            break
    return {"value": st["numel"] * k / el, "unit": "params/s", "cores": 1, "kind": "oracle",
            "sample": f"1 process, unit 0 of {w.name} ({st['numel']} params), {k} oracle steps ({strategy}), "
                      f"single thread, {el:.1f} s", "host": host_cpu(), "elapsed_s": el}


def oracle_host_or_one(w, strategy, procs=None, warmup=1, steps=0, min_seconds=10.0):
    """oracle_host_run; if that fails (a process died, the host ran short of memory),
    the same run in this process on one core, with the failure recorded beside it."""
    try:
        return oracle_host_run(w, strategy, procs=procs, warmup=warmup, steps=steps, min_seconds=min_seconds)
    except Exception as e:
        r = oracle_one_run(w, strategy, warmup=warmup, steps=steps, min_seconds=min_seconds)
        r["host_run_failed"] = repr(e)[:300]
        return r


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------
def setup_state(w, dev, rs_kernel="auto"):
    """The workload's sharded state on the device, resharded from its seeded full
    parameters, and its N seeded gradient replicas."""
    import torch

    import fsdp_sharded_state_gb300 as fs
    from fsdp_sharded_state_gb300 import synth
    fs.fsdp_set_rs_kernel(rs_kernel)
    st = fs.ShardedState(w.shapes, w.unit_ids, w.N, w.mode, param_dtype=w.param_dtype, device=dev)
    st.layout.prepare()
    L = st.layout
    offs = [L.tensor(t)["full_off"] for t in range(len(w.shapes))]
    full = synth.full_params(w, st.F, offs, device=dev)
    st.init_from_full(full)
    del full
    grads = synth.grad_replicas(w, st.F, 1, device=dev)
    torch.cuda.synchronize(dev)
    return st, grads


def time_steps(w, st, grads, dev, stream, strategy, steps, warmup, soak, dist=None):
    """Times `steps` sharded steps after an untimed clock soak and `warmup` steps, then
    the same number again with events around each fused launch.  Returns the timed
    region's ms, the per-launch ms of the fused kernel, the algorithmic bytes, whether
    L2 was flushed between steps, and the clock samples of the whole run."""
    import torch

    info = st.layout.info
    gb = 2 if w.grad_dtype == torch.bfloat16 else 4
    pb = 2 if w.param_dtype == torch.bfloat16 else 4
    ab = algorithmic_bytes(w.N, info["numel"], info["shard_numel"], info["full_numel"], w.mode, gb, pb)
    n_unshard = 2 if strategy == "full_shard" else 1

    def step(ev=None):
        for _ in range(n_unshard):
            st.unshard()
        if ev is not None:
            ev[0].record(stream)
        st.reduce_scatter_adamw(grads, w.hp)
        if ev is not None:
            ev[1].record(stream)

    # A step that touches less than 4x L2 would partly run from L2 if steps ran back to
    # back: then every timed step is bracketed by its own events and preceded by a write
    # of a scratch buffer four times the L2 (outside the step's events).
    step_bytes = ab["rs_adamw"] + n_unshard * ab["unshard"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = step_bytes < 4 * l2
    scratch = torch.empty(4 * l2 // 4 + 1, dtype=torch.float32, device=dev) if flush else None

    with ClockSampler(dev.index) as clk:
        t_end = time.time() + soak             # clock soak (untimed): clocks to their working point
        while time.time() < t_end:
            step()
            torch.cuda.synchronize(dev)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        sevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        # the timed steps: no event between the kernels of a step (an event recorded
        # between two kernels ends the programmatic overlap of the second's launch)
        t0.record(stream)
        for k in range(steps):
            if flush:
                scratch.fill_(float(k))
                sevs[k][0].record(stream)
            step()
            if flush:
                sevs[k][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        # the same steps again with events around the fused kernel: its launch times
        for k in range(steps):
            if flush:
                scratch.fill_(float(k))
            step(evs[k])
        torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in sevs) if flush else t0.elapsed_time(t1)
    rs_ms = [a.elapsed_time(b) for a, b in evs]
    l2_note = ("L2 flushed before every step (a %.0f MB write; the step touches %.3f GB)" % (4 * l2 / 1e6, step_bytes / 1e9)
               if flush else "inputs larger than L2 (step touches %.2f GB)" % (step_bytes / 1e9))
    return {"ms": ms, "rs_ms": rs_ms, "ab": ab, "step_bytes": step_bytes, "flush": flush, "l2": l2_note,
            "n_unshard": n_unshard, "clocks": parse_clocks(clk.out)}


def fused_roofline(fs, st, w, meas, workload_name):
    """The roofline object of the fused kernel from a time_steps() measurement."""
    peak, peak_kind = load_peaks()
    rs_avg = statistics.mean(meas["rs_ms"])
    rs_bytes = meas["ab"]["rs_adamw"]
    achieved = rs_bytes / (rs_avg * 1e-3) / 1e9
    kname = "k_rs_adamw_staged" if fs.fsdp_rs_kernel_for(st.layout, w.grad_dtype) == "staged" else "k_rs_adamw"
    traffic, traffic_src = profiled_traffic(kname, workload_name, with_source=True)
    return {"kernel": kname, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_kind": peak_kind, "bytes_per_launch": rs_bytes, "launch_ms": rs_avg,
            "traffic": traffic, "traffic_source": traffic_src, "launch_stats": launch_stats(meas["rs_ms"])}


# The configurations timed beside the headline one (the pages' other workloads), one
# after the other, each freed before the next: the 4-block Llama, the FSDP2 dim-0 group
# and the largest points of the one-unit sweep (2^29+1 parameters at N = 32 and N = 2) as
# the fused kernel's HBM rate, the tiny MLP as the latency of a step.
SIDE_CONFIGS = ("llama4", "dim0_n6", "tiny_mlp", "sweep_P536870913_N32", "sweep_P536870913_N2")
# Side configurations whose oracle step is not timed in the bench: one unit of 537M
# parameters per oracle process would take the host minutes to set up and step.
NO_CPU_SIDE = {"sweep_P536870913_N32": "not timed: one 537M-parameter unit per oracle process exceeds the bench's "
                                       "CPU time (about 20 GB of host buffers and minutes per step)",
               "sweep_P536870913_N2": "not timed: one 537M-parameter unit per oracle process exceeds the bench's "
                                      "CPU time (about 20 GB of host buffers and minutes per step)"}
GATE_GBS = 8000.0 * 0.75          # the pages' target: 75 % of ~8 TB/s


def side_config(args, name, dev, stream):
    import torch

    import fsdp_sharded_state_gb300 as fs
    from fsdp_sharded_state_gb300 import synth
    w = synth.workload(name)
    st, grads = setup_state(w, dev, args.rs_kernel)
    steps = max(args.steps, 20)
    meas = time_steps(w, st, grads, dev, stream, args.strategy, steps, max(args.warmup, 3), args.soak)
    fs.fsdp_check_status(stream)
    roof = fused_roofline(fs, st, w, meas, name)
    P = st.P
    out = {"workload": name, "params": P, "n_ranks_simulated": w.N,
           "layout": "flat" if w.mode == 0 else "dim0", "strategy": args.strategy,
           "param_dtype": str(w.param_dtype).replace("torch.", ""),
           "grad_dtype": str(w.grad_dtype).replace("torch.", ""), "steps": steps,
           "ms_per_step": meas["ms"] / steps, "params_per_s": P * steps / (meas["ms"] * 1e-3),
           "step_bytes": meas["step_bytes"], "step_hbm_gbs": meas["step_bytes"] / (meas["ms"] / steps * 1e-3) / 1e9,
           "l2": meas["l2"], "kernel": roof["kernel"], "launch_ms": roof["launch_ms"],
           "bytes_per_launch": roof["bytes_per_launch"], "achieved_gbs": roof["achieved"], "frac": roof["frac"],
           "traffic": roof["traffic"], "traffic_source": roof["traffic_source"],
           "peak_kind": roof["peak_kind"], "frac_of_8tbs": roof["achieved"] / 8000.0,
           "gate_75pct_of_8tbs": roof["achieved"] >= GATE_GBS, "launch_stats": roof["launch_stats"],
           "clocks": meas["clocks"]}
    if meas["flush"]:
        out["us_per_step"] = meas["ms"] / steps * 1e3        # latency-bound: the step's time is the figure
    del st, grads
    torch.cuda.empty_cache()
    if not args.no_cpu_baseline and name in NO_CPU_SIDE:
        out["cpu_baseline"] = {"kind": "oracle", "value": None, "note": NO_CPU_SIDE[name]}
    elif not args.no_cpu_baseline:
        # the oracle on this workload, on every host core (one oracle process per core)
        import oracle
        oracle.build()
        cb = oracle_host_or_one(w, args.strategy, procs=args.cpu_procs, warmup=0, min_seconds=args.cpu_seconds_side)
        out["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "host_run_failed")
                               if k in cb}
        out["cpu_baseline"]["per_process"] = cb["value"] / cb["cores"]
    return out


def run_ours(args, w, rank, world, dist):
    import torch

    import fsdp_sharded_state_gb300 as fs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    st, grads = setup_state(w, dev, args.rs_kernel)
    meas = time_steps(w, st, grads, dev, stream, args.strategy, args.steps, args.warmup, args.soak, dist)
    fs.fsdp_check_status(stream)
    ms_max = aggregate_max(meas["ms"], world, dist)

    # e2e through the public API with host buffers (pinned): every step copies its N
    # gradient replicas host -> device and its updated parameter shards back
    # (HostFeed overlaps those copies with the neighbouring steps' compute)
    host_grads = [g.cpu().pin_memory() for g in grads]
    out_host = torch.empty(st.param_shards.shape, dtype=st.param_shards.dtype).pin_memory()
    h2d = sum(g.numel() * g.element_size() for g in host_grads)
    d2h = out_host.numel() * out_host.element_size()
    feed = fs.HostFeed(st, w.grad_dtype, stream=stream)
    for _ in range(max(args.warmup, 1)):
        feed.step(host_grads, out_host, w.hp, args.strategy)
    feed.finish()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    feed.begin()
    for _ in range(args.steps):
        feed.step(host_grads, out_host, w.hp, args.strategy)
    feed.finish()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = aggregate_max(e0.elapsed_time(e1), world, dist)
    del feed
    roof = fused_roofline(fs, st, w, meas, w.name)
    info = st.layout.info
    P = info["numel"]
    launches_per_step = st.launches_per_step(args.strategy, w.grad_dtype)
    res = {
        "metric": METRIC,
        "value": world * P * args.steps / (ms_max * 1e-3),
        "unit": "params/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if w.param_dtype == torch.float32 else "bf16+f32",
        "data": "synthetic",
        "config": {"workload": w.name, "shapes": f"{len(w.shapes)} tensors, {P} params", "n_ranks_simulated": w.N,
                   "layout": "flat" if w.mode == 0 else "dim0", "strategy": args.strategy,
                   "param_dtype": str(w.param_dtype).replace("torch.", ""),
                   "grad_dtype": str(w.grad_dtype).replace("torch.", ""),
                   "master_moments": "float32", "step_bytes": meas["step_bytes"], "l2": meas["l2"],
                   "clock_soak_s": args.soak, "parallelism": f"replicas x{world}",
                   "collectives_per_rank": st.layout.collective_payload(args.strategy)},
        "step_hbm_gbs": meas["step_bytes"] / (ms_max / args.steps * 1e-3) / 1e9,
        "roofline": roof,
        "e2e": {"value": world * P * args.steps / (e2e_ms * 1e-3), "unit": "params/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": meas["clocks"],
    }
    del st, grads, host_grads, out_host
    torch.cuda.empty_cache()
    if world == 1 and args.side_configs:
        res["configs"] = {}
        for name in SIDE_CONFIGS:
            if name != w.name:
                res["configs"][name] = side_config(args, name, dev, stream)
    return res


def row_bytes(row, w, P, N, R=2):
    """Algorithmic HBM bytes of one call of a row (whole layout, logical elements).
    clip:  N replicas read; fp32 gradient shard written, re-read and rewritten
           (clipped); master/m/v read + written; bf16 params written.
    accum: per replica the micro-gradient read and the fp32 accumulator read + written.
    accum_step: the last micro-batch fused with the step: per replica the fp32
           accumulator and the micro-gradient read; master/m/v read + written; bf16 params.
    hsdp:  R*N replicas read; R copies of master/m/v read + written (+ bf16 params).
    zero1: N replicas read; the owner's m/v (and master, or its own fp32 replica)
           read + written; the updated parameter written into all N replicas."""
    import torch
    gb = 2 if w.grad_dtype == torch.bfloat16 else 4
    bf = w.param_dtype == torch.bfloat16
    if row == "clip":
        return N * P * gb + 4 * P + 8 * P + 24 * P + (2 * P if bf else 0)
    if row == "accum":
        return N * P * (gb + 8)
    if row == "accum_step":
        # the last micro-batch fused with the step: per replica the fp32 accumulator and
        # the micro-batch gradient read (nothing written back to them); the state as in the step
        return N * P * (4 + gb) + 24 * P + (2 * P if bf else 0)
    if row == "hsdp":
        return R * N * P * gb + R * P * (24 + (2 if bf else 0))
    if row == "zero1":
        return N * P * gb + P * (16 + (8 if bf else 4)) + N * P * (2 if bf else 4)
    raise KeyError(row)


def run_row(args, w):
    """Times one call of a row beyond the core step (clip / accum / hsdp / zero1)."""
    import torch

    import fsdp_sharded_state_gb300 as fs
    from fsdp_sharded_state_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fs.fsdp_set_rs_kernel(args.rs_kernel)
    N, R = w.N, args.groups
    mode = fs.FSDP_ZERO1 if args.row == "zero1" else w.mode
    L = fs.Layout(w.shapes, w.unit_ids, N, mode)
    L.prepare()
    P, F, stride = L.info["numel"], L.info["full_numel"], L.stride
    offs = [L.tensor(t)["full_off"] for t in range(len(w.shapes))]
    full = synth.full_params(w, F, offs, device=dev)
    bf = w.param_dtype == torch.bfloat16
    z = lambda *shape, dt=torch.float32: torch.zeros(*shape, dtype=dt, device=dev)
    if args.row in ("clip", "accum", "accum_step"):
        st = fs.ShardedState(w.shapes, w.unit_ids, N, w.mode, param_dtype=w.param_dtype, device=dev,
                             with_grad_out=True)
        st.init_from_full(full)
        grads = synth.grad_replicas(w, F, 1, device=dev)
        if args.row == "clip":
            ws = z(fs.fsdp_clip_workspace_bytes(), dt=torch.uint8)
            call = lambda t: fs.fsdp_reduce_scatter_clip_adamw(st.layout, 0, st.layout.n_units, grads,
                                                               st.master, st.exp_avg, st.exp_avg_sq, st.param,
                                                               st.grad_out, 1e-2, ws, None, w.hp, t)
        elif args.row == "accum":
            acc = [z(F) for _ in range(N)]
            call = lambda t: fs.fsdp_accumulate_grads(st.layout, 0, st.layout.n_units, acc, grads, first=False)
        else:
            acc = [z(F) for _ in range(N)]
            fs.fsdp_accumulate_grads(st.layout, 0, st.layout.n_units, acc, grads, first=True)
            call = lambda t: fs.fsdp_accumulate_reduce_scatter_adamw(st.layout, 0, st.layout.n_units, acc, grads,
                                                                    st.master, st.exp_avg, st.exp_avg_sq, st.param,
                                                                    None, w.hp, t)
    elif args.row == "hsdp":
        master = z(R, N, stride)
        param = z(R, N, stride, dt=torch.bfloat16) if bf else None
        fs.fsdp_reshard(L, 0, L.n_units, full, master[0], param[0] if bf else None)
        for rho in range(1, R):
            master[rho].copy_(master[0])
            if bf:
                param[rho].copy_(param[0])
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        grads = [synth.grad_replica(w, F, 1, k, device=dev) for k in range(R * N)]
        call = lambda t: fs.fsdp_hsdp_reduce_scatter_adamw(L, 0, L.n_units, R, grads, master, m, v, param, w.hp, t)
    else:   # zero1
        master = z(N, stride) if bf else None
        if bf:
            fs.fsdp_reshard(L, 0, L.n_units, full, master, None)
        m, v = z(N, stride), z(N, stride)
        params = [full.to(w.param_dtype).clone() for _ in range(N)]
        grads = synth.grad_replicas(w, F, 1, device=dev)
        call = lambda t: fs.fsdp_zero1_adamw_broadcast(L, 0, L.n_units, grads, master, m, v, params, w.hp, t)
    del full
    with ClockSampler(dev.index) as clk:
        t = 0
        t_end = time.time() + args.soak          # untimed: clocks to their working point, samples taken
        while time.time() < t_end:
            t += 1
            call(t)
            torch.cuda.synchronize()
        for k in range(args.warmup):
            t += 1
            call(t)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in evs:
            t += 1
            a.record()
            call(t)
            b.record()
        torch.cuda.synchronize()
    fs.fsdp_check_status()
    ms = [a.elapsed_time(b) for a, b in evs]
    med = statistics.median(ms)
    nbytes = row_bytes(args.row, w, P, N, R)
    peak, peak_kind = load_peaks()
    achieved = nbytes / (med * 1e-3) / 1e9
    return {"row": args.row, "metric": METRIC, "value": P / (med * 1e-3), "unit": "params/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_call": med, "higher_is_better": True,
            "data": "synthetic", "config": {"workload": w.name, "n_ranks_simulated": N,
                                            "groups": R if args.row == "hsdp" else None},
            "roofline": {"call": args.row, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind, "bytes_per_call": nbytes},
            "clocks": parse_clocks(clk.out)}


def torch_dtype_f32():
    import torch
    return torch.float32


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mlp128m")
    ap.add_argument("--strategy", choices=["full_shard", "shard_grad_op"], default="full_shard")
    ap.add_argument("--soak", type=float, default=1.0, help="untimed seconds of steps before warm-up")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-side-configs", dest="side_configs", action="store_false",
                    help="time the headline workload only (no 'configs' object)")
    ap.add_argument("--cpu-seconds-side", type=float, default=8.0,
                    help="seconds of host-wide oracle steps for each side configuration")
    ap.add_argument("--cpu-procs", type=int, default=None,
                    help="oracle processes of the host-wide CPU baseline (default: the core count)")
    ap.add_argument("--row", choices=["step", "clip", "accum", "accum_step", "hsdp", "zero1"], default="step",
                    help="time a row beyond the core step instead (one JSON line, no cpu baseline)")
    ap.add_argument("--groups", type=int, default=2, help="HSDP replica groups for --row hsdp")
    ap.add_argument("--rs-kernel", choices=["auto", "direct", "staged"], default="auto",
                    help="kernel of the fused reduce-scatter + AdamW step")
    args = ap.parse_args()

    from fsdp_sharded_state_gb300 import synth
    w = synth.workload(args.workload)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None

    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        # the oracle on every host core: one process per core, each stepping one unit
        # of its own copy of the workload; a step = one oracle step in every process
        cb = oracle_host_or_one(w, args.strategy, procs=args.cpu_procs, warmup=args.warmup, steps=args.steps)
        v = cb["value"]
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": "params/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["elapsed_s"] * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if w.param_dtype == torch_dtype_f32() else "bf16+f32", "data": "synthetic",
            "config": {"workload": w.name, "strategy": args.strategy},
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "host", "host_run_failed")
                             if k in cb},
            "e2e": {"value": v, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return

    if args.row != "step":
        print(json.dumps(run_row(args, w)))
        return

    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    res = run_ours(args, w, rank, world, dist)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        # the host's figure (every core, one oracle process each), with one core's beside it
        host = oracle_host_or_one(w, args.strategy, procs=args.cpu_procs, min_seconds=args.cpu_seconds)
        one = cpu_baseline(w, args.strategy, args.cpu_seconds)
        res["cpu_baseline"] = {k: host[k] for k in ("value", "unit", "cores", "kind", "sample", "host", "host_run_failed")
                               if k in host}
        res["cpu_baseline"]["single_core"] = {k: one[k] for k in ("value", "cores", "sample")}
    if rank == 0:
        print(json.dumps(res))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
