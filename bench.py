"""Benchmark of exact shared-prompt tree attention, forward + backward, on GB300.

One step = the whole hot path over one batch of seeded synthetic replay trees: prompt
prefill forward, response replay forward, replay backward (prompt K/V gradient summed
over all branches, split-K reduced without atomics) and prefill backward.  The
schedule (work queues) of a batch is built once, on the host, ahead of the step, the
way a planner prepares a batch while the GPU runs the previous one.

Metric: useful TFLOP/s of fwd+bwd, counting only non-redundant tree FLOPs:
4*D*Hq*N forward + 10*D*Hq*N backward, N = exact count of valid (query, key) pairs
with the prompt counted once.  Also tokens/s (unique tree tokens) and the fraction of
the measured dense-BF16 tensor peak.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica (the path has no
exchange step on one batch); value = all ranks' work / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

DEFAULT_WORKLOAD = "prompt_heavy"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


# DRAM bytes (read + write) per launch of a kernel on a full-size workload, from an ncu
# capture of dram__bytes_read.sum + dram__bytes_write.sum (the summary named in
# "profile" gives the command).  Each entry records a digest of the kernel's sources
# at capture time; once they change, the figure is reported as null.
TRAFFIC = {
    ("prompt_heavy", "bwd_key_side"): {
        "bytes_per_launch": 5.990e9,
        "sources": ["tc_bwd_kv.cu", "tc_common.cuh", "common.cuh", "internal.h", "host.cpp"],
        "digest": "5eb15c90ae7cca51",
        "profile": "profiles/dram_traffic_prompt_heavy.md (mean of 3 launches, ncu one pass)"},
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons in the background."""
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
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    self.rows.append(parts)

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def useful_flops(w):
    return w.useful_flops(True, True)


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (the identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, ms_local: float, world: int, device=None):
    """Whole-job rate of N independent replicas: every rank's units over the slowest
    rank's time.  Returns (rate in units/s, max-over-ranks ms)."""
    ms = max_over_ranks(ms_local, device)
    return units_per_rank * world / (ms * 1e-3), ms


# ---------------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on a bounded sample of the workload's structure.
# ---------------------------------------------------------------------------------
def oracle_sample(w):
    """A down-scaled sample with the same structure: the first group, prompt and
    branch lengths scaled by 1/16, one KV head and its query heads, bounded to a few
    seconds of fp64 work.  Returns (workload, description)."""
    import workloads as W
    lp = max(1, w.tree.prompt_lens[0] // 16)
    bl = [max(1, x // 16) for x in w.tree.branch_lens[0]]
    tree = W.Tree([lp], [bl])
    r = w.hq // w.hkv
    sample = W.custom(tree, hq=r, hkv=1, d=w.d, dtype=w.dtype, seed=w.seed, scale=w.scale, name=w.name + "_sample")
    desc = (f"group 0 of {w.name} with prompt and branch lengths /16 (L_P={lp}, G={len(bl)}, "
            f"sum L_i={sum(bl)}), one KV head with its {r} query heads, D={w.d}; fp64 numpy oracle "
            f"(tree-direct form), fwd+bwd; rate = useful FLOPs of the sample / time")
    return sample, desc


def time_oracle(w, min_seconds=10.0, max_reps=50):
    from oracle import attention as A
    import workloads as W
    sample, desc = oracle_sample(w)
    t = {n: W.tensor_rows_np(sample, n) for n in W.TENSORS}
    flops = useful_flops(sample)
    reps, t0 = 0, time.perf_counter()
    while True:
        A.tree_attention_direct(t, sample.tree.offsets(), A.default_scale(sample.d))
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    rate = flops * reps / el / 1e12
    return rate, desc, el / reps


def cpu_model():
    """The host CPU's model string (x86 'model name', else the Arm implementer/part)."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
        for key in ("model name", "Model"):
            for line in info:
                if line.startswith(key) and ":" in line:
                    return line.split(":", 1)[1].strip()
        impl = next((l.split(":", 1)[1].strip() for l in info if l.startswith("CPU implementer")), None)
        part = next((l.split(":", 1)[1].strip() for l in info if l.startswith("CPU part")), None)
        if impl or part:
            return f"{platform.machine()} implementer {impl} part {part}"
    except OSError:
        pass
    return platform.machine()


def oracle_fields(rate, desc, w):
    """cpu_baseline object: the oracle's rate on its sample, the host, and the full
    workload's step time at that rate (an extrapolation, labelled so)."""
    return {"value": round(rate, 6), "unit": "TFLOP/s", "cores": threads_used(), "kind": "oracle",
            "sample": desc, "cpu_model": cpu_model(),
            "full_step_s_extrapolated": round(useful_flops(w) / (rate * 1e12), 1) if rate > 0 else None,
            "extrapolation": ("rate-scaled estimate: the sample's rate applied to the full step's useful FLOPs; "
                              "the /16 sample's prompt/response mix differs from the full step's")}


def threads_used():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return int(max(x.get("num_threads", 1) for x in info))
    except Exception:
        pass
    return os.cpu_count()


# ---------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------
def kernel_source_digest(files):
    """First 16 hex digits of the SHA-256 of a kernel's source files (identifies the
    kernel version a DRAM-traffic capture was taken on)."""
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "shared_prompt_tree_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_entry(workload: str, kind: str):
    """(bytes per launch, note) of TRAFFIC for a kernel, or (None, why not)."""
    e = TRAFFIC.get((workload, kind))
    if e is None:
        return None, "no capture for this kernel and workload"
    if kernel_source_digest(e["sources"]) != e["digest"]:
        return None, "stale: the kernel's source changed since the capture"
    return e["bytes_per_launch"], e["profile"]


class Run:
    """Device buffers and plan of one workload, and its fwd+bwd step through the C ABI
    (prefill fwd, replay fwd, then one augtree_tree_bwd call, or replay_bwd +
    prefill_bwd)."""

    def __init__(self, w, at, dev, kernel, fused=True, schedule=0):
        import torch
        import workloads as W
        self.w, self.at, self.dev, self.fused = w, at, dev, fused
        dt = at.BF16 if w.dtype == "bf16" else at.FP32
        self.plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=dt, kernel=kernel, schedule=schedule)
        self.t = {n: W.tensor_torch(w, n, dev) for n in W.TENSORS}
        t = self.t
        f32 = torch.float32
        self.o_p, self.o_r = torch.empty_like(t["q_p"]), torch.empty_like(t["q_r"])
        self.lse_p = torch.empty(w.hq, w.tree.total_prompt, dtype=f32, device=dev)
        self.lse_r = torch.empty(w.hq, w.tree.total_resp, dtype=f32, device=dev)
        self.dq_p, self.dk_p, self.dv_p = (torch.empty_like(t[n]) for n in ("q_p", "k_p", "v_p"))
        self.dq_r, self.dk_r, self.dv_r = (torch.empty_like(t[n]) for n in ("q_r", "k_r", "v_r"))
        plan = self.plan
        n_fws = plan.workspace_bytes(at.OP_REPLAY_FWD)  # split-KV partials (short queues only)
        self.ws_f = torch.empty(n_fws, dtype=torch.uint8, device=dev) if n_fws else None
        if fused:
            self.ws_t = torch.empty(max(1, plan.workspace_bytes(at.OP_TREE_BWD)), dtype=torch.uint8, device=dev)
        else:
            self.dkp_sum = torch.empty(t["k_p"].shape, dtype=f32, device=dev)
            self.dvp_sum = torch.empty(t["v_p"].shape, dtype=f32, device=dev)
            self.ws_r = torch.empty(max(1, plan.workspace_bytes(at.OP_REPLAY_BWD)), dtype=torch.uint8, device=dev)
            self.ws_p = torch.empty(max(1, plan.workspace_bytes(at.OP_PREFILL_BWD)), dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream()
        self.n_ev = 4 if fused else 5

    def outputs(self):
        return [self.o_p, self.o_r, self.lse_p, self.lse_r, self.dq_p, self.dk_p, self.dv_p, self.dq_r, self.dk_r,
                self.dv_r]

    def step(self, evs=None):
        at, t, s, plan = self.at, self.t, self.stream, self.plan
        rec = (lambda i: evs[i].record(s)) if evs else (lambda i: None)
        rec(0)
        at.augtree_prefill_fwd(plan, t["q_p"], t["k_p"], t["v_p"], self.o_p, self.lse_p, stream=s)
        rec(1)
        at.augtree_replay_fwd(plan, t["q_r"], t["k_p"], t["v_p"], t["k_r"], t["v_r"], self.o_r, self.lse_r, self.ws_f,
                              stream=s)
        rec(2)
        if self.fused:
            at.augtree_tree_bwd(plan, t["q_p"], t["k_p"], t["v_p"], self.o_p, self.lse_p, t["do_p"], t["q_r"],
                                t["k_r"], t["v_r"], self.o_r, self.lse_r, t["do_r"], self.dq_p, self.dk_p, self.dv_p,
                                self.dq_r, self.dk_r, self.dv_r, self.ws_t, stream=s)
            rec(3)
            return
        at.augtree_replay_bwd(plan, t["q_r"], t["k_p"], t["v_p"], t["k_r"], t["v_r"], self.o_r, self.lse_r,
                              t["do_r"], self.dq_r, self.dk_r, self.dv_r, self.dkp_sum, self.dvp_sum, self.ws_r,
                              stream=s)
        rec(3)
        at.augtree_prefill_bwd(plan, t["q_p"], t["k_p"], t["v_p"], self.o_p, self.lse_p, t["do_p"], self.dkp_sum,
                               self.dvp_sum, self.dq_p, self.dk_p, self.dv_p, self.ws_p, stream=s)
        rec(4)

    def close(self):
        import torch
        self.plan.close()
        for k in list(vars(self)):
            if k not in ("w", "at", "dev", "fused", "n_ev"):
                delattr(self, k)
        torch.cuda.empty_cache()


def barrier(world):
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()


def measure(run, steps, warmup, world, local, sample_clocks=True):
    """Times `steps` fwd+bwd steps after `warmup` untimed ones (CUDA events on the calls'
    stream, barrier + synchronize on both sides) with per-kernel CUDA events recorded by
    the library.  Returns a dict of the step time (max over ranks), the per-call and
    per-kernel times and the sampled clocks."""
    import torch
    at, plan = run.at, run.plan
    for _ in range(warmup):
        run.step()
    barrier(world)
    clocks = ClockSampler(local) if sample_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(run.n_ev)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    plan.set_timing(steps <= at.TIMING_RING)
    barrier(world)
    start.record(run.stream)
    for k in range(steps):
        run.step(evs[k])
    end.record(run.stream)
    barrier(world)
    clk = clocks.stop() if clocks else None
    plan.check()  # raises if any kernel of the step gave up on a bounded wait
    kernel_ms = {}  # (op, kind) -> [ms per step summed over the step's launches, launches]
    if steps <= at.TIMING_RING:
        for op in range(5):
            for back in range(steps):
                try:
                    kt = plan.kernel_times(op, back)
                except at.AugtreeError:  # the step makes no timed call of this op
                    break
                for kind, t_ms in kt:
                    e = kernel_ms.setdefault((op, kind), [0.0, 0])
                    e[0] += t_ms / steps
                    e[1] += 1
        plan.set_timing(False)
    ms = max_over_ranks(start.elapsed_time(end), run.dev) / steps
    per_call = np.array([[evs[k][i].elapsed_time(evs[k][i + 1]) for i in range(run.n_ev - 1)]
                         for k in range(steps)]).mean(0)
    ms_median = float(np.median([evs[k][0].elapsed_time(evs[k][run.n_ev - 1]) for k in range(steps)]))
    return {"ms": ms, "ms_median": ms_median, "per_call": per_call, "kernel_ms": kernel_ms, "clocks": clk}


# GEMMs a kernel performs per valid pair (2 D Hq FLOPs each): forward S and PV; key side
# S^T, dP^T, dV, dK; query side S, dP, dQ; SIMT backward all five.
GEMMS = {"fwd_tc": 2, "fwd_simt": 2, "bwd_key_side": 4, "bwd_query_side": 3, "bwd_simt": 5}
KERNEL_NAMES = {"bwd_key_side": "tc_bwd_kv_kernel (backward, key side)",
                "bwd_query_side": "tc_bwd_dq_kernel (backward, query side)",
                "fwd_tc": "tc_fwd_kernel (forward)"}


def kernel_table(w, m):
    """Per kernel kind: [ms per step, launches per step, GEMM FLOPs per step]."""
    n_pairs_prompt = sum(lp * (lp + 1) // 2 for lp in w.tree.prompt_lens)
    n_pairs = w.tree.pair_count()
    pairs = {0: n_pairs_prompt, 1: n_pairs - n_pairs_prompt, 2: n_pairs - n_pairs_prompt, 3: n_pairs_prompt,
             4: n_pairs}
    steps = None
    kinds = {}
    for (op, kind), (t_ms, launches) in m["kernel_ms"].items():
        e = kinds.setdefault(kind, [0.0, 0, 0.0])
        e[0] += t_ms
        e[1] += launches
        e[2] += 2.0 * w.d * w.hq * pairs[op] * GEMMS.get(kind, 0)
    return kinds


def roofline(w, m, steps, peak_s, pk_kind):
    """The dominant kernel's live roofline: its GEMM FLOPs per step over its measured
    time per step (the library's CUDA events around each launch)."""
    kinds = kernel_table(w, m)
    if not kinds:
        return None, {}
    dom = max(kinds, key=lambda k: kinds[k][0])
    ms_k, launches, flops_k = kinds[dom]
    ach = flops_k / (ms_k * 1e-3) / 1e12
    traffic, note = traffic_entry(w.name, dom)
    return ({"bound": "tensor", "kernel": KERNEL_NAMES.get(dom, dom), "achieved": round(ach, 2), "peak": peak_s,
             "unit": "TFLOP/s", "frac": round(ach / peak_s, 4), "traffic": traffic, "traffic_source": note,
             "launches_per_step": launches / steps, "peak_kind": f"bf16 dense sustained ({pk_kind})"},
            {k: {"ms_per_step": round(v[0], 4), "launches_per_step": v[1] / steps,
                 "tflops": round(v[2] / (v[0] * 1e-3) / 1e12, 2) if v[2] > 0 else None}
             for k, v in sorted(kinds.items(), key=lambda kv: -kv[1][0])})


def run_ours(args):
    import torch
    import shared_prompt_tree_gb300 as at
    import workloads as W

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.workload(args.workload)
    if args.scale_down > 1:
        w = scaled_down(w, args.scale_down)
    kernel = {"auto": at.KERNEL_AUTO, "simt": at.KERNEL_SIMT, "tc": at.KERNEL_TC}[args.kernel]
    fused = args.bwd == "fused"
    sched = {"queue": at.SCHED_QUEUE, "persistent": at.SCHED_PERSISTENT}[args.schedule]
    run = Run(w, at, dev, kernel, fused, sched)
    m = measure(run, args.steps, args.warmup, world, local)
    ms_step = m["ms"]

    # e2e through the public API with host buffers: every step copies its inputs from
    # pinned host memory to the device, runs, and copies its results (outputs and all
    # gradients) back to pinned host memory, all inside the timed region.  The copies
    # are pipelined the way a trainer would: two device buffer sets, a copy-in and a
    # copy-out stream, so step k+1's inputs and step k-1's results move while step k
    # computes.
    host_in = {n: run.t[n].cpu().pin_memory() for n in W.TENSORS}
    host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in run.outputs()]
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in run.outputs())
    e_steps = max(2, min(args.steps, 10))
    runs = [run, Run(w, at, dev, kernel, fused, sched)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev() for _ in range(e_steps)], [ev() for _ in range(e_steps)], \
        [ev() for _ in range(e_steps)]
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(run.stream)
    s_in.wait_event(e0)
    for k in range(e_steps):
        rk = runs[k % 2]
        if k >= 2:
            s_in.wait_event(comp_done[k - 2])     # step k-2 has read this buffer set's inputs
        with torch.cuda.stream(s_in):
            for n in W.TENSORS:
                rk.t[n].copy_(host_in[n], non_blocking=True)
            in_done[k].record(s_in)
        run.stream.wait_event(in_done[k])
        if k >= 2:
            run.stream.wait_event(out_done[k - 2])  # step k-2's results have left this set
        rk.step()
        comp_done[k].record(run.stream)
        s_out.wait_event(comp_done[k])
        with torch.cuda.stream(s_out):
            for x, hx in zip(rk.outputs(), host_out):
                hx.copy_(x, non_blocking=True)
            out_done[k].record(s_out)
    run.stream.wait_event(out_done[e_steps - 1])
    e1.record(run.stream)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, dev)
    launches_per_step = count_launches(run.plan, at, fused)
    del host_in, host_out
    for r_ in runs:
        r_.close()

    flops = useful_flops(w)
    tflops = flops * world / (ms_step * 1e-3) / 1e12
    pk, pk_kind = peaks()
    peak_s = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    n_pairs_prompt = sum(lp * (lp + 1) // 2 for lp in w.tree.prompt_lens)
    n_pairs = w.tree.pair_count()
    if fused:
        names = ["prefill_fwd", "replay_fwd", "tree_bwd"]
        per_flops = [4 * w.d * w.hq * n_pairs_prompt, 4 * w.d * w.hq * (n_pairs - n_pairs_prompt),
                     10 * w.d * w.hq * n_pairs]
    else:
        names = ["prefill_fwd", "replay_fwd", "replay_bwd", "prefill_bwd"]
        per_flops = [4 * w.d * w.hq * n_pairs_prompt, 4 * w.d * w.hq * (n_pairs - n_pairs_prompt),
                     10 * w.d * w.hq * (n_pairs - n_pairs_prompt), 10 * w.d * w.hq * n_pairs_prompt]
    roof, ktab = roofline(w, m, args.steps, peak_s, pk_kind)

    result = {
        "metric": "tree-attn fwd+bwd useful TFLOP/s & tokens/s; % of GB300 BF16 tensor peak",
        "value": round(tflops, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "median_ms_per_step": round(m["ms_median"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "fp32",
        "data": "synthetic (seeded counter-hash N(0,1) values, bf16-rounded)",
        "config": {"workload": w.name, "groups": w.tree.n_groups, "prompt_lens": w.tree.prompt_lens[:4],
                   "branches": w.tree.n_branches, "total_prompt": w.tree.total_prompt,
                   "total_resp": w.tree.total_resp, "hq": w.hq, "hkv": w.hkv, "head_dim": w.d,
                   "parallelism": f"replicas x{world}", "kernel_family": args.kernel,
                   "backward": "one augtree_tree_bwd call" if fused else "augtree_replay_bwd + augtree_prefill_bwd",
                   "schedule": args.schedule,
                   "l2": "inputs larger than L2 (no flush)"},
        "tokens_per_s": round(w.tokens * world / (ms_step * 1e-3), 1),
        "flattened_tokens_per_s": round(w.tree.flattened_tokens() * world / (ms_step * 1e-3), 1),
        "pct_of_bf16_peak": round(100.0 * tflops / world / pk["bf16_tflops"], 2),
        "per_call_ms": {n: round(float(x), 4) for n, x in zip(names, m["per_call"])},
        "per_call_tflops": {n: round(f / (x * 1e-3) / 1e12, 2) for n, f, x in zip(names, per_flops, m["per_call"])},
        "roofline": roof,
        "kernels": ktab,
        "e2e": {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e_steps,
                "copies": "pinned host memory; H2D of step k+1 and D2H of step k-1 overlap step k "
                          "(two device buffer sets, copy-in and copy-out streams)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": m["clocks"],
    }
    if not args.no_flattened:
        # The same trees with no prompt reuse (every pair on its own): the speedup of the
        # shared-prompt tree over flattening, measured with the same kernels and the same
        # fused backward.
        wf = flattened(w)
        rf = Run(wf, at, dev, kernel, fused, sched)
        mf = measure(rf, max(1, min(args.steps, 3)), 1, world, local, sample_clocks=False)
        rf.close()
        result["flattened_per_pair"] = {
            "ms_per_step": round(mf["ms"], 3), "pairs": wf.tree.pair_count(), "tree_pairs": w.tree.pair_count(),
            "speedup_of_tree": round(mf["ms"] / ms_step, 3), "steps": max(1, min(args.steps, 3)),
            "backward": result["config"]["backward"]}
    if not args.no_split_kv and args.scale_down == 1 and w.dtype == "bf16" and kernel != at.KERNEL_SIMT:
        result["split_kv_replay_fwd"] = split_kv_probe(at, dev)
    if not args.no_per_workload and args.scale_down == 1:
        # The other bf16 configurations, each timed the same way (fewer steps for the
        # long one, whose step takes seconds).
        per = {}
        for name in [n for n in ("prompt_heavy", "response_heavy", "mixed", "long") if n != w.name]:
            wo = W.workload(name)
            st, wu = (2, 1) if name == "long" else (args.steps, args.warmup)
            ro = Run(wo, at, dev, kernel, fused, sched)
            mo = measure(ro, st, wu, world, local)
            ro.close()
            tf = useful_flops(wo) * world / (mo["ms"] * 1e-3) / 1e12
            roof_o, ktab_o = roofline(wo, mo, st, peak_s, pk_kind)
            per[name] = {"ms_per_step": round(mo["ms"], 4), "steps": st, "warmup": wu,
                         "useful_tflops": round(tf, 3), "pct_of_bf16_peak": round(100.0 * tf / world / pk["bf16_tflops"], 2),
                         "tokens_per_s": round(wo.tokens * world / (mo["ms"] * 1e-3), 1),
                         "roofline": roof_o, "kernels": ktab_o, "clocks": mo["clocks"]}
        result["per_workload"] = per
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, per_rep = time_oracle(w, min_seconds=args.cpu_seconds)
        result["cpu_baseline"] = oracle_fields(rate, desc, w)
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def split_kv_probe(at, dev, reps=20):
    """Replay forward of a queue too short for the GPU: one 8,192-token prompt under 32
    branches of 3 tokens (Hq 32, Hkv 8, one 128-row query tile, 16 two-head blocks when
    whole).  The split-KV queue (the device's SM count as balancing width) against the
    same tile unsplit (balancing width 1), CUDA events around `reps` calls each; the
    split call's kernels (forward and the merge of the partial states) from the plan's
    kernel timing."""
    import torch
    import workloads as W
    w = W.custom(W.Tree([8192], [[3] * 32]), hq=32, hkv=8, d=128, dtype="bf16", seed=5)
    t = {n: W.tensor_torch(w, n, dev) for n in ("q_r", "k_p", "v_p", "k_r", "v_r")}
    out = {"tree": "prompt 8192, 32 branches x 3 tokens, Hq 32, Hkv 8, D 128, bf16"}
    for label, sms in (("split", 0), ("whole", 1)):
        plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC, num_sms=sms)
        o = torch.empty_like(t["q_r"])
        lse = torch.empty(w.hq, w.tree.total_resp, dtype=torch.float32, device=dev)
        nb = plan.workspace_bytes(at.OP_REPLAY_FWD)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
        call = lambda: at.augtree_replay_fwd(plan, t["q_r"], t["k_p"], t["v_p"], t["k_r"], t["v_r"], o, lse, ws)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize()
        q = plan.schedule(at.OP_REPLAY_FWD)
        row = {"ms": round(e0.elapsed_time(e1) / reps, 4), "items": int(len(q)),
               "splits_per_tile": int(q[:, 4].max()) + 1, "workspace_bytes": int(nb)}
        if label == "split":
            plan.set_timing(True)
            call()
            torch.cuda.synchronize()
            row["kernels_ms"] = {k: round(m, 4) for k, m in plan.kernel_times(at.OP_REPLAY_FWD)}
        plan.check()
        plan.close()
        out[label] = row
    out["speedup"] = round(out["whole"]["ms"] / out["split"]["ms"], 3)
    return out


def flattened(w):
    """The workload with every prompt-response pair as its own group: each branch carries
    its own copy of its group's prompt, so the prompt is prefilled and attended once per
    branch (the no-reuse baseline the pages compare against, on this GPU)."""
    import workloads as W
    prompts, branches = [], []
    for lp, bl in zip(w.tree.prompt_lens, w.tree.branch_lens):
        if not bl:
            prompts.append(lp)
            branches.append([])
        for li in bl:
            prompts.append(lp)
            branches.append([li])
    return W.custom(W.Tree(prompts, branches), w.hq, w.hkv, w.d, w.dtype, w.seed, w.scale, name=f"{w.name}/flattened")


def scaled_down(w, k):
    """The workload's structure with every length divided by k (profiling cases)."""
    import workloads as W
    tree = W.Tree([max(1, x // k) for x in w.tree.prompt_lens], [[max(1, x // k) for x in b] for b in w.tree.branch_lens])
    return W.custom(tree, w.hq, w.hkv, w.d, w.dtype, w.seed, w.scale, name=f"{w.name}/{k}")


def count_launches(plan, at, fused=False):
    """Kernels one step launches: prefill fwd 1, replay fwd 1 (plus the split-KV merge
    when the replay queue is split); then either the fused backward (preprocess per
    side, key side, split reduce when a group is split, query side per side, the
    split-KV dQ sum) or replay bwd 4 (preprocess, key side, split reduce, query side;
    plus the dQ sum) and prefill bwd 3."""
    n = 0
    n += 1 if plan.schedule(at.OP_PREFILL_FWD).shape[0] else 0
    qf = plan.schedule(at.OP_REPLAY_FWD)
    fsplit = bool(qf.shape[0]) and bool((qf[:, 4] > 0).any())
    n += (1 if qf.shape[0] else 0) + (1 if fsplit else 0)
    if fused:
        q = plan.schedule(at.OP_TREE_BWD)
        split = bool(q.shape[0]) and bool((q[:, 4] > 0).any())
        n += 2 * (1 if plan.total_resp else 0) + 2 * (1 if plan.total_prompt else 0)
        n += (1 if q.shape[0] else 0) + (1 if split else 0) + (1 if fsplit else 0)
        return n
    n += 1 if fsplit else 0
    n += (1 if plan.total_resp else 0) + (1 if plan.schedule(at.OP_REPLAY_BWD).shape[0] else 0) \
        + (1 if plan.total_prompt else 0) + (1 if plan.total_resp else 0)
    n += 3 if plan.total_prompt else 0
    return n


def run_reference(args):
    """Reference arm: the fp64 CPU oracle, as it stands, on the host cores.  Each step
    is a bounded sample of the workload (see oracle_sample)."""
    world, rank, local = dist_setup()
    if rank != 0:
        return
    import workloads as W
    from oracle import attention as A
    w = W.workload(args.workload)
    sample, desc = oracle_sample(w)
    t = {n: W.tensor_rows_np(sample, n) for n in W.TENSORS}
    flops = useful_flops(sample)
    for _ in range(args.warmup):
        A.tree_attention_direct(t, sample.tree.offsets(), A.default_scale(sample.d))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        A.tree_attention_direct(t, sample.tree.offsets(), A.default_scale(sample.d))
    el = time.perf_counter() - t0
    rate = flops * args.steps / el / 1e12
    res = {"impl": "reference", "metric": "tree-attn fwd+bwd useful TFLOP/s & tokens/s; % of GB300 BF16 tensor peak",
           "value": round(rate, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
           "config": {"workload": w.name, "sample": desc},
           "cpu_baseline": oracle_fields(rate, desc, w),
           "e2e": {"value": round(rate, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def spawn_replicas(n: int) -> int:
    """`--gpus N` without a launcher: re-runs this script under torch.distributed.run
    with N ranks on this node (one GPU each), passing the same arguments.  Returns the
    launcher's exit code."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.run(cmd).returncode


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--kernel", choices=["auto", "simt", "tc"], default="auto")
    ap.add_argument("--bwd", choices=["fused", "two-call"], default="fused",
                    help="backward as one augtree_tree_bwd call, or replay_bwd then prefill_bwd")
    ap.add_argument("--schedule", choices=["queue", "persistent"], default="queue",
                    help="one block per work unit (queue) or persistent blocks on AssignGrid lanes")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scale-down", type=int, default=1, help="divide every length by this (profiling only)")
    ap.add_argument("--no-flattened", action="store_true",
                    help="skip timing the flattened-per-pair structure (no prompt reuse)")
    ap.add_argument("--no-per-workload", action="store_true", help="skip timing the other configurations")
    ap.add_argument("--no-split-kv", action="store_true",
                    help="skip timing the split-KV replay forward of a short-response tree")
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_replicas(args.gpus))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
