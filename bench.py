"""Benchmark of the block-FP8 MoE FFN layer on GB300.

One pass = one full layer forward (router, softmax/top-k, permutation,
gate/up + SwiGLU, down projection, combine) over one batch of synthetic tokens;
one step = M passes replayed from a CUDA graph (below).  The headline workload
is the Qwen3-MoE-shaped decode layer (hidden 2048, expert intermediate 768,
128 experts, top-8, block-FP8 E4M3 weights with 128x128 fp32 scales) at a
batch of 64 tokens.

Timing: each step replays one CUDA graph of M layer passes (each pass the
whole hot path over the batch) that rotate over R device copies of the layer,
R chosen so that R copies span at least 4x the L2 (a pass never finds the
previous passes' weights in L2, as when stepping through a model's layers);
M is chosen so the K timed steps last about 1.5 s, long enough for the
nvidia-smi clock samples taken meanwhile.  W warm-up steps, then K steps, each
bracketed by CUDA events on the launching stream; L2 is also flushed (a
512 MiB write) before every step, outside the events.  Max over ranks; under
torchrun each rank runs its own replica of the layer on its own tokens (weak
scaling, no collective in the data path).

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on a bounded token sample instead.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_inputs as mi  # noqa: E402

HEADLINE = ("qwen3moe_decode", 64)
METRIC = "MoE-layer tokens/s at decode & prefill; HBM GB/s or TC util vs GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["_source"] = "fallback"
    return d


def expert_bytes(H, I):
    """Codes + scales of one expert's gate, up and down matrices."""
    nb = lambda n: -(-n // 128)
    return 3 * H * I + 4 * (2 * nb(I) * nb(H) + nb(H) * nb(I))


def algorithmic(w: mi.Workload, T: int, D: int):
    """Bytes and FLOPs the layer must move/compute for one call: router
    weights, the D distinct experts hit (plus the shared expert), the tokens in
    and the output out; FLOPs of the router and of every (token, expert) pair."""
    B = w.E * w.H * 4 + D * expert_bytes(w.H, w.I) + 2 * T * w.H * 2
    F = T * w.k * 6 * w.H * w.I + 2 * T * w.H * w.E
    if w.I_shared:
        B += expert_bytes(w.H, w.I_shared)
        F += T * 6 * w.H * w.I_shared
    expert_B = D * expert_bytes(w.H, w.I) + T * w.H * 2
    if w.I_shared:
        expert_B += expert_bytes(w.H, w.I_shared)
    return B, F, expert_B


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def file_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_traffic(kernel_key: str, src_files):
    """DRAM bytes per launch from the committed ncu summary, only while the
    kernel sources still hash to the value the counters were taken at."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        table = json.load(f)
    ent = table.get(kernel_key)
    if not ent or ent.get("src_hash") != file_hash(src_files):
        return None
    return ent.get("bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------

def oracle_rate(layer, x_bits, reps=1):
    import oracle
    t = time.perf_counter()
    for _ in range(reps):
        oracle.moe_layer(x_bits, layer, keep_intermediates=False)
    dt = (time.perf_counter() - t) / reps
    return x_bits.shape[0] / dt, dt


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    global HEADLINE
    nm, tt = args.workload.split(":")
    HEADLINE = (nm, int(tt))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    name, T = HEADLINE
    w = mi.WORKLOADS[name]
    layer = mi.make_layer(name, seed=0)
    x_bits, _ = mi.make_tokens(layer, T, seed=0)
    # Bound the whole run to about two minutes of CPU time whatever K and W
    # are: time one small sample, then size every step's token sample.
    probe = oracle_rate(layer, x_bits[:1])[1]
    budget = 120.0 / (args.steps + args.warmup)
    sample = int(max(1, min(16, T, budget / max(probe, 1e-3))))
    xs = x_bits[:sample]
    for _ in range(args.warmup):
        oracle_rate(layer, xs)
    times = []
    for _ in range(args.steps):
        times.append(oracle_rate(layer, xs)[1])
    dt = sum(times) / len(times)
    val = sample / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{name}_T{T}", "H": w.H, "I": w.I, "E": w.E, "k": w.k,
                   "T": T, "sample_tokens_per_step": sample},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                         "sample": f"{sample} of the {T} tokens per step, fp64 NumPy oracle"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class LayerRun:
    """A captured layer forward for one (layer, T) with static buffers."""

    def __init__(self, torch, D, x_bits, graph=True, act8=False):
        from block_fp8_expert_gb300.device import x_to_device
        self.torch = torch
        self.D = D
        self.act8 = act8  # E4M3 activations (moe_layer_forward_act8)
        self.T = x_bits.shape[0]
        self.x = x_to_device(x_bits)
        self.out = torch.empty((self.T, D.H), dtype=torch.bfloat16, device="cuda")
        self.idx = torch.empty((self.T, D.k), dtype=torch.int32, device="cuda")
        self.w = torch.empty((self.T, D.k), dtype=torch.float32, device="cuda")
        self.ws = D.workspace(self.T)
        self.graph = None
        self.launches = None
        self.fwd()
        torch.cuda.synchronize()
        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                self.fwd()
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            from block_fp8_expert_gb300 import _lib
            self.graph = torch.cuda.CUDAGraph()
            n0 = _lib.kernel_launches()
            with torch.cuda.graph(self.graph):
                self.fwd()
            torch.cuda.synchronize()
            # this library's kernels in one captured layer call
            self.launches = _lib.kernel_launches() - n0

    def fwd(self):
        self.D.forward(self.x, out=self.out, ws=self.ws, topk_idx=self.idx, topk_w=self.w,
                       act8=self.act8)

    def step(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self.fwd()

    def distinct_experts(self):
        return int(np.unique(self.idx.cpu().numpy()).size)

    def device_status(self):
        """The workspace's status word and the record of any bounded wait that
        ran out (words 1-5), after the timed steps."""
        return self.ws[:24].view(self.torch.int32).cpu().numpy()[:6].tolist()


class PassGraph:
    """M layer passes rotating over R device copies of one layer, captured as
    one CUDA graph (one replay = one timed step).  The copies hold the same
    weights at different addresses, so a pass reads its weights from HBM
    whenever R copies exceed the L2."""

    def __init__(self, torch, D, host, x_bits, R, M, act8=False):
        from block_fp8_expert_gb300 import _lib
        from block_fp8_expert_gb300.device import DeviceLayer
        self.torch = torch
        self.R, self.M = R, M
        self.runs = [LayerRun(torch, D, x_bits, graph=False, act8=act8)]
        for _ in range(R - 1):
            self.runs.append(LayerRun(torch, DeviceLayer.from_host(host), x_bits, graph=False,
                                      act8=act8))
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for r in self.runs:
                r.fwd()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        n0 = _lib.kernel_launches()
        with torch.cuda.graph(self.graph):
            for p in range(M):
                self.runs[p % R].fwd()
        torch.cuda.synchronize()
        self.launches_per_pass = (_lib.kernel_launches() - n0) / M

    def step(self):
        self.graph.replay()

    def device_status(self):
        return max((r.device_status() for r in self.runs), key=lambda v: v[0] != 0)


def copies_for_l2(torch, bytes_per_pass, most=64):
    """Device copies of a layer so that a rotation over them touches at least
    4x the L2 between two visits of the same copy (at least 2, at most
    `most`: a layer of under 4x L2 / most bytes stays partly L2-resident)."""
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    return min(most, max(2, -(-4 * l2 // max(1, bytes_per_pass))))


def single_pass_time(torch, run, flush, n=5):
    """Mean time of one graph-replayed pass (L2 flushed before each)."""
    return sum(time_steps(torch, run.step, n, 3, flush)) / n


def passes_per_step(t_pass, steps, R, target_s, max_passes=4096):
    """M, a multiple of R, so that `steps` steps of M passes last about
    target_s."""
    m = int(target_s / max(steps * t_pass, 1e-9))
    m = max(R, min(max_passes, m))
    return -(-m // R) * R


def aggregate(t_rank: float, world: int, tokens_per_rank: int, steps: int, dist=None,
              device=None):
    """Whole-job throughput from each rank's summed step time: the slowest
    rank's time (max over ranks) bounds the job; every rank processed
    tokens_per_rank tokens per step.  Returns (tokens/s, max time)."""
    t_all = t_rank
    if dist is not None and world > 1:
        import torch
        tt = torch.tensor([t_rank], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t_all = float(tt.item())
    return world * tokens_per_rank * steps / t_all, t_all


# Nominal GB300 figures, for context beside the measured denominators.
NOMINAL_HBM_GBS = 7900.0


def other_denominators(pk, gbs, tflops, act8=False):
    """The same achieved figures against the nominal HBM rate and, for the
    contraction, the measured sustained bf16 rate (x2 for fp8)."""
    out = {"frac_hbm_nominal_7900gbs": gbs / NOMINAL_HBM_GBS}
    sus = pk.get("bf16_tflops_sustained")
    if sus:
        out["frac_tc_sustained"] = tflops / (sus * (2.0 if act8 else 1.0))
    return out


def step_stats(times, per=1):
    """Median, min, 90th percentile and max of the step times in ms, each
    divided by `per` (the passes a step replays), next to the mean that the
    line reports."""
    v = sorted(t * 1e3 / per for t in times)
    if not v:
        return None
    p90 = v[min(len(v) - 1, int(math.ceil(0.9 * len(v))) - 1)]
    return {"median": statistics.median(v), "min": v[0], "p90": p90, "max": v[-1],
            "n": len(v)}


def time_steps(torch, fn, steps, warmup, flush):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) * 1e-3)
    return times


def _nvtx_range(torch, name, fn):
    """fn() inside an NVTX push/pop range (host-side marker only; lets a
    profiler select the expert-FFN call's kernels: `--nvtx --nvtx-include
    moe_expert_ffn_fp8/`)."""
    torch.cuda.nvtx.range_push(name)
    try:
        return fn()
    finally:
        torch.cuda.nvtx.range_pop()


def record_traffic(csv_path, workload):
    """Store the DRAM bytes per expert-FFN call from an ncu CSV (metrics
    dram__bytes_read.sum and dram__bytes_write.sum of the kernels inside the
    `moe_expert_ffn_fp8` NVTX range) in profiles/dram_traffic.json under the
    workload's key, with the hash of the sources it was measured on."""
    import csv
    import collections
    rows = list(csv.reader(open(csv_path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    hdr = rows[hi]
    ki, mi_, vi, ii = (hdr.index("Kernel Name"), hdr.index("Metric Name"),
                       hdr.index("Metric Value"), hdr.index("ID"))
    per = collections.defaultdict(lambda: collections.defaultdict(float))
    for r in rows[hi + 1:]:
        if len(r) <= vi or r[mi_] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        unit = r[hdr.index("Metric Unit")] if "Metric Unit" in hdr else "byte"
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(unit, 1)
        name = r[ki].split("(")[0].replace("void ", "").replace("moe::", "")
        if name.startswith("k_"):  # this library's kernels only (not torch's fills)
            per[name][r[ii]] += float(r[vi].replace(",", "")) * scale
    kern = {k: sum(v.values()) / len(v) for k, v in per.items()}
    gemm = any("k_expert_ffn_ws" in k for k in kern)
    nm, T = workload.split(":")
    csrc = os.path.join("block_fp8_expert_gb300", "csrc")
    files = ["expert_gemm_tc.cu", "tcgen05.cuh", "moe_common.cuh"] if gemm else \
        ["expert_gemv.cu", "moe_common.cuh"]
    src = [os.path.join(csrc, f) for f in files]
    key = f"expert_ffn_{'gemm' if gemm else 'gemv'}_{nm}_T{T}"
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    table = json.load(open(path)) if os.path.exists(path) else {}
    table[key] = {
        "what": f"DRAM bytes (read + write) of one moe_expert_ffn_fp8 call at {nm} T={T}",
        "bytes_per_launch": int(round(sum(kern.values()))),
        "per_kernel": {k: int(round(v)) for k, v in kern.items()},
        "src_hash": file_hash([os.path.join(ROOT, f) for f in src]),
        "src": src,
        "command": f"ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,"
                   f"dram__bytes_write.sum --clock-control none --nvtx --nvtx-include "
                   f"moe_expert_ffn_fp8/ -c 10 --csv --log-file traffic.csv python bench.py "
                   f"--workload {workload} --steps 3 --warmup 3 --no-sweep --no-cpu-baseline "
                   f"--max-passes 2; python bench.py --record-traffic traffic.csv "
                   f"--workload {workload}",
        "note": "per kernel: the mean over its captured launches; the call's total is "
                "their sum"}
    with open(path, "w") as f:
        json.dump(table, f, indent=1)
        f.write("\n")
    print(json.dumps({key: table[key]}, indent=1))
    return 0


def phase_times(torch, D, run, steps, flush):
    """Per ABI call timing of one forward, split into route / permute /
    experts / combine (each call timed with events on the same stream)."""
    import block_fp8_expert_gb300 as m
    T = run.T
    d = D.dims(T)
    P = T * D.k
    dev = "cuda"
    idx = torch.empty((T, D.k), dtype=torch.int32, device=dev)
    w = torch.empty((T, D.k), dtype=torch.float32, device=dev)
    off = torch.empty(D.E + 1, dtype=torch.int32, device=dev)
    rt = torch.empty(P, dtype=torch.int32, device=dev)
    tsr = torch.empty(P, dtype=torch.int32, device=dev)
    y = torch.empty((P, D.H), dtype=torch.float32, device=dev)
    sy = None
    out = torch.empty((T, D.H), dtype=torch.bfloat16, device=dev)
    ws = run.ws
    calls = {
        "route": lambda: m.moe_route(run.x, D.Wr, D.bias, d, idx, w, ws),
        "permute": lambda: m.moe_permute(idx, d, off, rt, tsr, ws),
        "experts": lambda: _nvtx_range(torch, "moe_expert_ffn_fp8", lambda: m.moe_expert_ffn_fp8(
            run.x, off, rt, D.routed.abi(), d, y, ws)),
        "combine": lambda: m.moe_combine(y, tsr, w, sy, d, out),
    }
    res = {k: [] for k in calls}
    for it in range(steps + 2):
        flush()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
        ev[0].record()
        for i, f in enumerate(calls.values()):
            f()
            ev[i + 1].record()
        ev[-1].synchronize()
        if it >= 2:
            for i, k in enumerate(calls):
                res[k].append(ev[i].elapsed_time(ev[i + 1]) * 1e-3)
    return {k: sum(v) / len(v) for k, v in res.items()}


def measure_workload(torch, name, T, steps, warmup, flush, pk, dev_cache, seed=0,
                     target_s=0.4, act8=False):
    """One sweep entry: `steps` steps of M passes over rotating copies (about
    target_s of timed work), with its own clock record.  act8: the layer on
    E4M3 activations, whose contraction runs on the fp8 tensor rate (the
    measured bf16 peak times the nominal 4.5 / 2.25 ratio)."""
    from block_fp8_expert_gb300.device import DeviceLayer
    w = mi.WORKLOADS[name]
    key = (w.H, w.I, w.E, w.k, w.I_shared, w.zipf_s)
    if key not in dev_cache:
        dev_cache.clear()
        torch.cuda.empty_cache()
        host = mi.make_layer(w, seed=seed)
        dev_cache[key] = (host, DeviceLayer.from_host(host))
    host, D = dev_cache[key]
    x_bits, _ = mi.make_tokens(host, T, seed=seed)
    run = LayerRun(torch, D, x_bits, act8=act8)
    Dn = run.distinct_experts()
    B, F, _ = algorithmic(w, T, Dn)
    R = copies_for_l2(torch, B)
    M = passes_per_step(single_pass_time(torch, run, flush), steps, R, target_s)
    pg = PassGraph(torch, D, host, x_bits, R, M, act8=act8)
    for _ in range(warmup):
        pg.step()
    torch.cuda.synchronize()
    with Clocks(torch.cuda.current_device()) as clk:
        times = time_steps(torch, pg.step, steps, 0, flush)
    t = sum(times) / (len(times) * M)  # per pass
    t_hbm = B / (pk["hbm_gbs"] * 1e9)
    tc_peak = pk["bf16_tflops"] * (2.0 if act8 else 1.0)
    t_tc = F / (tc_peak * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    ck = clk.summary()
    res = {"workload": f"{name}_T{T}" + ("_act8" if act8 else ""), "T": T, "ms": t * 1e3,
           "tokens_per_s": T / t, "tensor_peak_tflops": tc_peak,
           "passes": len(times) * M, "layer_copies": R,
           "device_status": pg.device_status(), "distinct_experts": Dn, "bytes": B,
           "flops": F, "hbm_gbs": B / t / 1e9, "tflops": F / t / 1e12, "bound": bound,
           "ms_stats": step_stats(times, M),
           "other_denominators": other_denominators(pk, B / t / 1e9, F / t / 1e12, act8),
           "roofline_frac": max(t_hbm, t_tc) / t, "clocks": ck,
           "kcycles": t * ck["sm_mhz"] * 1e3 if ck["sm_mhz"] else None}
    del pg
    return res, run, D, host


def run_gpu(args):
    import torch
    global HEADLINE
    nm, tt = args.workload.split(":")
    HEADLINE = (nm, int(tt))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from block_fp8_expert_gb300 import build
    build.build()
    import block_fp8_expert_gb300 as m
    m.lib()
    pk = peaks()
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    flush = lambda: flush_buf.fill_(1)

    name, T = HEADLINE
    w = mi.WORKLOADS[name]
    dev_cache = {}
    # headline: graph replay, K timed steps
    from block_fp8_expert_gb300.device import DeviceLayer
    host = mi.make_layer(name, seed=rank)
    D = DeviceLayer.from_host(host)
    dev_cache[(w.H, w.I, w.E, w.k, w.I_shared, w.zipf_s)] = (host, D)
    x_bits, _ = mi.make_tokens(host, T, seed=rank)
    run = LayerRun(torch, D, x_bits)
    Dn = run.distinct_experts()
    B, F, expert_B = algorithmic(w, T, Dn)
    # M passes per step over R rotating copies: the K steps last ~1.5 s
    R = copies_for_l2(torch, B)
    M = passes_per_step(single_pass_time(torch, run, flush), args.steps, R, 1.5,
                        max_passes=args.max_passes)
    if dist:  # every rank runs the same number of passes
        import torch.distributed as _d
        mt = torch.tensor([M], dtype=torch.int64, device="cuda")
        _d.all_reduce(mt, op=_d.ReduceOp.MAX)
        M = -(-int(mt.item()) // R) * R
    pg = PassGraph(torch, D, host, x_bits, R, M)
    for _ in range(args.warmup):
        pg.step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        times = time_steps(torch, pg.step, args.steps, 0, flush)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    value, t_all = aggregate(sum(times), world, T * M, args.steps, dist, "cuda")
    ms_per_step = t_all / args.steps * 1e3
    ms_per_pass = ms_per_step / M
    headline_status = pg.device_status()
    launches_per_pass = pg.launches_per_pass
    del pg

    # phase table and the dominant unit's roofline: the expert FFN call, on
    # whichever path the library takes for this workload
    ph = phase_times(torch, D, run, max(5, min(args.steps, 20)), flush)
    dom = max(ph, key=ph.get)
    csrc = os.path.join(ROOT, "block_fp8_expert_gb300", "csrc")
    if m.expert_uses_gemm(D.dims(T)):
        kernel = ("expert FFN call: rows gathered into expert order + tcgen05 gate/up+SwiGLU "
                  "GEMM + down GEMM (moe_expert_ffn_fp8)")
        src = [os.path.join(csrc, f) for f in ("expert_gemm_tc.cu", "tcgen05.cuh",
                                               "moe_common.cuh")]
        tkey = f"expert_ffn_gemm_{name}_T{T}"
    else:
        kernel = ("expert FFN call: gate/up+SwiGLU GEMV and down GEMV (moe_expert_ffn_fp8)")
        src = [os.path.join(csrc, f) for f in ("expert_gemv.cu", "moe_common.cuh")]
        tkey = f"expert_ffn_gemv_{name}_T{T}"
    # routed experts only (the moe_expert_ffn_fp8 call): bytes and FLOPs
    expert_F = T * w.k * 6 * w.H * w.I
    t_exp = ph["experts"]
    if expert_B / (pk["hbm_gbs"] * 1e9) >= expert_F / (pk["bf16_tflops"] * 1e12):
        achieved = expert_B / t_exp / 1e9
        roof = {"bound": "hbm", "unit": "GB/s", "kernel": kernel, "achieved": achieved,
                "peak": pk["hbm_gbs"], "peak_source": pk["_source"] + " hbm_gbs",
                "frac": achieved / pk["hbm_gbs"],
                "algorithmic_bytes_per_launch": expert_B}
    else:
        # the call is timed alone (phase table): the burst bf16 figure
        achieved = expert_F / t_exp / 1e12
        roof = {"bound": "tensor", "unit": "TFLOP/s", "kernel": kernel, "achieved": achieved,
                "peak": pk["bf16_tflops"], "peak_source": pk["_source"] + " bf16_tflops",
                "frac": achieved / pk["bf16_tflops"],
                "algorithmic_flops_per_launch": expert_F}
    roof.update({"avg_duration_us": t_exp * 1e6, "traffic": kernel_traffic(tkey, src),
                 "traffic_unit": "DRAM bytes per launch (ncu)"})

    # runtime cross-check of the headline layer call on 16 sampled tokens
    # (independent GPU recomputation; outside every timed region)
    run.step()
    torch.cuda.synchronize()
    verify = D.verify(run.x, run.out, run.idx, run.w, list(range(0, T, max(1, T // 16)))[:16])

    # e2e: host buffers, copies inside the timed region
    x_host = torch.from_numpy(x_bits.view(np.int16)).pin_memory()
    out_host = torch.empty((T, w.H), dtype=torch.int16).pin_memory()

    def e2e_step():
        run.x.view(torch.int16).copy_(x_host, non_blocking=True)
        run.step()
        out_host.copy_(run.out.view(torch.int16), non_blocking=True)

    e2e_times = time_steps(torch, e2e_step, min(args.steps, 500), 3, flush)
    e2e_t = sum(e2e_times) / len(e2e_times)

    # this library's kernels per layer call, counted by the library itself
    # while the passes were captured into the replayed graph
    launches_per_step = int(round(launches_per_pass * M))

    sweep = []
    if not args.no_sweep and rank == 0:
        plan = [("qwen3moe_decode", 1), ("qwen3moe_decode", 8), ("qwen3moe_decode", 64),
                ("qwen3moe_prefill", 4096), ("skewed", 1), ("skewed", 16), ("skewed", 256),
                ("skewed", 2048), ("skewed", 16384), ("large_sparse", 1), ("large_sparse", 256),
                ("tiny", 8), ("qwen3moe_prefill", 4096, True), ("skewed", 2048, True)]
        for nm, tt_, *a8 in plan:
            try:
                r, *_ = measure_workload(torch, nm, tt_, args.sweep_steps, 3, flush, pk,
                                         dev_cache, act8=bool(a8 and a8[0]))
                sweep.append(r)
            except Exception as ex:  # report, do not hide
                sweep.append({"workload": f"{nm}_T{tt_}", "error": repr(ex)[:200]})

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        os.environ.setdefault("OPENBLAS_NUM_THREADS", str(cores()))
        rate, dt = oracle_rate(host, x_bits)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
               "sample": f"one full {name} layer call on all {T} tokens ({dt:.1f} s), "
                         "fp64 NumPy oracle"}

    if rank == 0:
        ck = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 activations in and out, E4M3 weights; fp16 MMA operands, "
                     "fp32 accumulation",
            "data": "synthetic",
            "config": {"workload": f"{name}_T{T}", "H": w.H, "I": w.I, "E": w.E, "k": w.k,
                       "T": T, "weights": "E4M3 codes + fp32 scale per 128x128 block",
                       "distinct_experts": Dn,
                       "passes_per_step": M, "layer_copies": R,
                       "l2": f"each step replays {M} layer passes rotating over {R} device "
                             f"copies of the layer (>= 4x L2 apart); L2 also flushed before "
                             f"every step (512 MiB write)",
                       "graph": "one CUDA graph replay per step",
                       "parallelism": f"replicas{world}"},
            "ms_per_pass": ms_per_pass,
            "kcycles_per_pass": ms_per_pass * ck["sm_mhz"] if ck["sm_mhz"] else None,
            "layer_roofline": {"bytes": B, "flops": F, "achieved_gbs": B / (ms_per_pass * 1e-3) / 1e9,
                               "frac_hbm": B / (ms_per_pass * 1e-3) / 1e9 / pk["hbm_gbs"],
                               **other_denominators(pk, B / (ms_per_pass * 1e-3) / 1e9,
                                                    F / (ms_per_pass * 1e-3) / 1e12)},
            "roofline": roof,
            "phases_us": {k: v * 1e6 for k, v in ph.items()},
            "cpu_baseline": cpu,
            "e2e": {"value": world * T / e2e_t, "unit": "tokens/s",
                    "h2d_bytes_per_step": T * w.H * 2, "d2h_bytes_per_step": T * w.H * 2},
            "gpu_launches": launches_per_step * args.steps,
            "device_status": headline_status,
            "verify": verify,
            "ms_step_max": max(times) * 1e3,
            "ms_per_pass_stats": step_stats(times, M),
            "clocks": ck,
            "sweep": sweep,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_oracle_sweep(args):
    """The fp64 oracle timed on this host's cores on every workload (one full
    layer call each, after a small warm-up call); no GPU is used.  Prints one
    JSON line."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", str(cores()))
    plan = [("tiny", 8), ("qwen3moe_decode", 1), ("qwen3moe_decode", 8),
            ("qwen3moe_decode", 64), ("qwen3moe_prefill", 4096), ("large_sparse", 1),
            ("large_sparse", 256), ("skewed", 1), ("skewed", 16), ("skewed", 256),
            ("skewed", 2048), ("skewed", 16384)]
    rows, cache = [], {}
    for nm, T in plan:
        w = mi.WORKLOADS[nm]
        key = (w.H, w.I, w.E, w.k, w.I_shared, w.zipf_s)
        if key not in cache:
            cache.clear()
            cache[key] = mi.make_layer(w, seed=0)
        layer = cache[key]
        x_bits, _ = mi.make_tokens(layer, T, seed=0)
        oracle_rate(layer, x_bits[:1])  # warm-up (first-call costs)
        rate, dt = oracle_rate(layer, x_bits)
        rows.append({"workload": f"{nm}_T{T}", "seconds": dt, "tokens_per_s": rate})
    print(json.dumps({"oracle_sweep": rows, "cores": cores(), "kind": "oracle",
                      "sample": "one full layer call per workload, fp64 NumPy oracle"}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="%s:%d" % HEADLINE,
                    help="name:T of the timed workload (default: the headline)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--sweep-steps", type=int, default=10)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--max-passes", type=int, default=4096,
                    help="at most this many layer passes per timed step (profiling runs)")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="store an ncu CSV's DRAM bytes per expert-FFN call for --workload "
                         "in profiles/dram_traffic.json and exit (no GPU)")
    ap.add_argument("--oracle-sweep", action="store_true",
                    help="time the fp64 oracle on every workload (host only) and exit")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.record_traffic:
        return record_traffic(args.record_traffic, args.workload)
    if args.oracle_sweep:
        return run_oracle_sweep(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
