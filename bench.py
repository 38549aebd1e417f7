#!/usr/bin/env python3
"""Benchmark of the GB300 SDPA forward (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload caseD] [--quick]

A step is one full forward pass (every stage of the path: QK^T, mask, online softmax,
PV, normalisation, O and LSE stores) over one batch of synthetic inputs of the chosen
workload (default caseD: B=8 H=32 L=512 d=128 causal, the largest head_dim-128 causal
case of "An Optimal Mapper Meets a Real GPU", "Experiment one").

Timing (ours): the K steps are captured in a CUDA graph and replayed, so the number is
device time, not Python launch overhead.  Consecutive steps cycle through R copies of
the inputs and outputs whose total is more than twice the L2 size, so every step reads
its Q, K, V from HBM (no L2 flush needed).  W warm-up steps run first.  A barrier and a
device synchronise bracket the timed region on every rank; the maximum over ranks is
used and rank 0 prints the line.  `value` is TFLOPS with causal FLOPs counted as half.

`e2e` is the same metric through the public API for host tensors (attn_fwd_host): per
step, the copy of Q, K, V from pinned host memory to the GPU, the forward pass, and the
copy of O and LSE back into pinned host memory, all inside the timed region (the library
overlaps the copies of one chunk of heads with the kernels of the others).

`per_config` times every forward workload; `decode` times the decode workloads (one
query row per head against 8192 and 1,048,576 cached keys) and reports them against the
HBM roofline (K and V are read once); `backward` times the backward pass (attn_bwd) of
caseC and caseD.  `--backward NAME` times one backward alone (for profiler runs).

`cpu_baseline` (rank 0, N=1 only) times the float64 CPU oracle (test infrastructure) on
the same workload on the host cores; `--impl reference` times that oracle as the
reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS (causal-halved) and % of GB300 FP16 tensor peak; µs/call"
L2_BYTES = 126.5 * 2 ** 20
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


# The sources each kernel family is built from (its own files, the shared PTX helpers, and
# the C ABI, whose launch plan decides how the kernel runs).
KERNEL_SOURCES = {
    "fwd": ("attn_fwd_d", "attn_fwd_pp_d", "attn_fwd_kernel.cuh", "attn_fwd_pp.cuh", "softmax_tile.cuh"),
    "decode": ("attn_decode", "attn_fwd_kernel.cuh"),
    "bwd": ("attn_bwd.cu", "attn_bwd.cuh", "attn_fwd_kernel.cuh"),
}
SHARED_SOURCES = ("ptx.cuh", "tmem_ldst.inc", "gbattn_abi.cu")


def _code_only(text: str) -> str:
    """C++ source without its comments and blank lines (comment edits leave a kernel's
    compiled code, and so its stored ncu capture, unchanged)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kind: str = "fwd") -> str:
    """Hash of the code (comments left out) of the sources a kernel family (fwd, decode,
    bwd) is built from, to tell whether a stored ncu capture still describes the current
    kernel."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "scaled_dot_product_sdpa_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith(KERNEL_SOURCES[kind]) or name in SHARED_SOURCES:
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode())
                h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def kernel_name(w, sm_count: int) -> str:
    """The kernel attn_fwd runs for workload w on a GPU with sm_count SMs (the library's
    own launch plan)."""
    import scaled_dot_product_sdpa_gb300 as gb
    kind = gb.attn_debug_plan(w.B, w.H, w.L, w.d, w.causal, sm_count)["kind"]
    return "attn_fwd_pp_kernel" if kind == 1 else "attn_fwd_kernel"


def stored_traffic(workload: str, kernel: str):
    """dram read+write bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling (read-only queries, every 100 ms).  stop() keeps
    only the samples whose timestamps fall inside a given host-clock window."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    @staticmethod
    def _epoch(stamp: str):
        """nvidia-smi's local-time stamp 'YYYY/MM/DD HH:MM:SS.mmm' as epoch seconds."""
        import datetime
        try:
            return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self, window=None):
        """Stop sampling; with window = (t0, t1) (time.time() values) keep only the samples
        taken inside it (a margin of half the sampling period on each side)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        os.unlink(self.path)
        if window is not None:
            t0, t1 = window
            rows = [r for r in rows if (e := self._epoch(r[0])) is not None and t0 - 0.05 <= e <= t1 + 0.05]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_config(w, world: int) -> dict:
    """The `config` of the JSON line, identical in both arms: the workload, and how the
    GPU arm keeps every step's inputs out of L2."""
    R = n_rotating_sets(w)
    return {"workload": w.name, "shape": w.describe(), "global_batch": w.B * world, "seq_len": w.L,
            "head_dim": w.d, "heads": w.H, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": f"GPU arm: {R} rotating input/output sets ({R * w.bytes() / 2**20:.0f} MiB > 2x L2); no flush",
            "timing": "GPU arm: CUDA graph of the steps, CUDA events on the replay stream; reference arm: "
                      "host wall clock"}


# ----------------------------------------------------------------------------- ours
def capture_graph(fn_list, stream, torch):
    """Capture the launches in fn_list, in order, into one CUDA graph on `stream`."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for fn in fn_list:
            fn(stream)
    torch.cuda.synchronize()
    return g


def make_sets(w, n_sets, device, torch, inputs):
    q, k, v = inputs.qkv(w.B, w.H, w.L, w.d, w.seed, w.sigma)
    sets = []
    for _ in range(n_sets):
        dq, dk, dv = (t.to(device) for t in (q, k, v))
        o = torch.empty_like(dq)
        lse = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=device)
        sets.append((dq, dk, dv, o, lse))
    return (q, k, v), sets


def n_rotating_sets(w):
    per = w.bytes()
    return max(2, math.ceil(2.0 * L2_BYTES / per) + 1)


def bench_workload(w, steps, warmup, device, torch, gb, inputs, world):
    """Device time per forward call of workload w: exactly `steps` launches, replayed
    from CUDA graphs, cycling through R rotating input/output sets."""
    R = n_rotating_sets(w)
    host, sets = make_sets(w, R, device, torch, inputs)

    def launcher(s):
        return lambda st: gb.attn_fwd(s[0], s[1], s[2], causal=w.causal, scale=w.scale, o=s[3], lse=s[4],
                                      stream=st)

    per = R * max(1, math.ceil(64 / R))  # launches per main graph, a multiple of R
    stream = torch.cuda.Stream(device=device)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # first calls (attributes, descriptors) outside capture
        for i in range(R):
            launcher(sets[i])(stream)
    torch.cuda.synchronize()
    main = capture_graph([launcher(sets[i % R]) for i in range(per)], stream, torch)
    n_main, n_tail = divmod(steps, per)
    tail = capture_graph([launcher(sets[i % R]) for i in range(n_tail)], stream, torch) if n_tail else None
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(warmup / per))):
            main.replay()
        if tail is not None:  # its first replay also uploads the graph: keep that untimed
            tail.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    h0 = time.time()
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(n_main):
            main.replay()
        if tail is not None:
            tail.replay()
        b.record(stream)
    b.synchronize()
    h1 = time.time()
    torch.cuda.synchronize()
    barrier(world)
    t = a.elapsed_time(b) * 1e-3 / steps
    return t, steps, R, host, sets, (main, stream, per, (h0, h1))


def bench_e2e(w, steps, warmup, device, torch, gb, host):
    """Through the public API for host tensors (attn_fwd_host): per step, Q, K, V go from
    pinned host memory to the GPU, the forward pass runs, O and LSE come back to pinned
    host memory -- chunked so that the copies overlap the kernels -- all inside the timed
    region."""
    q, k, v = (t.pin_memory() for t in host)
    o_h = torch.empty(q.shape, dtype=torch.float16).pin_memory()
    l_h = torch.empty((w.B, w.H, w.L), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()

    def step():
        gb.attn_fwd_host(q, k, v, causal=w.causal, scale=w.scale, o=o_h, lse=l_h, device=device, stream=stream)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    n = max(3, min(steps, 200))
    t0 = time.perf_counter()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        step()
    b.record(stream)
    b.synchronize()
    wall = time.perf_counter() - t0
    dev = a.elapsed_time(b) * 1e-3
    t = max(wall, dev) / n
    h2d = 3 * q.numel() * 2
    d2h = o_h.numel() * 2 + l_h.numel() * 4
    return t, h2d, d2h


def interleaved_per_call(workloads, reps, device, torch, gb, inputs):
    """Device time of single calls, `reps` rounds interleaved across the workloads (each
    round calls every workload once, on its next rotating input set, so inputs come
    from HBM).  A GPU-side sleep before each timed call keeps the stream busy while the
    host enqueues the call, so the events bracket the kernel and not the host's launch
    work.  Two brackets with the same sleep are timed alongside: nothing between the
    events ("events", what the bracket itself adds) and a torch kernel on one element
    ("launch", what any kernel launch adds on top).  Returns {name: (median, p10, p90,
    mean of the middle 80%) seconds}, the two brackets under the names "_events" and
    "_launch"."""
    prepared = {}
    for name, w in workloads.items():
        R = n_rotating_sets(w)
        _, sets = make_sets(w, R, device, torch, inputs)
        prepared[name] = (w, sets)
    stream = torch.cuda.current_stream()
    for name, (w, sets) in prepared.items():  # first calls (descriptors, plans) untimed
        s = sets[0]
        gb.attn_fwd(s[0], s[1], s[2], causal=w.causal, scale=w.scale, o=s[3], lse=s[4], stream=stream)
    torch.cuda.synchronize()
    events = {name: [] for name in list(prepared) + ["_events", "_launch"]}
    one = torch.zeros(1, device=device)
    one.add_(1.0)  # its kernel loaded before anything is timed
    torch.cuda.synchronize()
    for r in range(reps):
        for name in ("_events", "_launch"):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(200000)
            a.record(stream)
            if name == "_launch":
                one.add_(1.0)
            b.record(stream)
            events[name].append((a, b))
        for name, (w, sets) in prepared.items():
            s = sets[r % len(sets)]
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(200000)
            a.record(stream)
            gb.attn_fwd(s[0], s[1], s[2], causal=w.causal, scale=w.scale, o=s[3], lse=s[4], stream=stream)
            b.record(stream)
            events[name].append((a, b))
        if r % 50 == 49:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    out = {}
    for name, ev in events.items():
        ts = sorted(a.elapsed_time(b) * 1e-3 for a, b in ev)
        n = len(ts)
        mid = ts[n // 10:n - n // 10] or ts  # mean of the middle 80%: rare stalls left out
        out[name] = (ts[n // 2], ts[max(0, n // 10)], ts[min(n - 1, (9 * n) // 10)], sum(mid) / len(mid))
    del prepared
    return out


def bench_decode(device, torch, gb, inputs, hbm_peak, only=None):
    """Decode workloads (one query row per head against a long key/value sequence): mean
    time per call over 30 graph-replayed calls, CUDA events on the replay stream; K and V
    (1.1 and 4.3 GB) are far larger than L2, so every call reads them from HBM."""
    from scaled_dot_product_sdpa_gb300.configs import DECODE_WORKLOADS
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    out = {}
    for name, w in DECODE_WORKLOADS.items():
        if only is not None and name != only:
            continue
        q, k, v = inputs.decode_qkv(w.B, w.H, w.L, w.d, w.seed, w.sigma, device=device, draw_on_device=True)
        o = torch.empty(w.B, w.H, w.d, dtype=torch.float16, device=device)
        lse = torch.empty(w.B, w.H, dtype=torch.float32, device=device)
        stream = torch.cuda.Stream(device)
        with torch.cuda.stream(stream):
            for _ in range(3):
                gb.attn_decode(q, k, v, scale=w.scale, o=o, lse=lse, stream=stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for _ in range(10):
                    gb.attn_decode(q, k, v, scale=w.scale, o=o, lse=lse, stream=stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            g.replay()
            stream.synchronize()
            a.record(stream)
            for _ in range(3):
                g.replay()
            b.record(stream)
        b.synchronize()
        t = a.elapsed_time(b) * 1e-3 / 30
        plan = gb.attn_debug_decode_plan(w.B, w.H, w.L, w.d, sm_count, grouped=True)
        gbs = w.bytes() / t / 1e9
        out[name] = {"shape": w.describe(),
                     "kernels": ["attn_decode_kernel"] + (["attn_decode_merge_kernel"] if plan["groups"] > 1 else []),
                     "us": round(t * 1e6, 2), "hbm_gbs": round(gbs, 1), "pct_hbm_peak": round(100 * gbs / hbm_peak, 2),
                     "tflops": round(w.flops() / t / 1e12, 2), "ctas_per_cluster": plan["ranks"],
                     "clusters_per_head": plan["groups"], "keys_per_cta": plan["keys_per_rank"]}
        del q, k, v, g
        torch.cuda.empty_cache()
    return out


def bench_backward(device, torch, gb, inputs, tensor_peak, names=("caseC", "caseD")):
    """The backward pass (attn_bwd) of forward workloads: mean time per call over 30
    graph-replayed calls, CUDA events on the replay stream.  FLOPs are the usual 2.5x the
    forward's (five products of 2*L^2*d per head, halved when causal); the kernels execute
    seven such products."""
    from scaled_dot_product_sdpa_gb300.configs import WORKLOADS
    out = {}
    for name in names:
        w = WORKLOADS[name]
        q, k, v = (t.to(device) for t in inputs.qkv(w.B, w.H, w.L, w.d, w.seed, w.sigma))
        do = inputs.upstream_grad(w.B, w.H, w.L, w.d, w.seed + 100, device=device)
        o, lse = gb.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
        grads = [torch.empty_like(q) for _ in range(3)]
        stream = torch.cuda.Stream(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(3):
                gb.attn_bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, dq=grads[0], dk=grads[1],
                            dv=grads[2], stream=stream)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(10):
                    gb.attn_bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, dq=grads[0], dk=grads[1],
                                dv=grads[2], stream=stream)
            g.replay()
            stream.synchronize()
            a.record(stream)
            for _ in range(3):
                g.replay()
            b.record(stream)
        b.synchronize()
        t = a.elapsed_time(b) * 1e-3 / 30
        fl = 2.5 * w.flops()
        out[name] = {"shape": w.describe(), "kernels": ["attn_bwd_dkdv_kernel", "attn_bwd_dq_kernel"],
                     "us": round(t * 1e6, 2), "tflops": round(fl / t / 1e12, 1),
                     "pct_fp16_peak": round(100 * fl / t / 1e12 / tensor_peak, 2)}
        del g
    return out


def decode_only(name):
    """`--decode NAME`: the decode timing of one workload alone, as a JSON line."""
    import torch
    import scaled_dot_product_sdpa_gb300 as gb
    from scaled_dot_product_sdpa_gb300 import build as gbuild
    from scaled_dot_product_sdpa_gb300 import inputs
    from scaled_dot_product_sdpa_gb300.configs import DECODE_WORKLOADS
    if name not in DECODE_WORKLOADS:
        raise SystemExit(f"unknown decode workload {name!r}; known: {sorted(DECODE_WORKLOADS)}")
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    gb.load_library(gbuild.build())
    peaks, _ = load_peaks()
    res = bench_decode(device, torch, gb, inputs, peaks["hbm_gbs"], only=name)
    status = gb.attn_last_device_error()
    if status != 0:
        raise RuntimeError(f"device status {status}: {gb.attn_strerror(status)}")
    print(json.dumps({"decode": res}), flush=True)


def backward_only(name):
    """`--backward NAME`: the backward timing of one forward workload alone, as a JSON line."""
    import torch
    import scaled_dot_product_sdpa_gb300 as gb
    from scaled_dot_product_sdpa_gb300 import build as gbuild
    from scaled_dot_product_sdpa_gb300 import inputs
    from scaled_dot_product_sdpa_gb300.configs import WORKLOADS
    if name not in WORKLOADS or WORKLOADS[name].d > 128:
        raise SystemExit(f"no backward for {name!r} (head_dim 64 or 128 workloads: "
                         f"{sorted(n for n, w in WORKLOADS.items() if w.d <= 128)})")
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    gb.load_library(gbuild.build())
    peaks, _ = load_peaks()
    res = bench_backward(device, torch, gb, inputs, peaks["bf16_tflops"], names=(name,))
    status = gb.attn_last_device_error()
    if status != 0:
        raise RuntimeError(f"device status {status}: {gb.attn_strerror(status)}")
    print(json.dumps({"backward": res}), flush=True)


def matmul_tflops(torch, dtype, n=8192, reps=10):
    """Best of `reps` torch.matmul n x n x n products of `dtype` (2 n^3 FLOPs each), CUDA
    events: the library GEMM rate in this run, for the fp16/bf16 ratio of the tensor peak."""
    a = torch.randn(n, n, device="cuda", dtype=dtype)
    b = torch.randn(n, n, device="cuda", dtype=dtype)
    for _ in range(3):
        torch.matmul(a, b)
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b)
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e-3)
    del a, b
    torch.cuda.empty_cache()
    return 2.0 * n ** 3 / best / 1e12


def cpu_oracle_baseline(w, min_seconds=10.0, max_reps=20):
    """Float64 oracle, as it stands, on the host cores: whole workload, repeated until
    about `min_seconds` of CPU work (bounded by max_reps)."""
    import oracle
    from scaled_dot_product_sdpa_gb300 import inputs
    q, k, v = inputs.qkv(w.B, w.H, w.L, w.d, w.seed, w.sigma)
    scale = float(__import__("numpy").float32(w.scale))
    qf, kf, vf = (oracle._f64(t) for t in (q, k, v))
    reps, total, cores = 0, 0.0, 0
    while reps < max_reps and (total < min_seconds or reps == 0):
        t0 = time.perf_counter()
        o, lse = oracle.sdpa_fwd(qf, kf, vf, w.causal, scale)
        total += time.perf_counter() - t0
        reps += 1
    nthreads = int(os.environ.get("OMP_NUM_THREADS", "0")) or len(os.sched_getaffinity(0))
    t = total / reps
    return t, reps, nthreads


def oracle_one_thread(w, reps=5):
    """Seconds per call of the float64 oracle on one host thread for workload w."""
    import oracle
    from scaled_dot_product_sdpa_gb300 import inputs
    q, k, v = inputs.qkv(w.B, w.H, w.L, w.d, w.seed, w.sigma)
    qf, kf, vf = (oracle._f64(t) for t in (q, k, v))
    scale = float(__import__("numpy").float32(w.scale))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.sdpa_fwd(qf, kf, vf, w.causal, scale, nthreads=1)
    return (time.perf_counter() - t0) / reps


def bench_ours(args):
    import torch
    import scaled_dot_product_sdpa_gb300 as gb
    from scaled_dot_product_sdpa_gb300 import inputs
    from scaled_dot_product_sdpa_gb300.configs import WORKLOADS
    from scaled_dot_product_sdpa_gb300 import build as gbuild

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    gb.load_library(gbuild.build())
    peaks, peak_kind = load_peaks()
    from scaled_dot_product_sdpa_gb300.configs import EXTRA_WORKLOADS
    w = WORKLOADS[args.workload] if args.workload in WORKLOADS else EXTRA_WORKLOADS[args.workload]

    sampler = ClockSampler(local) if not args.quick else None
    if sampler:
        sampler.start()
    t, nsteps, R, host, sets, graph = bench_workload(w, args.steps, args.warmup, device, torch, gb, inputs, world)
    g_main, g_stream, per_graph, window = graph
    if sampler:
        # Only the samples taken inside the timed region count.
        clocks = sampler.stop(window)
        span_ms = (window[1] - window[0]) * 1e3
        clock_note = f"samples taken inside the timed region ({span_ms:.1f} ms)"
        if clocks.get("samples", 0) < 3:
            # The timed region is shorter than three sampling periods: sample over ~1.5 s
            # of the same graph replays right after it (untimed) and say so.
            sampler.start()
            h0 = time.time()
            with torch.cuda.stream(g_stream):
                t_end = time.perf_counter() + 1.5
                while time.perf_counter() < t_end:
                    for _ in range(20):
                        g_main.replay()
                    torch.cuda.synchronize()
            clocks = sampler.stop((h0, time.time()))
            clock_note = (f"timed region {span_ms:.1f} ms, shorter than three 100 ms sampling periods; sampled "
                          "over 1.5 s of the same graph replays right after it")
        clocks["note"] = clock_note
    else:
        clocks = None
    status = gb.attn_last_device_error()
    if status != 0:
        raise RuntimeError(f"device status {status}: {gb.attn_strerror(status)}")
    t_max = max_over_ranks(t, world, device)
    tflops = w.flops() / t_max / 1e12 * world
    fp16_peak = peaks["bf16_tflops"] * 1.0  # fp16 dense = bf16 dense (nominal ratio 1)
    hbm_peak = peaks["hbm_gbs"]
    achieved_gbs = w.bytes() / t_max / 1e9
    bound = "hbm" if w.flops() / w.bytes() < fp16_peak * 1e12 / (hbm_peak * 1e9) else "tensor"
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    kname = kernel_name(w, sm_count)
    traffic = stored_traffic(w.name, kname)
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved_gbs / hbm_peak, 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(w.flops() / t_max / 1e12, 1), "peak": fp16_peak,
                "unit": "TFLOP/s", "frac": round(w.flops() / t_max / 1e12 / fp16_peak, 4)}
    roof["traffic"] = traffic
    roof["kernel"] = kname
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback"
    roof["algorithmic_bytes_per_launch"] = w.bytes()
    roof["algorithmic_flops_per_launch"] = w.flops()
    roof["tensor_frac"] = round(w.flops() / t_max / 1e12 / fp16_peak, 4)
    roof["hbm_frac"] = round(achieved_gbs / hbm_peak, 4)

    line = {
        "metric": METRIC, "value": round(tflops, 2), "unit": "TFLOPS", "n_gpus": world, "steps": nsteps,
        "warmup": args.warmup, "ms_per_step": round(t_max * 1e3, 6), "us_per_call": round(t_max * 1e6, 3),
        "pct_fp16_peak": round(100 * w.flops() / t_max / 1e12 / fp16_peak, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "accumulate": "f32", "data": "synthetic",
        "config": workload_config(w, world),
        "gpu_launches": nsteps, "roofline": roof, "clocks": clocks,
    }
    if not args.quick:
        te, h2d, d2h = bench_e2e(w, args.steps, args.warmup, device, torch, gb, host)
        te = max_over_ranks(te, world, device)
        line["e2e"] = {"value": round(w.flops() / te / 1e12 * world, 3), "unit": "TFLOPS",
                       "us_per_call": round(te * 1e6, 2), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        per = {}
        for name, wk in WORKLOADS.items():
            tk = bench_workload(wk, 200, 10, device, torch, gb, inputs, world)[0]
            fl = wk.flops() / tk / 1e12
            # Attainable: the lower of the tensor roof and (FLOP/byte) x the HBM roof.
            attain = min(fp16_peak, wk.flops() / wk.bytes() * hbm_peak * 1e9 / 1e12)
            per[name] = {"shape": wk.describe(), "kernel": kernel_name(wk, sm_count), "us": round(tk * 1e6, 3),
                         "tflops": round(fl, 1), "pct_fp16_peak": round(100 * fl / fp16_peak, 2),
                         "hbm_gbs": round(wk.bytes() / tk / 1e9, 1),
                         "pct_hbm_peak": round(100 * wk.bytes() / tk / 1e9 / hbm_peak, 2),
                         "attainable_tflops": round(attain, 1), "pct_attainable": round(100 * fl / attain, 2)}
        # Per-call distribution, interleaved across the configs (300 rounds).
        dist_t = interleaved_per_call(WORKLOADS, 300, device, torch, gb, inputs)
        ev_floor = dist_t.pop("_events")
        launch_floor = dist_t.pop("_launch")
        for name, (med, p10, p90, mean) in dist_t.items():
            per[name].update({"per_call_us_median": round(med * 1e6, 3), "per_call_us_p10": round(p10 * 1e6, 3),
                              "per_call_us_p90": round(p90 * 1e6, 3), "per_call_us_mean": round(mean * 1e6, 3),
                              "per_call_us_mean_net_of_events": round((mean - ev_floor[3]) * 1e6, 3)})
        line["per_config"] = per
        line["per_call_floor_us"] = {"events_only": {"median": round(ev_floor[0] * 1e6, 3),
                                                     "mean": round(ev_floor[3] * 1e6, 3)},
                                     "one_element_kernel": {"median": round(launch_floor[0] * 1e6, 3),
                                                           "mean": round(launch_floor[3] * 1e6, 3)}}
        line["per_config_timing"] = ("us: mean of 200 graph-replayed calls over rotating input sets; "
                                     "per_call_*: 300 single calls interleaved across the configs, CUDA events "
                                     "around each call behind a GPU-side sleep; per_call_floor_us: the same "
                                     "bracket around nothing and around a torch kernel on one element; the event "
                                     "timestamps come in steps of up to ~2 us, so medians are coarse and "
                                     "the net figure uses means (of the middle 80% of the calls)")
        # fp16 and bf16 library GEMMs in this run: the roofline's peak is the measured bf16
        # figure of MEASURED_PEAKS.json, taken for fp16 at the nominal ratio of 1; this
        # records the measured ratio beside it.
        f16 = matmul_tflops(torch, torch.float16)
        b16 = matmul_tflops(torch, torch.bfloat16)
        roof["matmul_8192_tflops_this_run"] = {"fp16": round(f16, 1), "bf16": round(b16, 1),
                                               "fp16_over_bf16": round(f16 / b16, 4)}
        line["decode"] = bench_decode(device, torch, gb, inputs, hbm_peak)
        line["backward"] = bench_backward(device, torch, gb, inputs, fp16_peak)
        status = gb.attn_last_device_error()
        if status != 0:
            raise RuntimeError(f"device status {status}: {gb.attn_strerror(status)}")
        if rank == 0 and world == 1 and not args.no_cpu:
            tc, reps, cores = cpu_oracle_baseline(w)
            line["cpu_baseline"] = {"value": round(w.flops() / tc / 1e12, 6), "unit": "TFLOPS", "cores": cores,
                                    "kind": "oracle", "seconds_per_call": round(tc, 3),
                                    "sample": f"the whole {w.name} workload, {reps} call(s), float64 C oracle"}
            # The smallest config on one thread as well (the same oracle, nthreads = 1).
            t1 = oracle_one_thread(WORKLOADS["caseA"])
            line["cpu_baseline"]["caseA_one_thread_seconds"] = round(t1, 4)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference
def bench_reference(args):
    """The reference arm: the float64 CPU oracle, as it stands, on the host cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from scaled_dot_product_sdpa_gb300.configs import WORKLOADS
    import oracle
    import numpy as np
    from scaled_dot_product_sdpa_gb300 import inputs
    oracle.build()
    w = WORKLOADS[args.workload]
    q, k, v = inputs.qkv(w.B, w.H, w.L, w.d, w.seed, w.sigma)
    qf, kf, vf = (oracle._f64(t) for t in (q, k, v))
    # Bounded sample: a slice of the heads sized so that one step is ~1-2 s of CPU work.
    heads = w.B * w.H
    probe_heads = max(1, heads // 64)
    t0 = time.perf_counter()
    oracle.sdpa_fwd(qf.reshape(heads, 1, w.L, w.d)[:probe_heads], kf.reshape(heads, 1, w.L, w.d)[:probe_heads],
                    vf.reshape(heads, 1, w.L, w.d)[:probe_heads], w.causal, float(np.float32(w.scale)))
    per_head = (time.perf_counter() - t0) / probe_heads
    step_budget = min(1.5, 90.0 / (args.steps + args.warmup))  # whole run ~1.5 min at most
    nh = int(min(heads, max(1, step_budget / max(per_head, 1e-9))))
    sl = lambda x: np.ascontiguousarray(x.reshape(heads, 1, w.L, w.d)[:nh])
    qs, ks, vs = sl(qf), sl(kf), sl(vf)
    for _ in range(args.warmup):
        oracle.sdpa_fwd(qs, ks, vs, w.causal, float(np.float32(w.scale)))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.sdpa_fwd(qs, ks, vs, w.causal, float(np.float32(w.scale)))
    dt = (time.perf_counter() - t0) / args.steps
    flops = w.flops() * nh / heads
    value = flops / dt / 1e12
    cores = int(os.environ.get("OMP_NUM_THREADS", "0")) or len(os.sched_getaffinity(0))
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOPS", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, world),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                             "sample": f"{nh} of {heads} heads of {w.name} per step"},
            "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="caseD")
    ap.add_argument("--quick", action="store_true", help="timed region only (for profiler runs)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--decode", metavar="NAME", help="time only this decode workload (diagnostic; for profiler runs)")
    ap.add_argument("--backward", metavar="NAME", help="time only the backward pass of this workload (diagnostic)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.decode:
        decode_only(args.decode)
    elif args.backward:
        backward_only(args.backward)
    elif args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
