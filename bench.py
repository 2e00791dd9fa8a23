#!/usr/bin/env python3
"""Benchmark of the fused SGMV LoRA apply (lora_apply) on one or more GB300s.

One step = one lora_apply call: one batch of tokens through one LoRA layer (fused shrink +
expand over every segment).  Default workload: decode_distinct -- Llama-7B projection
h_in=h_out=4096, r=16, fp16, 64 tokens, each its own length-1 segment and its own adapter of a
64-adapter pool stacked over 32 layers; the steps sweep layer_idx 0..31 and rotate 32 x/y buffer
sets, so every step reads inputs that are not in L2 (the sweep touches ~0.55 GB > 129 MB L2).

Prints one JSON line (rank 0):
  value      achieved algorithmic HBM GB/s (bytes: each distinct adapter's A and B once, x
             once, y read + written), whole job, inputs resident in HBM, CUDA-graph replay,
             CUDA events on the launching stream;
  e2e        the same metric through the public API with pinned HOST buffers: every step copies
             its x, y_in and segment table host->device and reads y back;
  roofline   achieved / measured HBM copy bandwidth of the GB300s;
  cpu_baseline  the fp64 oracle (single thread) on a bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from segmented_gather_gemm_sgmv_gb300 import workloads  # noqa: E402

METRIC = "SGMV shrink+expand achieved HBM GB/s & tokens/s at h=4096,r=16 (% roofline)"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ accounting ----
def algorithmic_bytes(w, ss, sa):
    """Distinct adapters' A and B once + x read once + y read and written once."""
    M, D = 0, set()
    for i, k in enumerate(sa):
        n = int(ss[i + 1]) - int(ss[i])
        if n > 0 and k >= 0:
            M += n
            D.add(int(k))
    eb = w.elem_bytes
    return len(D) * (w.h_in * w.r + w.r * w.h_out) * eb + M * w.h_in * eb + 2 * M * w.h_out * eb, M


def flops(w, M):
    return 2 * M * w.r * (w.h_in + w.h_out)


def source_hash():
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "segmented_gather_gemm_sgmv_gb300", "csrc", "*"))):
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload):
    """dram read+write bytes per launch from the committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("source_hash") != source_hash():
        return None
    return d.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_ms=50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 9]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                smax.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- distributed ----
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value, world, device=None):
    """Max of a float over ranks (identity at world size 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, nbytes_per_rank, per_step_s):
    """Whole-job GB/s: every rank moves nbytes_per_rank per step (weak scaling, replicas) and a
    job step lasts as long as the slowest rank's (per_step_s is the max over ranks)."""
    return world * nbytes_per_rank / per_step_s / 1e9


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- our arm ----
class Setup:
    """Device-resident inputs of the workload: pool, NB rotating x/y sets, segment table."""

    def __init__(self, w, device, nbuf=32, seed=0, overlap=True, tensor_cores="auto",
                 long_batch=False, strided=False):
        import torch
        self.w = w
        self.overlap = overlap
        self.tensor_cores = tensor_cores
        self.long_batch = long_batch
        self.ss, self.sa = workloads.make_segments(w.name, seed)
        self.M = int(self.ss[-1])
        self.A, self.B = workloads.make_pool(w, device, seed=seed + 1)
        self.A_ptrs = workloads.pointer_table(self.A, device)
        self.B_ptrs = workloads.pointer_table(self.B, device)
        self.d_ss = torch.as_tensor(self.ss, device=device)
        self.d_sa = torch.as_tensor(self.sa, device=device)
        self.nbuf = nbuf
        self.x, self.y = [], []
        self.strided = strided
        for i in range(nbuf):
            x, y = workloads.make_activations(w, self.M, device, seed=seed + 100 + i)
            if strided:  # the middle third of 3x-wide rows, as q / k / v of a fused output
                X = torch.zeros((self.M, 3 * w.h_in), dtype=x.dtype, device=device)
                Y = torch.zeros((self.M, 3 * w.h_out), dtype=y.dtype, device=device)
                X[:, w.h_in:2 * w.h_in] = x
                Y[:, w.h_out:2 * w.h_out] = y
                x, y = X[:, w.h_in:2 * w.h_in], Y[:, w.h_out:2 * w.h_out]
            self.x.append(x)
            self.y.append(y)

    def call(self, step, stream=None):
        from segmented_gather_gemm_sgmv_gb300 import lora_apply
        i = step % self.nbuf
        lora_apply(self.y[i], self.x[i], self.A_ptrs, self.B_ptrs, self.d_ss, self.d_sa,
                   step % self.w.layers, self.w.r, self.w.scale, stream=stream,
                   overlap_prior=self.overlap, tensor_cores=self.tensor_cores,
                   long_batch=self.long_batch)


def capture(torch, fn, n, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in range(n):
            fn(s)
    return g


def time_graph_steps(torch, setup, K, W, stream, world):
    """Device time of K steps (graph replays of one layer sweep), CUDA events on `stream`."""
    per = setup.w.layers * max(1, setup.nbuf // setup.w.layers)
    per = max(per, setup.nbuf)
    with torch.cuda.stream(stream):
        for s in range(per):  # uncaptured first calls set kernel attributes
            setup.call(s, stream)
    torch.cuda.synchronize()
    g_full = capture(torch, lambda s: setup.call(s, stream), per, stream)
    rem = K % per
    g_rem = capture(torch, lambda s: setup.call(s, stream), rem, stream) if rem else None
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        for _ in range(max(1, (W + per - 1) // per)):
            g_full.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(K // per):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1)


def time_e2e(torch, setup, K, stream):
    """Public-API path with pinned host buffers.  Per step: ONE host->device copy of the step's
    inputs (x, y_in and the segment table packed in one pinned staging buffer), the lora_apply
    call on views of the device copy, ONE device->host copy of y.  Steps alternate between two
    streams and two device / host buffer sets, so that one step's copies overlap the other
    stream's kernel; each stream runs its steps in order (a buffer set is reused only after
    its previous step's copy back has completed)."""
    w = setup.w
    n = min(K, 2048)
    dt = workloads.torch_dtype(w.dtype)
    x0, y0 = setup.x[0], setup.y[0]
    eb = x0.element_size()

    def up16(v):
        return (v + 15) // 16 * 16

    nx, ny = x0.numel() * eb, y0.numel() * eb
    nss, nsa = 4 * len(setup.ss), 4 * len(setup.sa)
    off_y = up16(nx)
    off_ss = off_y + up16(ny)
    off_sa = off_ss + up16(nss)
    total = off_sa + up16(nsa)
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    host[0:nx].copy_(x0.cpu().contiguous().view(torch.uint8).view(-1))
    host[off_y:off_y + ny].copy_(y0.cpu().contiguous().view(torch.uint8).view(-1))
    host[off_ss:off_ss + nss].copy_(torch.as_tensor(setup.ss).view(torch.uint8))
    host[off_sa:off_sa + nsa].copy_(torch.as_tensor(setup.sa).view(torch.uint8))
    streams = [stream, torch.cuda.Stream(x0.device)]
    sets = []
    for _ in range(2):
        dev = torch.empty(total, dtype=torch.uint8, device=x0.device)
        sets.append(dict(dev=dev, x=dev[0:nx].view(dt).view(x0.shape),
                         y=dev[off_y:off_y + ny].view(dt).view(y0.shape),
                         ss=dev[off_ss:off_ss + nss].view(torch.int32),
                         sa=dev[off_sa:off_sa + nsa].view(torch.int32),
                         out=torch.empty(y0.shape, dtype=dt).pin_memory()))
    from segmented_gather_gemm_sgmv_gb300 import lora_apply

    def step(s):
        st, b = streams[s % 2], sets[s % 2]
        with torch.cuda.stream(st):
            b["dev"].copy_(host, non_blocking=True)
            lora_apply(b["y"], b["x"], setup.A_ptrs, setup.B_ptrs, b["ss"], b["sa"],
                       s % w.layers, w.r, w.scale, stream=st, overlap_prior=setup.overlap,
                       tensor_cores=setup.tensor_cores, long_batch=setup.long_batch)
            b["out"].copy_(b["y"], non_blocking=True)

    def sweep(n_steps):
        streams[1].wait_stream(streams[0])  # fork
        for s in range(n_steps):
            step(s)
        streams[0].wait_stream(streams[1])  # join

    per = w.layers if w.layers % 2 == 0 else 2 * w.layers
    with torch.cuda.stream(stream):
        sweep(4)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sweep(per)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    reps = max(1, n // per)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return ms / (reps * per), total, ny, reps * per


def cpu_baseline(w, setup, seconds=10.0):
    """The fp64 oracle, single-threaded, on the full batch at layer 0, repeated for ~seconds."""
    import oracle
    keys = sorted({int(k) for i, k in enumerate(setup.sa)
                   if k >= 0 and setup.ss[i + 1] > setup.ss[i]})
    A = [None] * setup.A.shape[0]
    B = [None] * setup.B.shape[0]
    for k in keys:
        A[k] = setup.A[k, 0:1].double().cpu().numpy()
        B[k] = setup.B[k, 0:1].double().cpu().numpy()
    call = oracle.PreparedApply(setup.y[0].double().cpu().numpy(),
                                setup.x[0].double().cpu().numpy(), A, B, setup.ss, setup.sa, 0,
                                w.scale)
    n, t0 = 0, time.perf_counter()
    while True:
        call()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    nbytes, M = algorithmic_bytes(w, setup.ss, setup.sa)
    per = el / n
    return {"value": round(nbytes / per / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"oracle_lora_apply (fp64, 1 thread) on the whole {w.name} batch "
                      f"({M} tokens, layer 0), {n} calls in {el:.1f} s",
            "tokens_per_s": round(M / per, 2), "us_per_call": round(per * 1e6, 1)}


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from segmented_gather_gemm_sgmv_gb300 import binding
    binding.lib()
    w = workloads.WORKLOADS[args.workload]
    long_batch = {"auto": w.prefill, "on": True, "off": False}[args.long_batch]
    setup = Setup(w, device, tensor_cores=args.tensor_cores, long_batch=long_batch,
                  strided=args.strided)
    stream = torch.cuda.Stream(device)
    nbytes, M = algorithmic_bytes(w, setup.ss, setup.sa)
    K, W = args.steps, args.warmup

    # isolated calls (each kernel waits for the previous one to finish): context figure
    setup.overlap = False
    ms_iso = time_graph_steps(torch, setup, min(K, 6400), W, stream, world)
    us_iso = ms_iso * 1e3 / min(K, 6400)
    setup.overlap = not args.no_overlap
    clocks = ClockSampler(torch.cuda.current_device()).start()
    time.sleep(0.3)
    ms = time_graph_steps(torch, setup, K, W, stream, world)
    clk = clocks.stop()
    ms = reduce_max(ms, world, device)
    if binding.sgmv_get_error(clear=True) != 0:
        raise RuntimeError("a device-side wait ran out during the timed region")
    per = ms / 1e3 / K
    e2e_s, h2d, d2h, e2e_n = time_e2e(torch, setup, K, stream)
    e2e_s = reduce_max(e2e_s, world, device) / 1e3
    if rank != 0:
        dist_finish(world)
        return
    hbm, peak_kind = measured_peaks()
    achieved = nbytes / per / 1e9
    line = {
        "metric": METRIC,
        "value": round(job_value(world, nbytes, per), 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(per * 1e3, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "impl": "ours",
        "tokens_per_s": round(world * M / per, 1),
        "us_per_call": round(per * 1e6, 3),
        "us_per_call_isolated": round(us_iso, 3),
        "launch": ("lora_apply_ex(SGMV_OVERLAP_PRIOR): each call's weight prefetch overlaps the "
                   "previous call (programmatic dependent launch)" if setup.overlap else
                   "lora_apply: each call starts after the previous one completes") +
                  ("; SGMV_LONG_BATCH (a prefill batch: one CTA per SM, whole shared memory)"
                   if setup.long_batch else ""),
        "config": {"workload": w.name, "h_in": w.h_in, "h_out": w.h_out, "r": w.r,
                   "tokens": M, "segments": int(len(setup.sa)),
                   "distinct_adapters": int(len({int(k) for k in setup.sa})),
                   "pool_adapters": w.num_adapters, "layers": w.layers,
                   "bytes_per_call": nbytes, "flops_per_call": flops(w, M),
                   "timing": "CUDA graph of one 32-layer sweep replayed; CUDA events on the "
                             "launching stream",
                   "l2": "inputs larger than L2: each step reads another layer's weights and "
                         "another x/y set (sweep footprint > 129 MB)",
                   "layout": ("x, y: middle column third of rows 3 h apart (lora_apply_strided)"
                              if setup.strided else "x [M][h_in], y [M][h_out] dense"),
                   "parallelism": f"replica x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": None if setup.strided else recorded_traffic(w.name),
                     "peak_source": peak_kind,
                     "kernel": "sgmv_kernel<fused> (lora_apply)"},
        "e2e": {"value": round(job_value(world, nbytes, e2e_s), 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_n, "us_per_step": round(e2e_s * 1e6, 3)},
        "gpu_launches": K,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, setup, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    dist_finish(world)


def dist_finish(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------ reference arm ----
def run_reference(args):
    """The fp64 oracle timed on the host cores, on this arm's workload: each step is one token
    of the batch (a length-1 segment with its adapter, layer 0), cycling over the batch."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = workloads.WORKLOADS[args.workload]
    ss, sa = workloads.make_segments(w.name, 0)
    rng = np.random.default_rng(0)
    keys = sorted({int(k) for i, k in enumerate(sa) if k >= 0 and ss[i + 1] > ss[i]})
    A = [None] * w.num_adapters
    B = [None] * w.num_adapters
    for k in keys:
        A[k] = rng.uniform(-1, 1, (1, w.h_in, w.r)) / np.sqrt(w.h_in)
        B[k] = rng.standard_normal((1, w.r, w.h_out)) / np.sqrt(w.r)
    M = int(ss[-1])
    x = rng.standard_normal((M, w.h_in))
    y = rng.standard_normal((M, w.h_out))
    rows = [(int(ss[i]), int(k)) for i, k in enumerate(sa) if ss[i + 1] > ss[i] and k >= 0]
    calls = []
    for t, k in rows:
        calls.append(oracle.PreparedApply(y[t:t + 1], x[t:t + 1], A, B, [0, 1], [k], 0, w.scale))
    for s in range(args.warmup):
        calls[s % len(calls)]()
    t0 = time.perf_counter()
    for s in range(args.steps):
        calls[s % len(calls)]()
    el = time.perf_counter() - t0
    per = el / args.steps
    eb = w.elem_bytes
    nbytes = (w.h_in * w.r + w.r * w.h_out) * eb + w.h_in * eb + 2 * w.h_out * eb
    val = nbytes / per / 1e9
    line = {"metric": METRIC, "value": round(val, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "h_in": w.h_in, "h_out": w.h_out, "r": w.r,
                       "step": "one token of the batch (its own adapter, layer 0)"},
            "tokens_per_s": round(1.0 / per, 2),
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle",
                             "sample": f"{args.steps} single-token oracle_lora_apply calls "
                                       f"(fp64, 1 thread) cycling over the {w.name} batch"},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=1000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_distinct", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tensor-cores", choices=["auto", "never", "always"], default="auto",
                    help="which adapter groups use the tensor cores (lora_apply_ex flags)")
    ap.add_argument("--long-batch", choices=["auto", "on", "off"], default="auto",
                    help="SGMV_LONG_BATCH launches; auto: for workloads that hold prefill "
                         "segments (prefill_mixed, mixed_70b)")
    ap.add_argument("--strided", action="store_true",
                    help="x and y are the middle column third of 3x-wide activations "
                         "(lora_apply_strided; the e2e figure stays on dense copies)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="plain lora_apply launches (no programmatic dependent launch)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
