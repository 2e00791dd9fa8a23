#!/usr/bin/env python3
"""Benchmark of the fused SGMV LoRA apply (lora_apply) on one or more GB300s.

Step.  One step is one decode step's LoRA pass over every layer of the model for one
projection: a layer sweep of lora_apply calls (one launch each) on one batch.  Headline
workload: decode_distinct -- Llama-7B projection h_in=h_out=4096, r=16, fp16, 64 tokens, each
its own length-1 segment and its own adapter of a 64-adapter pool stacked over 32 layers; a
step is 32 calls (layer_idx 0..31), each on its own x / y buffer set, so every call reads
weights and activations that are not in L2 (the sweep touches ~0.6 GB > 129 MB of L2).  The
calls of a step are replayed from one CUDA graph and launched with SGMV_OVERLAP_PRIOR.

Prints one JSON line (rank 0):
  value         algorithmic HBM GB/s, whole job (bytes per call: each distinct adapter's A
                and B once, x once, y read + written once), inputs resident in HBM, CUDA events
                on the launching stream around exactly K steps;
  e2e           the same metric through the public API with pinned HOST buffers: every step
                copies all its calls' x and y_in and the segment table host->device (one copy)
                and reads every call's y back (one copy);
  roofline      achieved / measured HBM copy bandwidth (and the FLOP term beside it);
  per_config    every named workload (decode_distinct, decode_zipf, decode_uniform,
                decode_same, prefill_mixed, mixed_70b): us per call chained and isolated, the
                unfused shrink + expand pair, GB/s, tokens/s, roofline fraction, clocks;
  cpu_baseline  the fp64 oracle on all host cores (threads over disjoint segment ranges) on
                one call of the headline batch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

--gpus N without an external launcher re-launches this script through torch.distributed.run
with N local ranks (one replica per GPU: the batches are independent, no collective on the data
path; only the barriers and the max over ranks of the step time).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import dataclasses
import glob
import hashlib
import json
import math
import os
import socket
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
FALLBACK_BF16_TFLOPS = 1700.0  # sustained, the profiling recipe's fallback
# FP32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz (unit counts and the
# maximum SM clock).
FP32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
PER_CONFIG = ("decode_distinct", "decode_zipf", "decode_uniform", "decode_same", "prefill_mixed",
              "mixed_70b")


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


def group_rows(ss, sa):
    rows = {}
    for i, k in enumerate(sa):
        n = int(ss[i + 1]) - int(ss[i])
        if n > 0 and k >= 0:
            rows[int(k)] = rows.get(int(k), 0) + n
    return rows


def tensor_core_rows(w, ss, sa, tensor_cores="auto"):
    """Rows that the library's documented routing rule sends to the tensor cores (fp16 / bf16,
    r >= 16, adapter groups of >= 64 rows whose CUDA-core items would re-read >= 32 MB of
    weights; include/sgmv.h, lora_apply)."""
    if w.dtype == "f32" or w.r < 16 or tensor_cores == "never":
        return 0
    wbytes = w.r * 2 * (w.h_in + w.h_out)
    need = 64 if tensor_cores == "always" else max(64, 4 * math.ceil(32 * 1048576 / wbytes))
    return sum(n for n in group_rows(ss, sa).values() if n >= need)


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
        return (float(d["hbm_gbs"]), float(d.get("bf16_tflops_sustained", FALLBACK_BF16_TFLOPS)),
                "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


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


def roofline(w, ss, sa, us_per_call, tensor_cores="auto"):
    """max(bytes / HBM, FLOPs / peak): the tensor-core FLOPs against the measured sustained
    bf16 (= fp16) peak, the CUDA-core FLOPs against the FP32 peak; fraction = roofline time /
    measured time."""
    hbm, tc_peak, kind = measured_peaks()
    nbytes, M = algorithmic_bytes(w, ss, sa)
    m_tc = tensor_core_rows(w, ss, sa, tensor_cores)
    f_tc, f_cc = flops(w, m_tc), flops(w, M - m_tc)
    t_mem = nbytes / (hbm * 1e9)
    t_flop = f_tc / (tc_peak * 1e12) + f_cc / (FP32_TFLOPS * 1e12)
    per = us_per_call * 1e-6
    achieved = nbytes / per / 1e9
    bound = "hbm" if t_mem >= t_flop else ("tensor" if f_tc / tc_peak >= f_cc / FP32_TFLOPS
                                          else "alu")
    out = {"bound": bound, "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
           "frac": round(max(t_mem, t_flop) / per, 4), "peak_source": kind,
           "t_mem_us": round(t_mem * 1e6, 3), "t_flop_us": round(t_flop * 1e6, 3),
           "flop_peaks_tflops": {"tensor_bf16_sustained": tc_peak, "fp32_cuda_cores":
                                 round(FP32_TFLOPS, 1)},
           "flops_tensor": f_tc, "flops_cuda_cores": f_cc}
    if bound != "hbm":  # the FLOP term dominates: report against its peak
        out.update(achieved=round((f_tc + f_cc) / per / 1e12, 2), unit="TFLOP/s",
                   peak=tc_peak if bound == "tensor" else round(FP32_TFLOPS, 1))
    return out


# ---------------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while a timed region runs."""

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


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def relaunch_cmd(argv, n):
    """The torch.distributed.run command that runs this script with n local ranks."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={n}", "--master-addr=127.0.0.1",
            f"--master-port={_free_port()}", os.path.abspath(__file__)] + list(argv)


# ----------------------------------------------------------------- our arm ----
def dense_grid_rule(w, ss, sa):
    """The caller-side rule for SGMV_DENSE_GRID, as a serving layer that built the table would
    apply it: a decode batch (no prefill segments) of at least 128 rows spread over at least 32
    adapter groups, i.e. many work items for each SM (measured: decode_zipf and decode_uniform
    gain; a batch of one row per adapter, or one adapter for every row, loses)."""
    if w.prefill:
        return False
    groups = group_rows(ss, sa)
    return sum(groups.values()) >= 128 and len(groups) >= 32


def sweep_len(w):
    """Calls per step: every layer of the pool once (a single-layer pool: 20 repeats)."""
    return w.layers if w.layers > 1 else 20


class Setup:
    """Device-resident inputs of the workload: pool, one x/y set per call of a step, table."""

    def __init__(self, w, device, seed=0, overlap=True, tensor_cores="auto", long_batch=False,
                 strided=False, dense_grid=False):
        import torch
        self.w = w
        self.overlap = overlap
        self.tensor_cores = tensor_cores
        self.long_batch = long_batch
        self.dense_grid = dense_grid
        self.ss, self.sa = workloads.make_segments(w.name, seed)
        self.M = int(self.ss[-1])
        self.A, self.B = workloads.make_pool(w, device, seed=seed + 1)
        self.A_ptrs = workloads.pointer_table(self.A, device)
        self.B_ptrs = workloads.pointer_table(self.B, device)
        self.d_ss = torch.as_tensor(self.ss, device=device)
        self.d_sa = torch.as_tensor(self.sa, device=device)
        self.calls = sweep_len(w)
        self.x, self.y = [], []
        self.strided = strided
        for i in range(self.calls):
            x, y = workloads.make_activations(w, self.M, device, seed=seed + 100 + i)
            if strided:  # the middle third of 3x-wide rows, as q / k / v of a fused output
                X = torch.zeros((self.M, 3 * w.h_in), dtype=x.dtype, device=device)
                Y = torch.zeros((self.M, 3 * w.h_out), dtype=y.dtype, device=device)
                X[:, w.h_in:2 * w.h_in] = x
                Y[:, w.h_out:2 * w.h_out] = y
                x, y = X[:, w.h_in:2 * w.h_in], Y[:, w.h_out:2 * w.h_out]
            self.x.append(x)
            self.y.append(y)
        self.v = None
        self.plan = None

    def make_plan(self):
        """The batch's plan (sgmv_plan), built once and reused by every planned call."""
        import torch
        from segmented_gather_gemm_sgmv_gb300 import sgmv_plan
        self.plan = sgmv_plan(self.d_ss, self.d_sa, self.M)
        torch.cuda.synchronize()

    def call_planned(self, i, stream=None):
        from segmented_gather_gemm_sgmv_gb300 import lora_apply_planned
        lora_apply_planned(self.y[i], self.x[i], self.A_ptrs, self.B_ptrs, self.plan,
                           i % self.w.layers, self.w.r, self.w.scale, stream=stream,
                           overlap_prior=self.overlap, tensor_cores=self.tensor_cores,
                           long_batch=self.long_batch, dense_grid=self.dense_grid)

    def call(self, i, stream=None):
        from segmented_gather_gemm_sgmv_gb300 import lora_apply
        lora_apply(self.y[i], self.x[i], self.A_ptrs, self.B_ptrs, self.d_ss, self.d_sa,
                   i % self.w.layers, self.w.r, self.w.scale, stream=stream,
                   overlap_prior=self.overlap, tensor_cores=self.tensor_cores,
                   long_batch=self.long_batch, dense_grid=self.dense_grid)

    def call_unfused(self, i, stream=None):
        """The pages' two launches per layer: sgmv_shrink into v, then sgmv_expand."""
        import torch
        from segmented_gather_gemm_sgmv_gb300 import sgmv_expand, sgmv_shrink
        if self.v is None:
            self.v = torch.zeros((self.M, self.w.r), dtype=torch.float32, device=self.x[0].device)
        kw = dict(stream=stream, tensor_cores=self.tensor_cores, long_batch=self.long_batch,
                  overlap_prior=self.overlap, dense_grid=self.dense_grid)
        sgmv_shrink(self.v, self.x[i], self.A_ptrs, self.d_ss, self.d_sa, i % self.w.layers,
                    self.w.r, **kw)
        sgmv_expand(self.y[i], self.v, self.B_ptrs, self.d_ss, self.d_sa, i % self.w.layers,
                    self.w.r, self.w.scale, **kw)

    def flags_text(self):
        t = ("lora_apply_ex(SGMV_OVERLAP_PRIOR): each call's weight prefetch overlaps the "
             "previous call (programmatic dependent launch)" if self.overlap else
             "lora_apply: each call starts after the previous one completes")
        if self.long_batch:
            t += "; SGMV_LONG_BATCH (a prefill batch: one CTA per SM, whole shared memory)"
        if self.dense_grid and not self.long_batch:
            t += ("; SGMV_DENSE_GRID (a decode batch of many work items: two CTAs of the call "
                  "per SM)")
        return t


def capture_step(torch, fn, n, stream):
    """A CUDA graph of one step (n calls)."""
    torch.cuda.synchronize()  # inputs made on other streams are complete before the first call
    with torch.cuda.stream(stream):
        for i in range(n):  # uncaptured first calls set the kernels' attributes
            fn(i, stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            fn(i, stream)
    return g


def time_steps(torch, g, K, W, stream, world=1):
    """Device time (ms) of exactly K replays of the step graph after W untimed ones; barrier +
    synchronize on both sides; CUDA events on the launching stream."""
    with torch.cuda.stream(stream):
        for _ in range(W):
            g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(K):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1)


def steps_for(torch, g, stream, seconds):
    """How many replays of g fill about `seconds` (measured on a few replays)."""
    ms = time_steps(torch, g, 3, 2, stream)
    return max(5, int(seconds * 1e3 / max(ms / 3, 1e-3)))


def measure_config(torch, name, device, stream, seconds, args):
    """One per_config entry: chained, isolated and unfused us per call, with clocks."""
    w = workloads.WORKLOADS[name]
    long_batch = {"auto": w.prefill, "on": True, "off": False}[args.long_batch]
    ss0, sa0 = workloads.make_segments(w.name, 0)
    dense = {"auto": dense_grid_rule(w, ss0, sa0), "on": True,
             "off": False}[args.dense_grid]
    setup = Setup(w, device, tensor_cores=args.tensor_cores, long_batch=long_batch,
                  dense_grid=dense)
    n = setup.calls
    out = {"calls_per_step": n, "layers": w.layers}
    nbytes, M = algorithmic_bytes(w, setup.ss, setup.sa)
    setup.make_plan()
    for label, overlap, fn in (("isolated", False, setup.call), ("unfused", True,
                                                                 setup.call_unfused),
                               ("planned_isolated", False, setup.call_planned),
                               ("planned_chained", True, setup.call_planned),
                               ("chained", True, setup.call)):
        setup.overlap = overlap
        g = capture_step(torch, fn, n, stream)
        K = steps_for(torch, g, stream, seconds)
        clocks = ClockSampler(torch.cuda.current_device()).start() if label == "chained" else None
        ms = time_steps(torch, g, K, 3, stream)
        us = ms * 1e3 / (K * n)
        out[f"us_per_call_{label}"] = round(us, 3)
        if clocks is not None:
            out["clocks"] = clocks.stop()
            out["timed_calls"] = K * n
        del g
    from segmented_gather_gemm_sgmv_gb300 import binding
    if binding.sgmv_get_error(clear=True) != 0:
        raise RuntimeError(f"{name}: a device-side wait ran out")
    us = out["us_per_call_chained"]
    out.update({
        "launch": setup.flags_text(),
        "unfused_launch": "sgmv_shrink_ex + sgmv_expand_ex (two launches per call, same flags)",
        "GB_per_s": round(nbytes / us / 1e3, 2),
        "tokens_per_s": round(M / us * 1e6, 1),
        "bytes_per_call": nbytes, "flops_per_call": flops(w, M), "tokens": M,
        "distinct_adapters": len(group_rows(setup.ss, setup.sa)),
        "tensor_core_rows": tensor_core_rows(w, setup.ss, setup.sa, args.tensor_cores),
        "roofline": roofline(w, setup.ss, setup.sa, us, args.tensor_cores),
        "roofline_isolated_frac": roofline(w, setup.ss, setup.sa, out["us_per_call_isolated"],
                                           args.tensor_cores)["frac"],
        "roofline_planned_frac": roofline(w, setup.ss, setup.sa, out["us_per_call_planned_chained"],
                                          args.tensor_cores)["frac"],
        "planned_launch": "sgmv_plan once per batch, then lora_apply_planned (same flags)",
    })
    del setup
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def measure_multi(torch, device, stream, seconds):
    """q, k and v of a Llama-7B attention block (h = 4096, r = 16, fp16, the decode_distinct
    batch and pool shape, each projection its own pool): one lora_apply_multi launch per layer
    against three lora_apply_planned launches per layer, over a 32-layer step."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_multi, lora_apply_planned
    w = workloads.WORKLOADS["decode_distinct"]
    setups = [Setup(w, device, seed=s) for s in (0, 10, 20)]
    for st in setups:
        st.overlap = True
    setups[0].make_plan()
    plan = setups[0].plan
    n = setups[0].calls

    # one launch carries three projections' work items (192 of them): the many-item geometry
    # (SGMV_DENSE_GRID, two CTAs per SM), as a caller batching projections would declare it
    def multi(i, stream=None):
        lora_apply_multi([(st.y[i], st.x[i], st.A_ptrs, st.B_ptrs, w.scale) for st in setups],
                         plan, i % w.layers, w.r, stream=stream, overlap_prior=True,
                         dense_grid=True)

    def three(i, stream=None):
        for st in setups:
            lora_apply_planned(st.y[i], st.x[i], st.A_ptrs, st.B_ptrs, plan, i % w.layers, w.r,
                               w.scale, stream=stream, overlap_prior=True)

    nbytes, M = algorithmic_bytes(w, setups[0].ss, setups[0].sa)
    out = {"projections": 3, "workload": "decode_distinct x 3 (q, k, v)",
           "bytes_per_layer": 3 * nbytes}
    for label, fn in (("multi", multi), ("three_planned", three)):
        g = capture_step(torch, fn, n, stream)
        K = steps_for(torch, g, stream, seconds)
        ms = time_steps(torch, g, K, 3, stream)
        us = ms * 1e3 / (K * n)
        out[f"us_per_layer_{label}"] = round(us, 3)
        out[f"GB_per_s_{label}"] = round(3 * nbytes / us / 1e3, 2)
        del g
    out["launch"] = ("lora_apply_multi (one launch per layer for q, k, v; SGMV_OVERLAP_PRIOR | "
                     "SGMV_DENSE_GRID) vs three lora_apply_planned launches (SGMV_OVERLAP_PRIOR)")
    del setups
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def measure_ranked(torch, device, stream, seconds):
    """Mixed ranks in one decode batch: the decode_distinct batch (64 one-token segments, h =
    4096, fp16, 32 layers) with adapter k of rank (8, 16, 32, 64)[k % 4], each stored at its own
    rank, through lora_apply_ranked (r_max = 64); beside it the same batch with every adapter
    padded to rank 64 through lora_apply."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply, lora_apply_ranked
    w = workloads.WORKLOADS["decode_distinct"]
    ranks = [(8, 16, 32, 64)[k % 4] for k in range(w.num_adapters)]
    ss, sa = workloads.make_segments(w.name, 0)
    M, L = int(ss[-1]), w.layers
    g = torch.Generator(device=device).manual_seed(5)
    A = [torch.randn((L, w.h_in, r), generator=g, device=device, dtype=torch.float16)
         for r in ranks]
    B = [torch.randn((L, r, w.h_out), generator=g, device=device, dtype=torch.float16)
         for r in ranks]
    A_ptrs = torch.tensor([a.data_ptr() for a in A], dtype=torch.int64, device=device)
    B_ptrs = torch.tensor([b.data_ptr() for b in B], dtype=torch.int64, device=device)
    Ap = torch.randn((w.num_adapters, L, w.h_in, 64), generator=g, device=device,
                     dtype=torch.float16)
    Bp = torch.randn((w.num_adapters, L, 64, w.h_out), generator=g, device=device,
                     dtype=torch.float16)
    Ap_ptrs, Bp_ptrs = workloads.pointer_table(Ap, device), workloads.pointer_table(Bp, device)
    d_rank = torch.tensor(ranks, dtype=torch.int32, device=device)
    d_scale = torch.tensor([16.0 / r for r in ranks], dtype=torch.float32, device=device)
    d_ss, d_sa = torch.as_tensor(ss, device=device), torch.as_tensor(sa, device=device)
    acts = [workloads.make_activations(w, M, device, seed=300 + i) for i in range(L)]

    def ranked(i, stream=None):
        x, y = acts[i]
        lora_apply_ranked(y, x, A_ptrs, B_ptrs, d_rank, d_scale, i, 64, seg_starts=d_ss,
                          seg_adapter=d_sa, stream=stream, overlap_prior=True)

    def padded(i, stream=None):
        x, y = acts[i]
        lora_apply(y, x, Ap_ptrs, Bp_ptrs, d_ss, d_sa, i, 64, 0.25, stream=stream,
                   overlap_prior=True)

    eb = 2
    act = M * w.h_in * eb + 2 * M * w.h_out * eb
    nbytes = sum((w.h_in + w.h_out) * ranks[int(k)] * eb for k in set(sa.tolist())) + act
    nbytes_padded = len(set(sa.tolist())) * (w.h_in + w.h_out) * 64 * eb + act
    out = {"workload": "decode_distinct batch, adapter ranks (8, 16, 32, 64) cycling, r_max 64",
           "bytes_per_call": nbytes, "bytes_per_call_padded": nbytes_padded}
    for label, fn, nb in (("ranked", ranked, nbytes), ("padded_r64", padded, nbytes_padded)):
        gr = capture_step(torch, fn, L, stream)
        K = steps_for(torch, gr, stream, seconds)
        ms = time_steps(torch, gr, K, 3, stream)
        us = ms * 1e3 / (K * L)
        out[f"us_per_call_{label}"] = round(us, 3)
        out[f"GB_per_s_{label}"] = round(nb / us / 1e3, 2)
        del gr
    hbm, _, kind = measured_peaks()
    out["roofline_frac_ranked"] = round(nbytes / (hbm * 1e9) / (out["us_per_call_ranked"] * 1e-6),
                                        4)
    out["launch"] = ("lora_apply_ranked (each adapter read at its own rank) vs lora_apply on "
                     "rank-64 copies, SGMV_OVERLAP_PRIOR, 32-layer steps")
    del A, B, Ap, Bp, acts
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def measure_base(torch, device, stream, seconds):
    """The base projection with the LoRA term in its epilogue (lora_apply_base) at the
    prefill_mixed shape (4096 -> 11008, r = 64, bf16, 8 segments of 128-1024 rows), against
    the same output made unfused: a cuBLAS GEMM (torch.matmul) writing x W0^T, then lora_apply
    reading and rewriting y; and against the cuBLAS GEMM alone (no LoRA term: the floor).  Two
    sets of (x, W0, y) alternate, so a call's footprint (~195 MB) is not in L2 from the call
    before."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply, lora_apply_base
    w = workloads.WORKLOADS["prefill_mixed"]
    ss, sa = workloads.make_segments(w.name, 0)
    M = int(ss[-1])
    A, B = workloads.make_pool(w, device, seed=41)
    A_ptrs, B_ptrs = workloads.pointer_table(A, device), workloads.pointer_table(B, device)
    d_ss, d_sa = torch.as_tensor(ss, device=device), torch.as_tensor(sa, device=device)
    g = torch.Generator(device=device).manual_seed(43)
    bound = 1.0 / np.sqrt(w.h_in)
    sets = []
    for i in range(2):
        x, y = workloads.make_activations(w, M, device, seed=600 + i)
        W0 = ((torch.rand((w.h_out, w.h_in), generator=g, device=device) * 2 - 1) *
              bound).to(torch.bfloat16)
        sets.append((x, W0, y))
    v_work = torch.empty((M, w.r), dtype=torch.float32, device=device)

    def fused(i, stream=None):
        x, W0, y = sets[i % 2]
        lora_apply_base(y, x, W0, A_ptrs, B_ptrs, d_ss, d_sa, 0, w.r, w.scale, v_work=v_work,
                        stream=stream, long_batch=True)

    def unfused(i, stream=None):
        x, W0, y = sets[i % 2]
        torch.matmul(x, W0.t(), out=y)
        lora_apply(y, x, A_ptrs, B_ptrs, d_ss, d_sa, 0, w.r, w.scale, stream=stream,
                   long_batch=True)

    def cublas(i, stream=None):
        x, W0, y = sets[i % 2]
        torch.matmul(x, W0.t(), out=y)

    _, tc_peak, kind = measured_peaks()
    hbm = measured_peaks()[0]
    f_base = 2.0 * M * w.h_in * w.h_out
    f_lora = 2.0 * M * w.r * (w.h_in + w.h_out)
    eb = 2
    nbytes = (M * w.h_in + w.h_out * w.h_in + M * w.h_out) * eb + \
        len(set(sa.tolist())) * w.r * (w.h_in + w.h_out) * eb
    out = {"workload": "prefill_mixed shape: x [%d, 4096] . W0^T [4096, 11008] + LoRA r=64, bf16"
                       % M, "flops_base": f_base, "flops_lora": f_lora, "bytes_min": nbytes}
    n = 8
    for label, fn in (("fused", fused), ("unfused", unfused), ("cublas_gemm_only", cublas)):
        gr = capture_step(torch, fn, n, stream)
        K = steps_for(torch, gr, stream, seconds)
        clocks = ClockSampler(torch.cuda.current_device()).start() if label == "fused" else None
        ms = time_steps(torch, gr, K, 3, stream)
        if clocks is not None:
            out["clocks"] = clocks.stop()
        us = ms * 1e3 / (K * n)
        out[f"us_per_call_{label}"] = round(us, 2)
        out[f"TFLOP_per_s_{label}"] = round((f_base + (f_lora if label != "cublas_gemm_only"
                                                       else 0.0)) / us / 1e6, 1)
        del gr
    us = out["us_per_call_fused"]
    t_flop = (f_base + f_lora) / (tc_peak * 1e12)
    t_mem = nbytes / (hbm * 1e9)
    out["roofline"] = {"bound": "tensor" if t_flop >= t_mem else "hbm",
                       "achieved": out["TFLOP_per_s_fused"], "peak": tc_peak, "unit": "TFLOP/s",
                       "frac": round(max(t_flop, t_mem) / (us * 1e-6), 4),
                       "peak_source": kind + " (bf16 sustained)",
                       "t_flop_us": round(t_flop * 1e6, 2), "t_mem_us": round(t_mem * 1e6, 2)}
    out["launch"] = ("lora_apply_base (sgmv_shrink_strided + the tcgen05 GEMM whose epilogue adds "
                     "the LoRA term; y written once) vs torch.matmul + lora_apply (y written, "
                     "then read and rewritten) vs torch.matmul alone")
    del sets, A, B, v_work
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def measure_paging(torch, device, stream, seconds):
    """Adapter paging (sgmv_pool_*): the decode_distinct shape (64 one-token segments, h = 4096,
    r = 16, fp16, 32 layers) with 128 adapters in pinned host memory and a 64-slot device pool;
    every step draws a new batch (64 distinct ids drawn by Zipf(1.2) weight over the 128, one
    token each), acquires it (cold adapters are
    copied on a copy stream while the previous step computes), replays the 32-layer graph and
    releases it; no host wait between steps.  Beside it: the same steps with every adapter
    resident (no pool)."""
    from segmented_gather_gemm_sgmv_gb300 import AdapterPool, SgmvError, lora_apply
    w = workloads.WORKLOADS["decode_distinct"]
    n_adapters, slots, L, M = 128, 64, w.layers, 64
    A, B = workloads.make_pool(w, device, seed=7, num_adapters=n_adapters)
    hA = [A[k].cpu().contiguous().pin_memory() for k in range(n_adapters)]
    hB = [B[k].cpu().contiguous().pin_memory() for k in range(n_adapters)]
    pool = AdapterPool(slots, n_adapters, L, w.h_in, w.h_out, w.r, torch.float16, device=device)
    for k in range(n_adapters):
        pool.register(k, hA[k], hB[k])
    rng = np.random.default_rng(11)
    ss = np.arange(M + 1, dtype=np.int32)
    d_ss = torch.as_tensor(ss, device=device)
    # 64 requests per step, each with its own adapter: distinct ids drawn by Zipf(1.2) weight
    # (hot adapters stay resident, cold ones stream in)
    zw = np.arange(1, n_adapters + 1, dtype=np.float64) ** -1.2
    batches = [rng.choice(n_adapters, size=M, replace=False, p=zw / zw.sum()).astype(np.int32)
               for _ in range(64)]
    host_sa = [torch.as_tensor(b).pin_memory() for b in batches]
    d_sa = torch.as_tensor(batches[0], device=device)  # the table every step rewrites
    acts = [workloads.make_activations(w, M, device, seed=500 + i) for i in range(L)]
    res_A, res_B = workloads.pointer_table(A, device), workloads.pointer_table(B, device)
    tables = {"pool": (pool.A_ptrs, pool.B_ptrs), "resident": (res_A, res_B)}
    copy_s = torch.cuda.Stream(device)

    def sweep(Ap, Bp):
        def fn(i, stream=None):
            x, y = acts[i]
            lora_apply(y, x, Ap, Bp, d_ss, d_sa, i, w.r, w.scale, stream=stream,
                       overlap_prior=True)
        return fn

    out = {"workload": "decode_distinct shape, 128 adapters on the host, 64-slot pool, 64 "
                       "distinct ids per step drawn by Zipf(1.2) weight, 32-layer steps",
           "slot_bytes": pool.slot_bytes}
    nbytes_call, _ = algorithmic_bytes(w, ss, batches[0])
    for label in ("resident", "pool"):
        if label == "pool":  # the capture's first pass reads the pool's tables: fill them
            pool.acquire(batches[0], copy_s, stream)
            pool.release(batches[0], stream)
        g = capture_step(torch, sweep(*tables[label]), L, stream)
        copied = 0

        def one(j):
            nonlocal copied
            b = batches[j % len(batches)]
            if label == "pool":
                while True:
                    try:
                        copied += pool.acquire(b, copy_s, stream)
                        break
                    except SgmvError as e:
                        if e.status != -7:
                            raise
                        stream.synchronize()  # too few idle slots: let the last step finish
            d_sa.copy_(host_sa[j % len(batches)], non_blocking=True)
            g.replay()
            if label == "pool":
                pool.release(b, stream)

        with torch.cuda.stream(stream):
            for j in range(8):
                one(j)
            torch.cuda.synchronize()
            copied = 0
            n = 64
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for j in range(n):
                one(8 + j)
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        out[f"us_per_step_{label}"] = round(ms * 1e3, 2)
        out[f"us_per_call_{label}"] = round(ms * 1e3 / L, 3)
        if label == "pool":
            out["adapters_copied_per_step"] = round(copied / n, 2)
            out["copy_GB_per_step"] = round(copied / n * pool.slot_bytes / 1e9, 4)
        del g
    out["pool_stats"] = pool.stats()
    out["launch"] = ("per step: sgmv_pool_acquire (copy stream), segment ids H2D, the 32-call "
                     "lora_apply graph (SGMV_OVERLAP_PRIOR), sgmv_pool_release; no host waits")
    pool.close()
    del A, B, hA, hB, acts, pool
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def time_e2e(torch, setup, K, stream):
    """Public-API path with pinned host buffers, one host->device copy and one device->host copy
    per step: the step's inputs (every call's x and y_in, then the segment table, packed in one
    pinned staging buffer) go in with ONE copy, the step's calls run on views of the device
    copy (the same lora_apply calls and flags as the device-timed step), and every call's y
    comes back with ONE copy (measured: one copy per direction per step doubled the figure
    against one per call; cutting each copy into four chunks on streams of their own lowered
    it again).  Steps alternate between two streams and two device / host buffer
    sets, so that one step's copies overlap the other step's kernels; a CUDA graph holds four
    steps.  Returns seconds per step and the bytes copied in and out per step."""
    w = setup.w
    dt = workloads.torch_dtype(w.dtype)
    x0, y0 = setup.x[0], setup.y[0]
    eb = x0.element_size()
    n = setup.calls

    def up16(v):
        return (v + 15) // 16 * 16

    nx, ny = up16(x0.numel() * eb), up16(y0.numel() * eb)
    nss, nsa = 4 * len(setup.ss), 4 * len(setup.sa)
    off_y = n * nx
    off_ss = off_y + n * ny
    off_sa = off_ss + up16(nss)
    total = off_sa + up16(nsa)
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for i in range(n):
        host[i * nx:i * nx + x0.numel() * eb].copy_(
            setup.x[i].cpu().contiguous().view(torch.uint8).view(-1))
        host[off_y + i * ny:off_y + i * ny + y0.numel() * eb].copy_(
            setup.y[i].cpu().contiguous().view(torch.uint8).view(-1))
    host[off_ss:off_ss + nss].copy_(torch.as_tensor(setup.ss).view(torch.uint8))
    host[off_sa:off_sa + nsa].copy_(torch.as_tensor(setup.sa).view(torch.uint8))
    streams = [stream, torch.cuda.Stream(x0.device)]
    sets = []
    for _ in range(2):
        dev = torch.empty(total, dtype=torch.uint8, device=x0.device)
        sets.append(dict(
            dev=dev,
            x=[dev[i * nx:i * nx + x0.numel() * eb].view(dt).view(x0.shape) for i in range(n)],
            y=[dev[off_y + i * ny:off_y + i * ny + y0.numel() * eb].view(dt).view(y0.shape)
               for i in range(n)],
            ys=dev[off_y:off_ss],
            ss=dev[off_ss:off_ss + nss].view(torch.int32),
            sa=dev[off_sa:off_sa + nsa].view(torch.int32),
            out=torch.empty(off_ss - off_y, dtype=torch.uint8).pin_memory()))
    from segmented_gather_gemm_sgmv_gb300 import lora_apply

    def one_step(j):
        st, b = streams[j % 2], sets[j % 2]
        with torch.cuda.stream(st):
            b["dev"].copy_(host, non_blocking=True)
            for i in range(n):
                lora_apply(b["y"][i], b["x"][i], setup.A_ptrs, setup.B_ptrs, b["ss"], b["sa"],
                           i % w.layers, w.r, w.scale, stream=st, overlap_prior=setup.overlap,
                           tensor_cores=setup.tensor_cores, long_batch=setup.long_batch,
                           dense_grid=setup.dense_grid)
            b["out"].copy_(b["ys"], non_blocking=True)

    per_graph = 4

    def steps():
        streams[1].wait_stream(streams[0])  # fork
        for j in range(per_graph):
            one_step(j)
        streams[0].wait_stream(streams[1])  # join

    with torch.cuda.stream(stream):
        steps()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        steps()
    reps = max(2, (K + per_graph - 1) // per_graph)
    ms = time_steps(torch, g, reps, 3, stream)
    return ms / 1e3 / (reps * per_graph), total, off_ss - off_y


def cpu_baseline(w, setup, seconds=10.0):
    """The fp64 oracle on all host cores: the headline batch at layer 0 split into disjoint
    segment ranges, one per thread (the oracle's C loop runs with the GIL released), repeated
    for ~seconds; the single-thread figure is reported beside it."""
    import oracle
    keys = sorted({int(k) for i, k in enumerate(setup.sa)
                   if k >= 0 and setup.ss[i + 1] > setup.ss[i]})
    A = [None] * setup.A.shape[0]
    B = [None] * setup.B.shape[0]
    for k in keys:
        A[k] = setup.A[k, 0:1].double().cpu().numpy()
        B[k] = setup.B[k, 0:1].double().cpu().numpy()
    y = setup.y[0].double().cpu().numpy()
    x = setup.x[0].double().cpu().numpy()
    ss, sa = np.asarray(setup.ss), np.asarray(setup.sa)
    nbytes, M = algorithmic_bytes(w, ss, sa)
    cores = max(1, min(os.cpu_count() or 1, len(sa)))
    parts = [p for p in np.array_split(np.arange(len(sa)), cores) if len(p)]
    calls = [oracle.PreparedApply(y, x, A, B, ss[p[0]:p[-1] + 2], sa[p[0]:p[-1] + 1], 0, w.scale)
             for p in parts]
    single = oracle.PreparedApply(y, x, A, B, ss, sa, 0, w.scale)

    def timed(fn, budget):
        n, t0 = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            el = time.perf_counter() - t0
            if el >= budget:
                return el / n, n, el

    with cf.ThreadPoolExecutor(max_workers=len(calls)) as ex:
        per, n, el = timed(lambda: list(ex.map(lambda c: c(), calls)), seconds)
    per1, n1, _ = timed(single, min(seconds, 3.0))
    return {"value": round(nbytes / per / 1e9, 4), "unit": "GB/s", "cores": len(calls),
            "kind": "oracle",
            "sample": f"oracle_lora_apply (fp64) on the whole {w.name} batch ({M} tokens, layer "
                      f"0), split into {len(calls)} disjoint segment ranges on {len(calls)} "
                      f"threads; {n} calls in {el:.1f} s",
            "tokens_per_s": round(M / per, 2), "us_per_call": round(per * 1e6, 1),
            "single_thread": {"value": round(nbytes / per1 / 1e9, 4), "unit": "GB/s",
                              "us_per_call": round(per1 * 1e6, 1), "calls": n1}}


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
    stream = torch.cuda.Stream(device)
    K, W = args.steps, args.warmup

    per_config = {}
    if world == 1 and not args.no_per_config:
        for name in PER_CONFIG:
            per_config[name] = measure_config(torch, name, device, stream, args.config_seconds,
                                              args)
        per_config["qkv_multi"] = measure_multi(torch, device, stream, args.config_seconds)
        per_config["mixed_rank"] = measure_ranked(torch, device, stream, args.config_seconds)
        if args.paging:
            per_config["paging"] = measure_paging(torch, device, stream, args.config_seconds)

    w = workloads.WORKLOADS[args.workload]
    if args.pool_layers > 0:
        w = dataclasses.replace(w, layers=args.pool_layers)
    long_batch = {"auto": w.prefill, "on": True, "off": False}[args.long_batch]
    ss0, sa0 = workloads.make_segments(w.name, 0)
    dense = {"auto": dense_grid_rule(w, ss0, sa0), "on": True, "off": False}[args.dense_grid]
    setup = Setup(w, device, tensor_cores=args.tensor_cores, long_batch=long_batch,
                  strided=args.strided, dense_grid=dense)
    nbytes, M = algorithmic_bytes(w, setup.ss, setup.sa)
    n = setup.calls

    setup.overlap = False  # isolated calls (each kernel waits for the previous one to finish)
    g_iso = capture_step(torch, setup.call, n, stream)
    ms_iso = time_steps(torch, g_iso, max(K, 3), 3, stream, world)
    us_iso = ms_iso * 1e3 / (max(K, 3) * n)
    del g_iso
    setup.overlap = not args.no_overlap
    g = capture_step(torch, setup.call, n, stream)
    clocks = ClockSampler(torch.cuda.current_device()).start()
    ms = time_steps(torch, g, K, W, stream, world)
    # nvidia-smi samples every 50 ms: a short timed region is extended, for the clock record
    # only, by untimed replays of the same graph (the same load) for 0.3 s after it.
    extra = 0
    if ms < 300.0:
        per_ms = max(ms / K, 1e-3)
        extra = int(300.0 / per_ms) + 1
        with torch.cuda.stream(stream):
            for _ in range(extra):
                g.replay()
        torch.cuda.synchronize()
    clk = clocks.stop()
    clk["window"] = ("the W warm-up replays, the K timed steps" +
                     (f" and {extra} untimed replays of the same step after them" if extra else ""))
    ms = reduce_max(ms, world, device)
    if binding.sgmv_get_error(clear=True) != 0:
        raise RuntimeError("a device-side wait ran out during the timed region")
    per_step = ms / 1e3 / K
    us_call = per_step / n * 1e6
    e2e_s, h2d, d2h = time_e2e(torch, setup, max(3, min(K, 200)), stream)
    e2e_s = reduce_max(e2e_s, world, device)
    if world == 1 and not args.no_per_config:
        # the GEMM leg runs the GPU at its power cap: after the headline's timed region, so
        # that the lower clocks it leaves behind do not carry into it
        per_config["base_fused"] = measure_base(torch, device, stream, args.config_seconds)
    if rank != 0:
        dist_finish(world)
        return
    line = {
        "metric": METRIC,
        "value": round(job_value(world, nbytes * n, per_step), 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(per_step * 1e3, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "impl": "ours",
        "tokens_per_s": round(world * M / (us_call * 1e-6), 1),
        "us_per_call": round(us_call, 3),
        "us_per_call_isolated": round(us_iso, 3),
        "launch": setup.flags_text(),
        "config": {"workload": w.name, "h_in": w.h_in, "h_out": w.h_out, "r": w.r,
                   "tokens": M, "segments": int(len(setup.sa)),
                   "distinct_adapters": len(group_rows(setup.ss, setup.sa)),
                   "pool_adapters": w.num_adapters, "layers": w.layers,
                   "calls_per_step": n,
                   "step": f"one layer sweep: {n} lora_apply calls (layer_idx 0..{w.layers - 1}"
                           f"{', repeated' if w.layers == 1 else ''}), each on its own x / y "
                           "set, replayed from one CUDA graph",
                   "bytes_per_call": nbytes, "flops_per_call": flops(w, M),
                   "timing": "CUDA events on the launching stream around exactly K graph "
                             "replays, after W untimed ones",
                   "l2": "inputs larger than L2: each call reads another layer's weights and "
                         "another x/y set (the footprint of a step is > 129 MB)",
                   "layout": ("x, y: middle column third of rows 3 h apart (lora_apply_strided)"
                              if setup.strided else "x [M][h_in], y [M][h_out] dense"),
                   "parallelism": f"replica x{world}"},
        "roofline": dict(roofline(w, setup.ss, setup.sa, us_call, args.tensor_cores),
                         traffic=None if setup.strided else recorded_traffic(w.name),
                         kernel="sgmv_kernel<fused> (lora_apply)"),
        "e2e": {"value": round(job_value(world, nbytes * n, e2e_s), 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_call": round(e2e_s / n * 1e6, 3)},
        "gpu_launches": K * n,
        "clocks": clk,
    }
    if per_config:
        line["per_config"] = per_config
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
    """The fp64 oracle timed on the host cores, on this arm's workload and step: one step is the
    same layer sweep (the batch once per layer), every call split into disjoint segment ranges
    over all host cores.  Rank 0 only."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = workloads.WORKLOADS[args.workload]
    ss, sa = workloads.make_segments(w.name, 0)
    rng = np.random.default_rng(0)
    n_calls = sweep_len(w)
    layers = min(w.layers, 2)  # the work of a call does not depend on the layer's values
    keys = sorted({int(k) for i, k in enumerate(sa) if k >= 0 and ss[i + 1] > ss[i]})
    A = [None] * w.num_adapters
    B = [None] * w.num_adapters
    for k in keys:
        A[k] = rng.uniform(-1, 1, (layers, w.h_in, w.r)) / np.sqrt(w.h_in)
        B[k] = rng.standard_normal((layers, w.r, w.h_out)) / np.sqrt(w.r)
    M = int(ss[-1])
    x = rng.standard_normal((M, w.h_in))
    y = rng.standard_normal((M, w.h_out))
    cores = max(1, min(os.cpu_count() or 1, len(sa)))
    parts = [p for p in np.array_split(np.arange(len(sa)), cores) if len(p)]
    calls = [oracle.PreparedApply(y, x, A, B, ss[p[0]:p[-1] + 2], sa[p[0]:p[-1] + 1], 0, w.scale)
             for p in parts]
    with cf.ThreadPoolExecutor(max_workers=len(parts)) as ex:
        def step():
            for i in range(n_calls):
                list(ex.map(lambda c: c(i % layers), calls))
        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        el = time.perf_counter() - t0
    per = el / args.steps
    nbytes, _ = algorithmic_bytes(w, ss, sa)
    val = nbytes * n_calls / per / 1e9
    line = {"metric": METRIC, "value": round(val, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "h_in": w.h_in, "h_out": w.h_out, "r": w.r,
                       "tokens": M, "calls_per_step": n_calls,
                       "step": f"one layer sweep: the whole batch through {n_calls} oracle "
                               f"calls (fp64; layers alternate over {layers} weight layers), "
                               "each split over the host cores"},
            "tokens_per_s": round(M * n_calls / per, 2),
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": len(parts),
                             "kind": "oracle",
                             "sample": f"{args.steps} steps of {n_calls} oracle_lora_apply "
                                       f"calls on the {w.name} batch, {len(parts)} threads over "
                                       "disjoint segment ranges"},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_distinct", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config sweep of every named workload")
    ap.add_argument("--paging", action="store_true",
                    help="add the adapter-pool paging measurement to per_config")
    ap.add_argument("--config-seconds", type=float, default=0.4,
                    help="timed seconds per per_config measurement")
    ap.add_argument("--tensor-cores", choices=["auto", "never", "always"], default="auto",
                    help="which adapter groups use the tensor cores (lora_apply_ex flags)")
    ap.add_argument("--long-batch", choices=["auto", "on", "off"], default="auto",
                    help="SGMV_LONG_BATCH launches; auto: for workloads that hold prefill "
                         "segments (prefill_mixed, mixed_70b)")
    ap.add_argument("--dense-grid", choices=["auto", "on", "off"], default="auto",
                    help="SGMV_DENSE_GRID launches (two CTAs of a call per SM); auto: decode "
                         "batches of >= 128 rows over >= 32 adapter groups (decode_zipf, "
                         "decode_uniform)")
    ap.add_argument("--strided", action="store_true",
                    help="x and y are the middle column third of 3x-wide activations "
                         "(lora_apply_strided; the e2e figure stays on dense copies)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="plain lora_apply launches (no programmatic dependent launch)")
    ap.add_argument("--pool-layers", type=int, default=0,
                    help="pool layers of the workload (default: its own); a smaller pool for "
                         "profiling captures of the same kernel, whose work per call does not "
                         "depend on the layer count")
    ap.add_argument("--only-base", action="store_true",
                    help="run only the base_fused measurement (lora_apply_base at the "
                         "prefill_mixed shape) and print it; for profiling that kernel")
    argv = sys.argv[1:] if argv is None else argv
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" in os.environ:
        if int(os.environ["WORLD_SIZE"]) != args.gpus:
            ap.error(f"--gpus {args.gpus} disagrees with WORLD_SIZE={os.environ['WORLD_SIZE']}")
    elif args.gpus > 1:  # one process per GPU: re-launch with N local ranks
        sys.exit(subprocess.call(relaunch_cmd(argv, args.gpus)))
    if args.impl == "reference":
        run_reference(args)
    elif args.only_base:
        import torch
        device = torch.device("cuda", 0)
        torch.cuda.set_device(device)
        print(json.dumps({"base_fused": measure_base(torch, device, torch.cuda.Stream(device),
                                                     args.config_seconds)}), flush=True)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
