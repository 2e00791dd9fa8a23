"""Shared helpers of the GPU parity tests: seeded cases on the device, fp64 oracle inputs built
from exactly the stored values, and the elementwise tolerance check.

Tolerance (fp16/bf16/fp32 outputs): |y - y_ref| <= 1e-2 + 1e-2 * |y_ref| elementwise, y_ref the
fp64 oracle.  Index handling is checked bit-exactly by the integer-valued cases.
"""
from __future__ import annotations

import dataclasses

import numpy as np

import oracle
from segmented_gather_gemm_sgmv_gb300 import workloads

ATOL = 1e-2
RTOL = 1e-2


@dataclasses.dataclass
class Case:
    w: workloads.Workload
    ss: np.ndarray          # seg_starts (host)
    sa: np.ndarray          # seg_adapter (host)
    x: object               # torch [M, h_in] on device
    y0: object              # torch [M, h_out] base output (kept pristine)
    A: object               # torch [n, L, h_in, r]
    B: object               # torch [n, L, r, h_out]
    A_ptrs: object
    B_ptrs: object
    d_ss: object
    d_sa: object

    @property
    def M(self):
        return self.x.shape[0]


def make_case(w: workloads.Workload, ss, sa, device="cuda", seed=0, M=None,
              num_adapters=None, layers=None, pool=None):
    import torch
    ss = np.asarray(ss, np.int32)
    sa = np.asarray(sa, np.int32)
    M = int(max(ss[-1], ss.max(initial=0))) if M is None else M
    if pool is None:
        A, B = workloads.make_pool(w, device, seed=seed + 1, num_adapters=num_adapters,
                                   layers=layers)
    else:
        A, B = pool
    x, y0 = workloads.make_activations(w, M, device, seed=seed + 2)
    return Case(w, ss, sa, x, y0, A, B, workloads.pointer_table(A, device),
                workloads.pointer_table(B, device),
                torch.as_tensor(ss, device=device), torch.as_tensor(sa, device=device))


def touched(sa, ss):
    out = set()
    for i, k in enumerate(sa):
        if k >= 0 and ss[i + 1] > ss[i]:
            out.add(int(k))
    return out


def oracle_blocks(pool, keys, layer):
    """fp64 single-layer blocks of the adapters in `keys` (others None), exact widening."""
    n = pool.shape[0]
    blocks = [None] * n
    for k in keys:
        blocks[k] = pool[k, layer:layer + 1].double().cpu().numpy()
    return blocks


def oracle_apply(c: Case, layer, y_in=None, x=None, rows=None):
    """fp64 reference of lora_apply for case c at `layer`.

    rows=None: every row.  Otherwise only the listed rows are computed (each as its own
    length-1 segment with its adapter); returns (rows, y_ref[rows]).
    """
    y_in = c.y0 if y_in is None else y_in
    x = c.x if x is None else x
    keys = touched(c.sa, c.ss)
    A = oracle_blocks(c.A, keys, layer)
    B = oracle_blocks(c.B, keys, layer)
    if rows is None:
        return oracle.lora_apply(y_in.double().cpu().numpy(), x.double().cpu().numpy(), A, B,
                                 c.ss, c.sa, 0, c.w.scale)
    rows = np.asarray(sorted(set(int(r) for r in rows)), np.int64)
    adapter_of = row_adapters(c.ss, c.sa, c.M)
    sub_sa = adapter_of[rows].astype(np.int32)
    sub_ss = np.arange(len(rows) + 1, dtype=np.int32)
    idx = __import__("torch").as_tensor(rows, device=x.device)
    ref = oracle.lora_apply(y_in[idx].double().cpu().numpy(), x[idx].double().cpu().numpy(), A, B,
                            sub_ss, sub_sa, 0, c.w.scale)
    return rows, ref


def row_adapters(ss, sa, M):
    """Adapter id of every row (-1 for rows in no segment or with no adapter)."""
    out = np.full(M, -1, np.int64)
    for i, k in enumerate(sa):
        out[ss[i]:ss[i + 1]] = k
    return out


def assert_close(y, y_ref, what="", atol=ATOL, rtol=RTOL):
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    assert y.shape == y_ref.shape, (what, y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - y_ref)
    bound = atol + rtol * np.abs(y_ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: got {y[i]!r} want {y_ref[i]!r}")
    return float(err.max()) if err.size else 0.0


def run_apply(c: Case, layer, y=None, x=None, tensor_cores="auto", long_batch=False):
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    y = c.y0.clone() if y is None else y
    lora_apply(y, c.x if x is None else x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, layer, c.w.r,
               c.w.scale, tensor_cores=tensor_cores, long_batch=long_batch)
    return y
