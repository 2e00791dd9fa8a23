"""Seeded synthetic inputs for segmented LoRA apply.

This module only draws random numbers and lays them out; it performs none of the method's
arithmetic.  Both the CUDA path (through the tests and the benchmark) and the fp64 oracle are
fed from it.  There is no dataset and there are no trained weights: shapes, value
distributions and segment structure follow five named workloads:

  tiny             h_in=h_out=256, r=8, fp32, 4 adapters, 6 segments of 1..4 tokens with
                   uniform ids in [0,4), alpha=16, 1 layer.
  decode_distinct  Llama-7B projection h=4096, r=16, fp16, 64 tokens, each its own length-1
                   segment and its own adapter of a 64-adapter pool stacked over 32 layers.
  decode_zipf      h=4096, r=16, fp16, 256 tokens whose ids are drawn from a Zipf(a=1.5)
                   law truncated to a 1024-adapter pool, sorted, one segment per run of equal
                   ids; variants decode_uniform (uniform ids) and decode_same (one id).
                   The pool is stacked over 16 layers so that a layer sweep leaves L2 cold.
  prefill_mixed    MLP up-projection 4096 -> 11008, r=64, bf16, 8 segments of 128..1024
                   tokens with 8 distinct adapters, 1 layer.
  mixed_70b        Llama-70B projection h=8192, r=64, bf16, 512 tokens: two prefill segments
                   of 16 tokens then 480 length-1 decode segments, 482 ids drawn i.i.d. from
                   a Zipf(a=1.2) law over 256 adapters (not sorted, so one adapter can own
                   several non-adjacent segments), pool stacked over 80 layers.

prefill_mixed and mixed_70b hold prefill segments: a serving layer knows that of its batch and
launches them with SGMV_LONG_BATCH (Workload.prefill).

Value distributions (all workloads): x ~ N(0,1); A ~ U(-1/sqrt(h_in), +1/sqrt(h_in));
B ~ N(0, sd=1/sqrt(r)); y_in ~ N(0,1) (the base output x W0 the LoRA term is added to);
scale = alpha / r with alpha = 16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

DTYPES = ("f32", "f16", "bf16")
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    h_in: int
    h_out: int
    r: int
    dtype: str
    num_adapters: int
    layers: int
    alpha: float = 16.0
    prefill: bool = False  # the batch holds prefill segments (a caller passes SGMV_LONG_BATCH)

    @property
    def scale(self) -> float:
        return self.alpha / self.r

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]


WORKLOADS = {
    "tiny": Workload("tiny", 256, 256, 8, "f32", 4, 1),
    "decode_distinct": Workload("decode_distinct", 4096, 4096, 16, "f16", 64, 32),
    "decode_zipf": Workload("decode_zipf", 4096, 4096, 16, "f16", 1024, 16),
    "decode_uniform": Workload("decode_uniform", 4096, 4096, 16, "f16", 1024, 16),
    "decode_same": Workload("decode_same", 4096, 4096, 16, "f16", 1024, 16),
    "prefill_mixed": Workload("prefill_mixed", 4096, 11008, 64, "bf16", 8, 1, prefill=True),
    "mixed_70b": Workload("mixed_70b", 8192, 8192, 64, "bf16", 256, 80, prefill=True),
}


def _runs_to_segments(ids_sorted: np.ndarray):
    """One segment per run of equal consecutive ids."""
    starts, adapters = [0], []
    for t, k in enumerate(ids_sorted):
        if t > 0 and k != ids_sorted[t - 1]:
            starts.append(t)
        if t == 0 or k != ids_sorted[t - 1]:
            adapters.append(int(k))
    starts.append(len(ids_sorted))
    return np.asarray(starts, np.int32), np.asarray(adapters, np.int32)


def zipf_ids(rng: np.random.Generator, n: int, pool: int, a: float) -> np.ndarray:
    """n i.i.d. ids in [0, pool) with P(k) proportional to (k+1)^-a (truncated Zipf)."""
    w = np.arange(1, pool + 1, dtype=np.float64) ** (-a)
    return rng.choice(pool, size=n, p=w / w.sum()).astype(np.int32)


def make_segments(name: str, seed: int = 0):
    """Return (seg_starts[int32, S+1], seg_adapter[int32, S]) for a named workload."""
    rng = np.random.default_rng(seed)
    if name == "tiny":
        lens = rng.integers(1, 5, size=6)
        ids = rng.integers(0, 4, size=6)
        starts = np.concatenate([[0], np.cumsum(lens)])
        return starts.astype(np.int32), ids.astype(np.int32)
    if name == "decode_distinct":
        ids = rng.permutation(64)
        return np.arange(65, dtype=np.int32), ids.astype(np.int32)
    if name == "decode_zipf":
        return _runs_to_segments(np.sort(zipf_ids(rng, 256, 1024, 1.5)))
    if name == "decode_uniform":
        return _runs_to_segments(np.sort(rng.integers(0, 1024, size=256)))
    if name == "decode_same":
        return np.array([0, 256], np.int32), np.array([0], np.int32)
    if name == "prefill_mixed":
        lens = rng.integers(128, 1025, size=8)
        ids = rng.permutation(8)
        starts = np.concatenate([[0], np.cumsum(lens)])
        return starts.astype(np.int32), ids.astype(np.int32)
    if name == "mixed_70b":
        ids = zipf_ids(rng, 482, 256, 1.2)
        starts = np.concatenate([[0, 16, 32], 32 + np.arange(1, 481)])
        return starts.astype(np.int32), ids
    raise KeyError(name)


def random_segments(rng: np.random.Generator, num_segments: int, max_len: int,
                    num_adapters: int, p_empty: float = 0.0, first: int = 0):
    """A random segment table: lengths in [1, max_len] (or 0 with probability p_empty)."""
    lens = rng.integers(1, max_len + 1, size=num_segments)
    if p_empty > 0:
        lens = np.where(rng.random(num_segments) < p_empty, 0, lens)
    starts = first + np.concatenate([[0], np.cumsum(lens)])
    ids = rng.integers(0, num_adapters, size=num_segments)
    return starts.astype(np.int32), ids.astype(np.int32)


# ---------------------------------------------------------------------------------------
# Tensors (torch is imported lazily so that the segment recipes work without it).
# ---------------------------------------------------------------------------------------

def torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def _gen(device, seed: int):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_pool(w: Workload, device, seed: int = 1, num_adapters: Optional[int] = None,
              layers: Optional[int] = None):
    """Adapter pool: A [n, L, h_in, r] ~ U(+-1/sqrt(h_in)), B [n, L, r, h_out] ~ N(0, 1/sqrt(r)).

    Each adapter owns one contiguous [L][h_in][r] block of A and [L][r][h_out] block of B.
    Filled one adapter at a time on `device` so that pools of tens of GB never need a
    full-size fp32 temporary.
    """
    import torch
    n = w.num_adapters if num_adapters is None else num_adapters
    L = w.layers if layers is None else layers
    dt = torch_dtype(w.dtype)
    g = _gen(device, seed)
    A = torch.empty((n, L, w.h_in, w.r), dtype=dt, device=device)
    B = torch.empty((n, L, w.r, w.h_out), dtype=dt, device=device)
    a_lim = 1.0 / math.sqrt(w.h_in)
    b_sd = 1.0 / math.sqrt(w.r)
    for k in range(n):
        t = torch.rand((L, w.h_in, w.r), generator=g, device=device, dtype=torch.float32)
        A[k].copy_(t.mul_(2.0 * a_lim).sub_(a_lim))
        t = torch.randn((L, w.r, w.h_out), generator=g, device=device, dtype=torch.float32)
        B[k].copy_(t.mul_(b_sd))
    return A, B


def make_activations(w: Workload, M: int, device, seed: int = 2):
    """x [M, h_in] ~ N(0,1) and the base output y_in [M, h_out] ~ N(0,1)."""
    import torch
    dt = torch_dtype(w.dtype)
    g = _gen(device, seed)
    x = torch.randn((M, w.h_in), generator=g, device=device, dtype=torch.float32).to(dt)
    y = torch.randn((M, w.h_out), generator=g, device=device, dtype=torch.float32).to(dt)
    return x, y


def pointer_table(pool, device):
    """int64 tensor of per-adapter base addresses of a [n, L, ...] pool (for A_ptrs/B_ptrs)."""
    import torch
    n = pool.shape[0]
    stride = pool.stride(0) * pool.element_size()
    base = pool.data_ptr()
    return torch.tensor([base + k * stride for k in range(n)], dtype=torch.int64, device=device)
