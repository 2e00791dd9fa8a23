"""fp64 CPU oracle for segmented LoRA apply (SGMV shrink, expand and the fused apply).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The CUDA library never imports it, and it never
imports the CUDA library: the two meet only through the seeded inputs that a test hands to
both.

The arithmetic lives in ``sgmv_oracle.c`` (plain C, fp64, one token at a time); this module
compiles it with gcc on first use and marshals numpy arrays into it.  What it computes, per
"Punica Guide: Multi-Tenant LoRA Serving with SGMV" (section "The Heterogeneous Batching
Bottleneck", equation for y_i; section "The SGMV Mathematical Formulation"):

    for each segment i with adapter k = seg_adapter[i] (k < 0: no adapter),
        for each token t in [seg_starts[i], seg_starts[i+1]):
            y[t] += scale * (x[t] @ A_k[layer]) @ B_k[layer]

Inputs are float64 arrays holding the exact stored values (fp16/bf16/fp32 widen exactly).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgmv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_sgmv.so")
_lock = threading.Lock()
_lib = None

# Bits returned by validate(); they are the ones the library header documents.
BAD_ORDER = 1
BAD_FIRST = 2
BAD_LAST = 4
BAD_ADAPTER = 8
BAD_A_PTR = 16
BAD_B_PTR = 32


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile an oracle C source into a shared object (gcc, -O2, no FMA contraction)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stale = (not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src))
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-o", tmp, src]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


class _PtrTable:
    """A C array of per-adapter block pointers; keeps the blocks alive."""

    def __init__(self, blocks):
        self.blocks = [None if b is None else _f64(b) for b in blocks]
        n = max(1, len(self.blocks))
        self.table = (ctypes.c_void_p * n)()
        for k, b in enumerate(self.blocks):
            self.table[k] = None if b is None else b.ctypes.data

    @property
    def ptr(self):
        return ctypes.cast(self.table, ctypes.c_void_p)


def _check_segments(seg_starts, seg_adapter, nblocks, M):
    S = len(seg_adapter)
    if len(seg_starts) != S + 1:
        raise ValueError("seg_starts must hold num_segments + 1 offsets")
    for i in range(S):
        k = int(seg_adapter[i])
        lo, hi = int(seg_starts[i]), int(seg_starts[i + 1])
        if hi > lo and k >= 0:
            if k >= nblocks:
                raise ValueError(f"segment {i}: adapter {k} has no weight block")
            if lo < 0 or hi > M:
                raise ValueError(f"segment {i}: rows [{lo},{hi}) outside [0,{M})")


def _rank(blocks) -> int:
    for b in blocks:
        if b is not None:
            return int(np.shape(b)[-1])
    return 1


class OracleLib:
    """The oracle's entry points bound to one compiled shared object."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i32, dp = ctypes.c_int32, ctypes.c_void_p
        lib.oracle_lora_apply.argtypes = [dp, dp, dp, dp, dp, dp, i32, i32, i32, i32, i32,
                                          ctypes.c_double]
        lib.oracle_lora_apply.restype = ctypes.c_int
        lib.oracle_sgmv_shrink.argtypes = [dp, dp, dp, dp, dp, i32, i32, i32, i32]
        lib.oracle_sgmv_shrink.restype = ctypes.c_int
        lib.oracle_sgmv_expand.argtypes = [dp, dp, dp, dp, dp, i32, i32, i32, i32,
                                           ctypes.c_double]
        lib.oracle_sgmv_expand.restype = ctypes.c_int
        lib.oracle_validate.argtypes = [dp, dp, i32, i32, i32]
        lib.oracle_validate.restype = ctypes.c_int32
        lib.oracle_validate_pointers.argtypes = [dp, dp, dp, dp, i32, i32]
        lib.oracle_validate_pointers.restype = ctypes.c_int32
        lib.oracle_plan.argtypes = [dp, dp, i32, i32, dp, dp, dp]
        lib.oracle_lora_apply_ranked.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i32, i32, i32,
                                                 i32]
        lib.oracle_lora_apply_ranked.restype = ctypes.c_int
        lib.oracle_plan.restype = ctypes.c_int32
        lib.oracle_base_lora.argtypes = [dp, dp, dp, dp, dp, dp, dp, i32, i32, i32, i32, i32,
                                         i32, ctypes.c_double]
        lib.oracle_base_lora.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    def lora_apply(self, y, x, A_blocks, B_blocks, seg_starts, seg_adapter, layer_idx, scale):
        """Return y + scale * (x A_k) B_k per segment (fp64).  y is not modified.

        y: (M, h_out); x: (M, h_in); A_blocks[k]: (L, h_in, r) or None for an adapter no
        segment uses; B_blocks[k]: (L, r, h_out) or None.
        """
        y = _f64(y).copy()
        x = _f64(x)
        ss, sa = _i32(seg_starts), _i32(seg_adapter)
        _check_segments(ss, sa, len(A_blocks), y.shape[0])
        At, Bt = _PtrTable(A_blocks), _PtrTable(B_blocks)
        rc = self.lib.oracle_lora_apply(y.ctypes.data, x.ctypes.data, At.ptr, Bt.ptr,
                                        ss.ctypes.data, sa.ctypes.data, len(sa),
                                        int(layer_idx), x.shape[1], y.shape[1],
                                        _rank(A_blocks), float(scale))
        if rc != 0:
            raise MemoryError("oracle_lora_apply failed")
        return y

    def sgmv_shrink(self, v, x, A_blocks, seg_starts, seg_adapter, layer_idx):
        """Return v with v[t] = x[t] A_k[layer] on every segment row (other rows kept)."""
        v = _f64(v).copy()
        x = _f64(x)
        ss, sa = _i32(seg_starts), _i32(seg_adapter)
        _check_segments(ss, sa, len(A_blocks), x.shape[0])
        At = _PtrTable(A_blocks)
        self.lib.oracle_sgmv_shrink(v.ctypes.data, x.ctypes.data, At.ptr, ss.ctypes.data,
                                    sa.ctypes.data, len(sa), int(layer_idx), x.shape[1],
                                    v.shape[1])
        return v

    def sgmv_expand(self, y, v, B_blocks, seg_starts, seg_adapter, layer_idx, scale):
        """Return y + scale * v[t] B_k[layer] on every segment row."""
        y = _f64(y).copy()
        v = _f64(v)
        ss, sa = _i32(seg_starts), _i32(seg_adapter)
        _check_segments(ss, sa, len(B_blocks), y.shape[0])
        Bt = _PtrTable(B_blocks)
        self.lib.oracle_sgmv_expand(y.ctypes.data, v.ctypes.data, Bt.ptr, ss.ctypes.data,
                                    sa.ctypes.data, len(sa), int(layer_idx), v.shape[1],
                                    y.shape[1], float(scale))
        return y

    def validate(self, seg_starts, seg_adapter, num_adapters, M) -> int:
        """OR of BAD_* bits for a segment table (0 = valid)."""
        ss, sa = _i32(seg_starts), _i32(seg_adapter)
        if len(ss) != len(sa) + 1:
            raise ValueError("seg_starts must hold num_segments + 1 offsets")
        return int(self.lib.oracle_validate(ss.ctypes.data, sa.ctypes.data, len(sa),
                                            int(num_adapters), int(M)))

    def validate_pointers(self, A_addr, B_addr, seg_starts, seg_adapter, num_adapters) -> int:
        """OR of BAD_A_PTR / BAD_B_PTR for the weight addresses (integer sequences of
        num_adapters entries, or None) that the table's non-empty segments use."""
        ss, sa = _i32(seg_starts), _i32(seg_adapter)
        if len(ss) != len(sa) + 1:
            raise ValueError("seg_starts must hold num_segments + 1 offsets")
        keep = []

        def arr(a):
            if a is None:
                return None
            v = np.ascontiguousarray(np.asarray(a, dtype=np.uint64))
            if len(v) < num_adapters:
                raise ValueError("an address array needs num_adapters entries")
            keep.append(v)
            return v.ctypes.data

        return int(self.lib.oracle_validate_pointers(arr(A_addr), arr(B_addr), ss.ctypes.data,
                                                     sa.ctypes.data, len(sa),
                                                     int(num_adapters)))


    def lora_apply_ranked(self, y, x, A_blocks, B_blocks, rank, scale, seg_starts, seg_adapter,
                          layer_idx):
        """Return y + scale[k] * (x A_k) B_k per segment (fp64), adapter k of rank rank[k]:
        A_blocks[k] (L, h_in, rank[k]) and B_blocks[k] (L, rank[k], h_out), or None for an
        adapter no segment uses.  y is not modified."""
        y = _f64(y).copy()
        x = _f64(x)
        ss, sa = _i32(seg_starts), _i32(seg_adapter)
        _check_segments(ss, sa, len(A_blocks), y.shape[0])
        rk = _i32(rank)
        sc = _f64(scale)
        if len(rk) < len(A_blocks) or len(sc) < len(A_blocks):
            raise ValueError("rank and scale need one entry per adapter")
        for k, (a, b) in enumerate(zip(A_blocks, B_blocks)):
            if a is not None and (np.shape(a)[-1] != rk[k] or np.shape(b)[-2] != rk[k]):
                raise ValueError(f"adapter {k}: blocks do not have rank {rk[k]}")
        At, Bt = _PtrTable(A_blocks), _PtrTable(B_blocks)
        rc = self.lib.oracle_lora_apply_ranked(y.ctypes.data, x.ctypes.data, At.ptr, Bt.ptr,
                                               rk.ctypes.data, sc.ctypes.data, ss.ctypes.data,
                                               sa.ctypes.data, len(sa), int(layer_idx),
                                               x.shape[1], y.shape[1])
        if rc != 0:
            raise MemoryError("oracle_lora_apply_ranked failed")
        return y

    def base_lora(self, x, W0, A_blocks, B_blocks, seg_starts, seg_adapter, layer_idx, scale):
        """Return y = x W0^T + scale * (x A_k) B_k per segment row (fp64, a new array).

        x: (M, h_in); W0: (h_out, h_in), one row per output feature; A_blocks / B_blocks as for
        lora_apply.  Rows outside every segment, or of a segment without an adapter, get the
        base projection only.
        """
        x = _f64(x)
        W0 = _f64(W0)
        M, h_in = x.shape
        h_out = W0.shape[0]
        if W0.shape[1] != h_in:
            raise ValueError("W0 must be (h_out, h_in)")
        ss, sa = _i32(seg_starts), _i32(seg_adapter)
        _check_segments(ss, sa, len(A_blocks), M)
        y = np.full((M, h_out), np.nan)  # every element is written
        At, Bt = _PtrTable(A_blocks), _PtrTable(B_blocks)
        rc = self.lib.oracle_base_lora(y.ctypes.data, x.ctypes.data, W0.ctypes.data, At.ptr,
                                       Bt.ptr, ss.ctypes.data, sa.ctypes.data, len(sa), M,
                                       int(layer_idx), h_in, h_out, _rank(A_blocks),
                                       float(scale))
        if rc != 0:
            raise MemoryError("oracle_base_lora failed")
        return y

    def plan(self, seg_starts, seg_adapter, max_rows):
        """The adapter grouping of a table: (g_starts[G+1], g_adapter[G], rows[n]) as int32
        arrays, or None when more than max_rows rows would be listed."""
        ss, sa = _i32(seg_starts), _i32(seg_adapter)
        if len(ss) != len(sa) + 1:
            raise ValueError("seg_starts must hold num_segments + 1 offsets")
        S = len(sa)
        gs = np.zeros(S + 1, np.int32)
        ga = np.zeros(max(S, 1), np.int32)
        rows = np.zeros(max(int(max_rows), 1), np.int32)
        G = int(self.lib.oracle_plan(ss.ctypes.data, sa.ctypes.data, S, int(max_rows),
                                     gs.ctypes.data, ga.ctypes.data, rows.ctypes.data))
        if G < 0:
            return None
        return gs[:G + 1].copy(), ga[:G].copy(), rows[:gs[G]].copy()


def _load() -> OracleLib:
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build())
    return _lib


def lora_apply(*args, **kw):
    return _load().lora_apply(*args, **kw)


def sgmv_shrink(*args, **kw):
    return _load().sgmv_shrink(*args, **kw)


def sgmv_expand(*args, **kw):
    return _load().sgmv_expand(*args, **kw)


def validate(*args, **kw):
    return _load().validate(*args, **kw)


def validate_pointers(*args, **kw):
    return _load().validate_pointers(*args, **kw)


def plan(*args, **kw):
    return _load().plan(*args, **kw)


def lora_apply_ranked(*args, **kw):
    return _load().lora_apply_ranked(*args, **kw)


def base_lora(*args, **kw):
    return _load().base_lora(*args, **kw)


lora_apply.__doc__ = OracleLib.lora_apply.__doc__
sgmv_shrink.__doc__ = OracleLib.sgmv_shrink.__doc__
sgmv_expand.__doc__ = OracleLib.sgmv_expand.__doc__
validate.__doc__ = OracleLib.validate.__doc__
validate_pointers.__doc__ = OracleLib.validate_pointers.__doc__
plan.__doc__ = OracleLib.plan.__doc__
lora_apply_ranked.__doc__ = OracleLib.lora_apply_ranked.__doc__
base_lora.__doc__ = OracleLib.base_lora.__doc__


class PreparedApply:
    """Holds marshalled fp64 inputs so that repeated oracle calls time only the arithmetic.

    Used by the CPU-baseline leg of the benchmark; each call() adds the LoRA term into the
    held y buffer once more (the value grows, the work per call is identical).
    """

    def __init__(self, y, x, A_blocks, B_blocks, seg_starts, seg_adapter, layer_idx, scale):
        self._lib = _load().lib
        self.y = _f64(y).copy()
        self.x = _f64(x)
        self.ss, self.sa = _i32(seg_starts), _i32(seg_adapter)
        _check_segments(self.ss, self.sa, len(A_blocks), self.y.shape[0])
        self.At, self.Bt = _PtrTable(A_blocks), _PtrTable(B_blocks)
        self.args = (self.y.ctypes.data, self.x.ctypes.data, self.At.ptr, self.Bt.ptr,
                     self.ss.ctypes.data, self.sa.ctypes.data, len(self.sa), int(layer_idx),
                     self.x.shape[1], self.y.shape[1], _rank(A_blocks), float(scale))

    def __call__(self, layer_idx=None):
        args = self.args if layer_idx is None else (
            self.args[:7] + (int(layer_idx),) + self.args[8:])
        rc = self._lib.oracle_lora_apply(*args)
        if rc != 0:
            raise MemoryError("oracle_lora_apply failed")
