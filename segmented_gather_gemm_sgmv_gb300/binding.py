"""ctypes binding of libsgmv_gb300.so -- argument marshalling only.

Every function here has the name of a C entry point in include/sgmv.h, takes torch CUDA tensors
(PyTorch provides device memory and streams, nothing else), extracts pointers and sizes and
calls the library.  No step of the computation runs in Python, and there is no fallback: a
missing library, a CPU tensor or a failing status raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

SGMV_OK, SGMV_EINVAL, SGMV_EALIGN, SGMV_EUNSUPPORTED, SGMV_ECUDA, SGMV_ETIMEOUT = 0, -1, -2, -3, -4, -5
SGMV_EPLAN = -6
SGMV_ENOSPACE = -7
SGMV_EBUSY = -8
SGMV_MAX_PROJECTIONS = 4
SGMV_STATIC_PLAN_MAX_ROWS = 65536
PLAN_HEADER = 16  # int32 words before a plan's group table (include/sgmv.h)
SGMV_MAX_SEGMENTS = 4096
SGMV_MAX_HIDDEN = 65536
SGMV_OVERLAP_PRIOR = 1
SGMV_NO_TENSOR_CORES = 2
SGMV_TENSOR_CORES_ALWAYS = 4
SGMV_LONG_BATCH = 8
SGMV_DENSE_GRID = 16
SGMV_MAX_LD = 1 << 24
SYMBOLS = ("lora_apply", "lora_apply_ex", "lora_apply_strided", "sgmv_shrink", "sgmv_shrink_ex",
           "sgmv_shrink_strided", "sgmv_expand", "sgmv_expand_ex", "sgmv_expand_strided",
           "sgmv_validate", "sgmv_validate_pointers", "sgmv_get_error", "sgmv_set_wait_limit",
           "sgmv_status_string", "sgmv_version", "sgmv_plan_size", "sgmv_plan",
           "lora_apply_planned", "sgmv_shrink_planned", "sgmv_expand_planned", "lora_apply_multi",
           "lora_apply_ranked", "sgmv_pool_slot_bytes", "sgmv_pool_create", "sgmv_pool_destroy",
           "sgmv_pool_register", "sgmv_pool_acquire", "sgmv_pool_release", "sgmv_pool_stats",
           "lora_apply_static_plan", "lora_apply_base")


class Projection(ctypes.Structure):
    """sgmv_projection_t of include/sgmv.h."""
    _fields_ = [("y", ctypes.c_void_p), ("x", ctypes.c_void_p), ("A_ptrs", ctypes.c_void_p),
                ("B_ptrs", ctypes.c_void_p), ("ldy", ctypes.c_int32), ("ldx", ctypes.c_int32),
                ("h_in", ctypes.c_int32), ("h_out", ctypes.c_int32), ("scale", ctypes.c_float),
                ("reserved", ctypes.c_int32)]


class SgmvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def lib(build_if_stale: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the shared library and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if build_if_stale and _build.is_stale():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing; build it with "
                               "`python -m segmented_gather_gemm_sgmv_gb300.build`")
        L = ctypes.CDLL(path)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        L.lora_apply.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, ctypes.c_int,
                                 vp]
        L.lora_apply_ex.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32,
                                    ctypes.c_int, ctypes.c_uint32, vp]
        L.sgmv_shrink.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_int, vp]
        L.sgmv_expand.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, ctypes.c_int, vp]
        L.sgmv_shrink_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_int,
                                     ctypes.c_uint32, vp]
        L.sgmv_expand_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, ctypes.c_int,
                                     ctypes.c_uint32, vp]
        L.lora_apply_strided.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32,
                                         i32, f32, ctypes.c_int, ctypes.c_uint32, vp]
        L.sgmv_shrink_strided.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, i32, i32,
                                          ctypes.c_int, ctypes.c_uint32, vp]
        L.sgmv_expand_strided.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, f32,
                                          ctypes.c_int, ctypes.c_uint32, vp]
        L.sgmv_validate.argtypes = [vp, vp, i32, i32, i32, vp, vp]
        L.sgmv_validate_pointers.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp]
        u32, ci = ctypes.c_uint32, ctypes.c_int
        L.sgmv_plan_size.argtypes = [i32, i32]
        L.sgmv_plan_size.restype = ctypes.c_size_t
        L.sgmv_plan.argtypes = [vp, vp, i32, i32, vp, ctypes.c_size_t, vp]
        L.lora_apply_planned.argtypes = [vp, i32, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32,
                                         f32, ci, u32, vp]
        L.sgmv_shrink_planned.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, i32, ci, u32, vp]
        L.sgmv_expand_planned.argtypes = [vp, i32, vp, vp, vp, i32, i32, i32, i32, f32, ci, u32,
                                          vp]
        L.lora_apply_multi.argtypes = [ctypes.POINTER(Projection), i32, vp, i32, i32, i32, ci,
                                       u32, vp]
        L.lora_apply_ranked.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                        i32, i32, i32, ci, u32, vp]
        L.sgmv_pool_slot_bytes.argtypes = [i32, i32, i32, i32, ci]
        L.sgmv_pool_slot_bytes.restype = ctypes.c_size_t
        L.sgmv_pool_create.argtypes = [ctypes.POINTER(vp), vp, ctypes.c_size_t, i32, i32, i32,
                                       i32, i32, i32, ci]
        L.sgmv_pool_destroy.argtypes = [vp]
        L.sgmv_pool_register.argtypes = [vp, i32, vp, vp]
        L.sgmv_pool_acquire.argtypes = [vp, vp, i32, vp, vp, vp, vp, ctypes.POINTER(i32)]
        L.sgmv_pool_release.argtypes = [vp, vp, i32, vp]
        L.sgmv_pool_stats.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64),
                                      ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(i32)]
        L.lora_apply_base.argtypes = [vp, i32, vp, i32, i32, vp, i32, vp, vp, vp, vp, i32, i32,
                                      i32, i32, i32, f32, vp, ci, u32, vp]
        L.lora_apply_static_plan.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, i32, i32, i32,
                                             i32, i32, i32, f32, ci, u32, vp]
        L.sgmv_get_error.argtypes = [ctypes.POINTER(ctypes.c_int32), i32, vp]
        L.sgmv_set_wait_limit.argtypes = [ctypes.c_uint64, i32]
        L.sgmv_status_string.argtypes = [ctypes.c_int]
        L.sgmv_status_string.restype = ctypes.c_char_p
        L.sgmv_version.argtypes = []
        for name in SYMBOLS:
            if name not in ("sgmv_status_string", "sgmv_plan_size", "sgmv_pool_slot_bytes"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().sgmv_status_string(int(status)).decode()


def _dtype_code(t) -> int:
    import torch
    codes = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _cuda(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _rows(t, name):
    """A CUDA matrix whose rows may be apart by more than their length (a column slice of a
    wider tensor): returns the row stride in elements."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1) or t.stride(0) < t.shape[1]:
        raise ValueError(f"{name} must be a 2-D matrix with unit column stride")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


def _stream(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _on(t, *others):
    """The library plans a launch for the CURRENT device: make the tensors' device current
    (every tensor of the call must live on it)."""
    import torch
    for o in others:
        if o is not None and o.device != t.device:
            raise ValueError(f"all tensors of a call must be on one device ({t.device}, not "
                             f"{o.device})")
    return torch.cuda.device(t.device)


def _table(seg_starts, seg_adapter):
    import torch
    _cuda(seg_starts, "seg_starts")
    _cuda(seg_adapter, "seg_adapter")
    if seg_starts.dtype != torch.int32 or seg_adapter.dtype != torch.int32:
        raise TypeError("seg_starts and seg_adapter must be int32")
    S = seg_adapter.numel()
    if seg_starts.numel() != S + 1:
        raise ValueError("seg_starts must hold num_segments + 1 offsets")
    return S


def _ptrs(t, name):
    import torch
    _cuda(t, name)
    if t.dtype != torch.int64:
        raise TypeError(f"{name} must be an int64 tensor of device addresses")
    return t.data_ptr()


def _flags(overlap_prior, tensor_cores, long_batch=False, dense_grid=False) -> int:
    mode = {True: "auto", False: "never"}.get(tensor_cores, tensor_cores)
    if mode not in ("auto", "never", "always"):
        raise ValueError(f"tensor_cores must be 'auto', 'never' or 'always', not {tensor_cores!r}")
    return ((SGMV_OVERLAP_PRIOR if overlap_prior else 0) | (SGMV_LONG_BATCH if long_batch else 0) |
            (SGMV_DENSE_GRID if dense_grid else 0) |
            {"auto": 0, "never": SGMV_NO_TENSOR_CORES, "always": SGMV_TENSOR_CORES_ALWAYS}[mode])


def _check(rc: int, where: str):
    if rc != SGMV_OK:
        raise SgmvError(rc, where)


def lora_apply(y, x, A_ptrs, B_ptrs, seg_starts, seg_adapter, layer_idx, r, scale, stream=None,
               overlap_prior=False, tensor_cores="auto", long_batch=False, dense_grid=False):
    """y[t] += scale * (x[t] A_k) B_k for every segment row (in place on y).

    overlap_prior=True calls lora_apply_ex with SGMV_OVERLAP_PRIOR: the kernel may stream
    weights while the previous kernel on the stream is still running (see include/sgmv.h).
    tensor_cores: "auto" (the library's cost rule), "never" (SGMV_NO_TENSOR_CORES) or "always"
    (SGMV_TENSOR_CORES_ALWAYS); True / False mean "auto" / "never".
    long_batch=True adds SGMV_LONG_BATCH: one CTA per SM with the whole shared memory, for
    prefill-sized calls (see include/sgmv.h).  dense_grid=True adds SGMV_DENSE_GRID: two CTAs
    of the call per SM, for decode batches with many work items (see include/sgmv.h).
    x and y may be column slices of wider matrices (unit column stride, row stride a multiple
    of 8 elements): they then go through lora_apply_strided.
    """
    ldy, ldx = _rows(y, "y"), _rows(x, "x")
    if x.dtype != y.dtype or x.shape[0] != y.shape[0]:
        raise ValueError("x [M, h_in] and y [M, h_out] must share M and dtype")
    S = _table(seg_starts, seg_adapter)
    flags = _flags(overlap_prior, tensor_cores, long_batch, dense_grid)
    with _on(x, y, A_ptrs, B_ptrs, seg_starts, seg_adapter):
        return _lora_apply(y, x, A_ptrs, B_ptrs, seg_starts, seg_adapter, layer_idx, r, scale,
                           stream, flags, ldx, ldy, S)


def _lora_apply(y, x, A_ptrs, B_ptrs, seg_starts, seg_adapter, layer_idx, r, scale, stream,
                flags, ldx, ldy, S):
    if ldx != x.shape[1] or ldy != y.shape[1]:  # column slices of wider activations
        rc = lib().lora_apply_strided(
            y.data_ptr(), ldy, x.data_ptr(), ldx, _ptrs(A_ptrs, "A_ptrs"), _ptrs(B_ptrs, "B_ptrs"),
            seg_starts.data_ptr(), seg_adapter.data_ptr(), S, int(layer_idx), x.shape[1],
            y.shape[1], int(r), float(scale), _dtype_code(x), flags, _stream(stream, x.device))
        _check(rc, "lora_apply_strided")
        return y
    args = (y.data_ptr(), x.data_ptr(), _ptrs(A_ptrs, "A_ptrs"), _ptrs(B_ptrs, "B_ptrs"),
            seg_starts.data_ptr(), seg_adapter.data_ptr(), S, int(layer_idx), x.shape[1],
            y.shape[1], int(r), float(scale), _dtype_code(x))
    if flags:
        rc = lib().lora_apply_ex(*args, flags, _stream(stream, x.device))
        _check(rc, "lora_apply_ex")
    else:
        rc = lib().lora_apply(*args, _stream(stream, x.device))
        _check(rc, "lora_apply")
    return y


def sgmv_shrink(v, x, A_ptrs, seg_starts, seg_adapter, layer_idx, r, stream=None,
                tensor_cores="auto", long_batch=False, overlap_prior=False, dense_grid=False):
    """v[t] = x[t] A_k (fp32) for every segment row (tensor_cores, long_batch, overlap_prior as
    for lora_apply)."""
    import torch
    _cuda(v, "v")
    ldx = _rows(x, "x")
    if v.dtype != torch.float32 or v.dim() != 2 or v.shape[1] != r or v.shape[0] != x.shape[0]:
        raise ValueError("v must be float32 [M, r]")
    S = _table(seg_starts, seg_adapter)
    flags = _flags(overlap_prior, tensor_cores, long_batch, dense_grid)
    with _on(x, v, A_ptrs, seg_starts, seg_adapter):
        return _sgmv_shrink(v, x, A_ptrs, seg_starts, seg_adapter, layer_idx, r, stream, flags,
                            ldx, S)


def _sgmv_shrink(v, x, A_ptrs, seg_starts, seg_adapter, layer_idx, r, stream, flags, ldx, S):
    if ldx != x.shape[1]:
        _check(lib().sgmv_shrink_strided(
            v.data_ptr(), x.data_ptr(), ldx, _ptrs(A_ptrs, "A_ptrs"), seg_starts.data_ptr(),
            seg_adapter.data_ptr(), S, int(layer_idx), x.shape[1], int(r), _dtype_code(x), flags,
            _stream(stream, x.device)), "sgmv_shrink_strided")
        return v
    args = (v.data_ptr(), x.data_ptr(), _ptrs(A_ptrs, "A_ptrs"), seg_starts.data_ptr(),
            seg_adapter.data_ptr(), S, int(layer_idx), x.shape[1], int(r), _dtype_code(x))
    if flags:
        _check(lib().sgmv_shrink_ex(*args, flags, _stream(stream, x.device)), "sgmv_shrink_ex")
    else:
        _check(lib().sgmv_shrink(*args, _stream(stream, x.device)), "sgmv_shrink")
    return v


def sgmv_expand(y, v, B_ptrs, seg_starts, seg_adapter, layer_idx, r, scale, stream=None,
                tensor_cores="auto", long_batch=False, overlap_prior=False, dense_grid=False):
    """y[t] += scale * v[t] B_k for every segment row (in place on y; tensor_cores, long_batch,
    overlap_prior as for lora_apply)."""
    import torch
    _cuda(v, "v")
    ldy = _rows(y, "y")
    if v.dtype != torch.float32 or v.dim() != 2 or v.shape[1] != r or v.shape[0] != y.shape[0]:
        raise ValueError("v must be float32 [M, r]")
    S = _table(seg_starts, seg_adapter)
    flags = _flags(overlap_prior, tensor_cores, long_batch, dense_grid)
    with _on(y, v, B_ptrs, seg_starts, seg_adapter):
        return _sgmv_expand(y, v, B_ptrs, seg_starts, seg_adapter, layer_idx, r, scale, stream,
                            flags, ldy, S)


def _sgmv_expand(y, v, B_ptrs, seg_starts, seg_adapter, layer_idx, r, scale, stream, flags, ldy,
                 S):
    if ldy != y.shape[1]:
        _check(lib().sgmv_expand_strided(
            y.data_ptr(), ldy, v.data_ptr(), _ptrs(B_ptrs, "B_ptrs"), seg_starts.data_ptr(),
            seg_adapter.data_ptr(), S, int(layer_idx), int(r), y.shape[1], float(scale),
            _dtype_code(y), flags, _stream(stream, y.device)), "sgmv_expand_strided")
        return y
    args = (y.data_ptr(), v.data_ptr(), _ptrs(B_ptrs, "B_ptrs"), seg_starts.data_ptr(),
            seg_adapter.data_ptr(), S, int(layer_idx), int(r), y.shape[1], float(scale),
            _dtype_code(y))
    if flags:
        _check(lib().sgmv_expand_ex(*args, flags, _stream(stream, y.device)), "sgmv_expand_ex")
    else:
        _check(lib().sgmv_expand(*args, _stream(stream, y.device)), "sgmv_expand")
    return y


def sgmv_validate(seg_starts, seg_adapter, num_adapters, M, d_err, stream=None):
    """Writes the table-check bits into the device int32 tensor d_err (see include/sgmv.h)."""
    import torch
    S = _table(seg_starts, seg_adapter)
    _cuda(d_err, "d_err")
    if d_err.dtype != torch.int32 or d_err.numel() < 1:
        raise TypeError("d_err must be a device int32 tensor")
    with _on(seg_starts, seg_adapter, d_err):
        rc = lib().sgmv_validate(seg_starts.data_ptr(), seg_adapter.data_ptr(), S,
                                 int(num_adapters), int(M), d_err.data_ptr(),
                                 _stream(stream, seg_starts.device))
    _check(rc, "sgmv_validate")
    return d_err


def sgmv_validate_pointers(A_ptrs, B_ptrs, seg_starts, seg_adapter, d_err, stream=None):
    """Writes the pointer-check bits (16: a used A pointer is null or misaligned, 32: the same
    for B) into the device int32 tensor d_err.  A_ptrs / B_ptrs: int64 device tensors of
    addresses (one may be None); reads pointer values only (see include/sgmv.h)."""
    import torch
    S = _table(seg_starts, seg_adapter)
    _cuda(d_err, "d_err")
    if d_err.dtype != torch.int32 or d_err.numel() < 1:
        raise TypeError("d_err must be a device int32 tensor")
    tabs = [t for t in (A_ptrs, B_ptrs) if t is not None]
    if not tabs:
        raise ValueError("A_ptrs and B_ptrs cannot both be None")
    n = tabs[0].numel()
    if any(t.numel() != n for t in tabs):
        raise ValueError("A_ptrs and B_ptrs must have one entry per adapter")
    a = _ptrs(A_ptrs, "A_ptrs") if A_ptrs is not None else None
    b = _ptrs(B_ptrs, "B_ptrs") if B_ptrs is not None else None
    with _on(seg_starts, seg_adapter, d_err, A_ptrs, B_ptrs):
        rc = lib().sgmv_validate_pointers(a, b, seg_starts.data_ptr(), seg_adapter.data_ptr(), S,
                                          n, d_err.data_ptr(), _stream(stream, seg_starts.device))
    _check(rc, "sgmv_validate_pointers")
    return d_err


def sgmv_get_error(clear: bool = True, stream=None, device=None) -> int:
    """Synchronises and returns the library's device error word (0 or SGMV_ETIMEOUT)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    out = ctypes.c_int32(0)
    _check(lib().sgmv_get_error(ctypes.byref(out), 1 if clear else 0, _stream(stream, dev)),
           "sgmv_get_error")
    return int(out.value)


def sgmv_set_wait_limit(limit_ns: int, inject_stall: bool = False):
    """Bound of every device-side wait (0: default 2 s); inject_stall forces one to run out."""
    _check(lib().sgmv_set_wait_limit(int(limit_ns), 1 if inject_stall else 0),
           "sgmv_set_wait_limit")


def sgmv_version() -> int:
    return int(lib().sgmv_version())


# ---------------------------------------------------------------------------- plans ----
class Plan:
    """A device plan (sgmv_plan): the segment table grouped by adapter once, for reuse by
    every planned call of the batch.  `buf` is the caller-side device allocation (torch int32);
    num_segments is the plan's capacity, which every planned call passes back."""

    def __init__(self, buf, num_segments, max_rows):
        self.buf = buf
        self.num_segments = int(num_segments)
        self.max_rows = int(max_rows)

    @property
    def device(self):
        return self.buf.device

    def groups(self):
        """(g_starts, g_adapter, rows) as host numpy arrays, or None for an invalid plan
        (synchronises)."""
        import numpy as np
        h = self.buf.cpu().numpy()
        S = self.num_segments
        if int(h[1]) != 0:
            return None
        G, n = int(h[3]), int(h[4])
        gs = h[PLAN_HEADER:PLAN_HEADER + G + 1].astype(np.int32)
        ga = h[PLAN_HEADER + S + 1:PLAN_HEADER + S + 1 + G].astype(np.int32)
        rows = h[PLAN_HEADER + 2 * S + 1:PLAN_HEADER + 2 * S + 1 + n].astype(np.int32)
        return gs, ga, rows


def sgmv_plan_size(num_segments, max_rows) -> int:
    return int(lib().sgmv_plan_size(int(num_segments), int(max_rows)))


def sgmv_plan(seg_starts, seg_adapter, max_rows, stream=None, out=None) -> Plan:
    """Groups the device segment table by adapter into a plan (a torch int32 device buffer the
    binding allocates unless `out` is given); max_rows: capacity of the row list (>= the rows
    with an adapter, e.g. M)."""
    import torch
    S = _table(seg_starts, seg_adapter)
    nbytes = sgmv_plan_size(S, max_rows)
    if nbytes == 0:
        raise ValueError("bad plan size arguments")
    if out is None:
        out = torch.empty((nbytes + 3) // 4, dtype=torch.int32, device=seg_starts.device)
    _cuda(out, "out")
    with _on(seg_starts, seg_adapter, out):
        rc = lib().sgmv_plan(seg_starts.data_ptr(), seg_adapter.data_ptr(), S, int(max_rows),
                             out.data_ptr(), out.numel() * out.element_size(),
                             _stream(stream, seg_starts.device))
    _check(rc, "sgmv_plan")
    return Plan(out, S, max_rows)


def lora_apply_planned(y, x, A_ptrs, B_ptrs, plan: Plan, layer_idx, r, scale, stream=None,
                       overlap_prior=False, tensor_cores="auto", long_batch=False, dense_grid=False):
    """lora_apply with a plan instead of the segment table (x, y may be column slices)."""
    ldy, ldx = _rows(y, "y"), _rows(x, "x")
    if x.dtype != y.dtype or x.shape[0] != y.shape[0]:
        raise ValueError("x [M, h_in] and y [M, h_out] must share M and dtype")
    flags = _flags(overlap_prior, tensor_cores, long_batch, dense_grid)
    with _on(x, y, A_ptrs, B_ptrs, plan.buf):
        rc = lib().lora_apply_planned(
            y.data_ptr(), ldy, x.data_ptr(), ldx, _ptrs(A_ptrs, "A_ptrs"), _ptrs(B_ptrs, "B_ptrs"),
            plan.buf.data_ptr(), plan.num_segments, int(layer_idx), x.shape[1], y.shape[1],
            int(r), float(scale), _dtype_code(x), flags, _stream(stream, x.device))
    _check(rc, "lora_apply_planned")
    return y


def lora_apply_static_plan(y, x, A_ptrs, B_ptrs, seg_starts, seg_adapter, max_rows, layer_idx, r,
                           scale, stream=None, tensor_cores="auto", long_batch=False, dense_grid=False):
    """lora_apply_planned with the plan built inside the library's fixed device array: the call
    allocates no device memory (for callers that may not).  Calls that overlap on the GPU
    share that array and must be ordered; overlap_prior is not available here."""
    ldy, ldx = _rows(y, "y"), _rows(x, "x")
    if x.dtype != y.dtype or x.shape[0] != y.shape[0]:
        raise ValueError("x [M, h_in] and y [M, h_out] must share M and dtype")
    S = _table(seg_starts, seg_adapter)
    flags = _flags(False, tensor_cores, long_batch, dense_grid)
    with _on(x, y, A_ptrs, B_ptrs, seg_starts, seg_adapter):
        rc = lib().lora_apply_static_plan(
            y.data_ptr(), ldy, x.data_ptr(), ldx, _ptrs(A_ptrs, "A_ptrs"), _ptrs(B_ptrs, "B_ptrs"),
            seg_starts.data_ptr(), seg_adapter.data_ptr(), S, int(max_rows), int(layer_idx),
            x.shape[1], y.shape[1], int(r), float(scale), _dtype_code(x), flags,
            _stream(stream, x.device))
    _check(rc, "lora_apply_static_plan")
    return y


def lora_apply_base(y, x, W0, A_ptrs, B_ptrs, seg_starts, seg_adapter, layer_idx, r, scale,
                    v_work=None, stream=None, overlap_prior=False, tensor_cores="auto",
                    long_batch=False, dense_grid=False):
    """y = x W0^T + scale * (x A_k) B_k per segment row (x W0^T alone on other rows), written
    into y (fp16 / bf16).  W0 is [h_out, h_in] (a linear layer's weight).  v_work: fp32
    [M, r] workspace (made here with torch when not given).  Flags as for lora_apply; they
    apply to the shrink."""
    import torch
    ldy, ldx = _rows(y, "y"), _rows(x, "x")
    ldw = _rows(W0, "W0")
    if x.dtype != y.dtype or W0.dtype != x.dtype or x.shape[0] != y.shape[0]:
        raise ValueError("x [M, h_in], W0 [h_out, h_in] and y [M, h_out] share a dtype and M")
    if W0.shape[0] != y.shape[1] or W0.shape[1] != x.shape[1]:
        raise ValueError("W0 must be [h_out, h_in]")
    S = _table(seg_starts, seg_adapter)
    M = x.shape[0]
    if v_work is None and S > 0:
        v_work = torch.empty((M, int(r)), dtype=torch.float32, device=x.device)
    if v_work is not None:
        _cuda(v_work, "v_work")
        if v_work.dtype != torch.float32 or v_work.numel() < M * int(r):
            raise ValueError("v_work must hold M * r fp32 values")
    flags = _flags(overlap_prior, tensor_cores, long_batch, dense_grid)
    with _on(x, y, W0, seg_starts, seg_adapter):
        rc = lib().lora_apply_base(
            y.data_ptr(), ldy, x.data_ptr(), ldx, M, W0.data_ptr(), ldw,
            _ptrs(A_ptrs, "A_ptrs") if S else None, _ptrs(B_ptrs, "B_ptrs") if S else None,
            seg_starts.data_ptr(), seg_adapter.data_ptr(), S, int(layer_idx), x.shape[1],
            y.shape[1], int(r), float(scale), v_work.data_ptr() if v_work is not None else None,
            _dtype_code(x), flags, _stream(stream, x.device))
    _check(rc, "lora_apply_base")
    return y


def sgmv_shrink_planned(v, x, A_ptrs, plan: Plan, layer_idx, r, stream=None,
                        tensor_cores="auto", long_batch=False, overlap_prior=False, dense_grid=False):
    import torch
    _cuda(v, "v")
    ldx = _rows(x, "x")
    if v.dtype != torch.float32 or v.dim() != 2 or v.shape[1] != r or v.shape[0] != x.shape[0]:
        raise ValueError("v must be float32 [M, r]")
    flags = _flags(overlap_prior, tensor_cores, long_batch, dense_grid)
    with _on(x, v, A_ptrs, plan.buf):
        rc = lib().sgmv_shrink_planned(v.data_ptr(), x.data_ptr(), ldx, _ptrs(A_ptrs, "A_ptrs"),
                                       plan.buf.data_ptr(), plan.num_segments, int(layer_idx),
                                       x.shape[1], int(r), _dtype_code(x), flags,
                                       _stream(stream, x.device))
    _check(rc, "sgmv_shrink_planned")
    return v


def sgmv_expand_planned(y, v, B_ptrs, plan: Plan, layer_idx, r, scale, stream=None,
                        tensor_cores="auto", long_batch=False, overlap_prior=False, dense_grid=False):
    import torch
    _cuda(v, "v")
    ldy = _rows(y, "y")
    if v.dtype != torch.float32 or v.dim() != 2 or v.shape[1] != r or v.shape[0] != y.shape[0]:
        raise ValueError("v must be float32 [M, r]")
    flags = _flags(overlap_prior, tensor_cores, long_batch, dense_grid)
    with _on(y, v, B_ptrs, plan.buf):
        rc = lib().sgmv_expand_planned(y.data_ptr(), ldy, v.data_ptr(), _ptrs(B_ptrs, "B_ptrs"),
                                       plan.buf.data_ptr(), plan.num_segments, int(layer_idx),
                                       int(r), y.shape[1], float(scale), _dtype_code(y), flags,
                                       _stream(stream, y.device))
    _check(rc, "sgmv_expand_planned")
    return y


def lora_apply_multi(projections, plan: Plan, layer_idx, r, stream=None, overlap_prior=False,
                     tensor_cores="auto", long_batch=False, dense_grid=False):
    """One launch over several projections: projections is a list of
    (y, x, A_ptrs, B_ptrs, scale) tuples sharing the plan, layer, rank and dtype."""
    if not 1 <= len(projections) <= SGMV_MAX_PROJECTIONS:
        raise ValueError(f"1 to {SGMV_MAX_PROJECTIONS} projections")
    arr = (Projection * len(projections))()
    dt = None
    tensors = []
    for q, (y, x, A_ptrs, B_ptrs, scale) in enumerate(projections):
        ldy, ldx = _rows(y, "y"), _rows(x, "x")
        if x.dtype != y.dtype or x.shape[0] != y.shape[0]:
            raise ValueError("x [M, h_in] and y [M, h_out] must share M and dtype")
        if dt is not None and x.dtype != dt:
            raise ValueError("all projections share one dtype")
        dt = x.dtype
        arr[q] = Projection(y.data_ptr(), x.data_ptr(), _ptrs(A_ptrs, "A_ptrs"),
                            _ptrs(B_ptrs, "B_ptrs"), ldy, ldx, x.shape[1], y.shape[1],
                            float(scale), 0)
        tensors += [y, x, A_ptrs, B_ptrs]
    x0 = projections[0][1]
    flags = _flags(overlap_prior, tensor_cores, long_batch, dense_grid)
    with _on(x0, plan.buf, *tensors):
        rc = lib().lora_apply_multi(arr, len(projections), plan.buf.data_ptr(), plan.num_segments,
                                    int(layer_idx), int(r), _dtype_code(x0), flags,
                                    _stream(stream, x0.device))
    _check(rc, "lora_apply_multi")


def lora_apply_ranked(y, x, A_ptrs, B_ptrs, adapter_rank, adapter_scale, layer_idx, r_max,
                      seg_starts=None, seg_adapter=None, plan: Plan = None, stream=None,
                      overlap_prior=False, tensor_cores="auto", long_batch=False, dense_grid=False):
    """y[t] += adapter_scale[k] (x[t] A_k) B_k with adapter k of rank adapter_rank[k] (device
    int32 and float32 tensors, one entry per adapter); the table, or a plan."""
    import torch
    ldy, ldx = _rows(y, "y"), _rows(x, "x")
    if x.dtype != y.dtype or x.shape[0] != y.shape[0]:
        raise ValueError("x [M, h_in] and y [M, h_out] must share M and dtype")
    _cuda(adapter_rank, "adapter_rank")
    _cuda(adapter_scale, "adapter_scale")
    if adapter_rank.dtype != torch.int32 or adapter_scale.dtype != torch.float32:
        raise TypeError("adapter_rank must be int32 and adapter_scale float32")
    if (plan is None) == (seg_starts is None):
        raise ValueError("pass either the segment table or a plan")
    if plan is None:
        S = _table(seg_starts, seg_adapter)
        ss, sa, pl = seg_starts.data_ptr(), seg_adapter.data_ptr(), None
        extra = (seg_starts, seg_adapter)
    else:
        S, ss, sa, pl = plan.num_segments, None, None, plan.buf.data_ptr()
        extra = (plan.buf,)
    flags = _flags(overlap_prior, tensor_cores, long_batch, dense_grid)
    with _on(x, y, A_ptrs, B_ptrs, adapter_rank, adapter_scale, *extra):
        rc = lib().lora_apply_ranked(
            y.data_ptr(), ldy, x.data_ptr(), ldx, _ptrs(A_ptrs, "A_ptrs"), _ptrs(B_ptrs, "B_ptrs"),
            adapter_rank.data_ptr(), adapter_scale.data_ptr(), ss, sa, pl, S, int(layer_idx),
            x.shape[1], y.shape[1], int(r_max), _dtype_code(x), flags, _stream(stream, x.device))
    _check(rc, "lora_apply_ranked")
    return y


# ----------------------------------------------------------------------- adapter pool ----
class AdapterPool:
    """sgmv_pool_*: `slots` device slots (one adapter's A and B blocks each) in a device slab the
    binding allocates with torch, filled on demand from registered host copies (pinned CPU
    tensors).  acquire() returns how many adapters it copied; the device pointer tables it
    writes (A_ptrs / B_ptrs, int64 [num_adapters]) are what lora_apply takes."""

    def __init__(self, slots, num_adapters, layers, h_in, h_out, r, dtype, device=None):
        import torch
        device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.code = _dtype_code(torch.empty(0, dtype=dtype))
        self.slot_bytes = int(lib().sgmv_pool_slot_bytes(layers, h_in, h_out, r, self.code))
        if self.slot_bytes == 0:
            raise ValueError("bad pool shape")
        self.slab = torch.empty(slots * self.slot_bytes + 256, dtype=torch.uint8, device=device)
        off = (-self.slab.data_ptr()) % 256
        self.num_adapters = int(num_adapters)
        self.A_ptrs = torch.zeros(num_adapters, dtype=torch.int64, device=device)
        self.B_ptrs = torch.zeros(num_adapters, dtype=torch.int64, device=device)
        self._keep = {}
        self.handle = ctypes.c_void_p()
        with torch.cuda.device(device):
            _check(lib().sgmv_pool_create(ctypes.byref(self.handle), self.slab.data_ptr() + off,
                                          slots * self.slot_bytes, int(slots), int(num_adapters),
                                          int(layers), int(h_in), int(h_out), int(r), self.code),
                   "sgmv_pool_create")
        self.device = device

    def register(self, adapter, host_A, host_B):
        for t in (host_A, host_B):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("host copies must be contiguous CPU tensors (pinned: async)")
        _check(lib().sgmv_pool_register(self.handle, int(adapter), host_A.data_ptr(),
                                        host_B.data_ptr()), "sgmv_pool_register")
        self._keep[int(adapter)] = (host_A, host_B)

    def _ids(self, ids):
        import numpy as np
        arr = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        return arr, arr.ctypes.data

    def acquire(self, ids, copy_stream, compute_stream) -> int:
        arr, ptr = self._ids(ids)
        copied = ctypes.c_int32(0)
        with torch_device(self.device):
            _check(lib().sgmv_pool_acquire(self.handle, ptr, len(arr), self.A_ptrs.data_ptr(),
                                           self.B_ptrs.data_ptr(),
                                           ctypes.c_void_p(copy_stream.cuda_stream),
                                           ctypes.c_void_p(compute_stream.cuda_stream),
                                           ctypes.byref(copied)), "sgmv_pool_acquire")
        return int(copied.value)

    def release(self, ids, compute_stream):
        arr, ptr = self._ids(ids)
        with torch_device(self.device):
            _check(lib().sgmv_pool_release(self.handle, ptr, len(arr),
                                           ctypes.c_void_p(compute_stream.cuda_stream)),
                   "sgmv_pool_release")

    def stats(self):
        h, m, r = ctypes.c_uint64(0), ctypes.c_uint64(0), ctypes.c_int32(0)
        _check(lib().sgmv_pool_stats(self.handle, ctypes.byref(h), ctypes.byref(m),
                                     ctypes.byref(r)), "sgmv_pool_stats")
        return {"hits": int(h.value), "misses": int(m.value), "resident": int(r.value)}

    def close(self):
        if self.handle:
            with torch_device(self.device):
                lib().sgmv_pool_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def torch_device(device):
    import torch
    return torch.cuda.device(device)
