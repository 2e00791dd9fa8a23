"""The C-ABI library without a GPU: it builds, loads, exports every entry point that
include/sgmv.h declares, and its host-side argument checks return the documented statuses
before any CUDA call."""
import ctypes
import os
import re

import pytest

from segmented_gather_gemm_sgmv_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sgmv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char \*)\s*\**\s*(\w+)\s*\(", text,
                                 flags=re.M)))


@pytest.fixture(scope="module")
def L():
    return binding.lib()


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert set(binding.SYMBOLS) <= set(names), names
    for name in names:
        assert hasattr(L, name), f"{name} declared in sgmv.h but not exported"


def test_header_constants_match_binding():
    text = open(HEADER).read()
    assert f"#define SGMV_MAX_SEGMENTS {binding.SGMV_MAX_SEGMENTS}" in text
    assert f"#define SGMV_MAX_HIDDEN {binding.SGMV_MAX_HIDDEN}" in text
    assert f"#define SGMV_OVERLAP_PRIOR {binding.SGMV_OVERLAP_PRIOR}u" in text
    assert f"#define SGMV_NO_TENSOR_CORES {binding.SGMV_NO_TENSOR_CORES}u" in text
    assert f"#define SGMV_TENSOR_CORES_ALWAYS {binding.SGMV_TENSOR_CORES_ALWAYS}u" in text
    assert f"#define SGMV_LONG_BATCH {binding.SGMV_LONG_BATCH}u" in text
    assert f"#define SGMV_DENSE_GRID {binding.SGMV_DENSE_GRID}u" in text
    assert "#define SGMV_MAX_LD (1 << 24)" in text and binding.SGMV_MAX_LD == 1 << 24
    assert f"#define SGMV_MAX_PROJECTIONS {binding.SGMV_MAX_PROJECTIONS}" in text
    assert f"#define SGMV_STATIC_PLAN_MAX_ROWS {binding.SGMV_STATIC_PLAN_MAX_ROWS}" in text
    for name, val in [("SGMV_EINVAL", -1), ("SGMV_EALIGN", -2), ("SGMV_EUNSUPPORTED", -3),
                      ("SGMV_ECUDA", -4), ("SGMV_ETIMEOUT", -5), ("SGMV_EPLAN", -6),
                      ("SGMV_ENOSPACE", -7), ("SGMV_EBUSY", -8)]:
        assert re.search(rf"{name}\s*=\s*{val}\b", text), name


def test_version_and_strings(L):
    assert L.sgmv_version() == 200
    for s in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert binding.status_string(s).startswith("SGMV_")


# Fake but aligned device addresses: the host checks never dereference them.
P = 0x7F0000000000
OK_ARGS = dict(y=P, x=P + 0x10000, A=P + 0x20000, B=P + 0x30000, ss=P + 0x40000, sa=P + 0x50000,
               S=4, layer=0, h_in=4096, h_out=4096, r=16, scale=1.0, dt=1)


def apply(L, **kw):
    a = dict(OK_ARGS, **kw)
    return L.lora_apply(a["y"], a["x"], a["A"], a["B"], a["ss"], a["sa"], a["S"], a["layer"],
                        a["h_in"], a["h_out"], a["r"], a["scale"], a["dt"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(y=None), -1), (dict(x=None), -1), (dict(A=None), -1), (dict(ss=None), -1),
    (dict(S=-1), -1), (dict(layer=-2), -1), (dict(dt=7), -1), (dict(h_in=0), -1),
    (dict(y=P + 8), -2), (dict(x=P + 0x10004), -2), (dict(h_in=4100), -2), (dict(h_out=12), -2),
    (dict(ss=P + 0x40002), -2),
    (dict(r=12), -3), (dict(r=128), -3), (dict(S=4097), -3), (dict(h_out=65544), -3),
    (dict(S=0), 0), (dict(S=0, sa=None), 0), (dict(S=1, sa=None), -1),
])
def test_lora_apply_host_checks(L, kw, status):
    assert apply(L, **kw) == status


def test_lora_apply_ex_flags(L):
    a = OK_ARGS
    args = (a["y"], a["x"], a["A"], a["B"], a["ss"], a["sa"], 0, a["layer"], a["h_in"],
            a["h_out"], a["r"], a["scale"], a["dt"])
    for flags in (0, 1, 2, 3, 4, 5, 8, 9, 10, 13, 16, 17, 25):  # num_segments = 0: no launch
        assert L.lora_apply_ex(*args, flags, None) == 0
    assert L.lora_apply_ex(*args, 6, None) == -1  # never + always
    assert L.lora_apply_ex(*args, 14, None) == -1
    assert L.lora_apply_ex(*args, 32, None) == -1  # unknown bit


def test_strided_host_checks(L):
    """Row strides: below the row length -> EINVAL, not a multiple of 8 -> EALIGN, above
    SGMV_MAX_LD -> EUNSUPPORTED; valid strides with num_segments = 0 -> OK (no launch)."""
    a = OK_ARGS
    h_in, h_out = a["h_in"], a["h_out"]

    def fused(ldy, ldx, S=0):
        return L.lora_apply_strided(a["y"], ldy, a["x"], ldx, a["A"], a["B"], a["ss"], a["sa"], S,
                                    a["layer"], h_in, h_out, a["r"], a["scale"], a["dt"], 0, None)
    assert fused(h_out, h_in) == 0
    assert fused(h_out + 64, h_in + 8) == 0
    assert fused(h_out - 8, h_in, S=4) == -1
    assert fused(h_out, h_in - 8, S=4) == -1
    assert fused(h_out + 4, h_in, S=4) == -2
    assert fused(h_out, h_in + 12, S=4) == -2
    assert fused(h_out, (1 << 24) + 8, S=4) == -3
    assert L.sgmv_shrink_strided(a["y"], a["x"], h_in - 8, a["A"], a["ss"], a["sa"], 4, 0, h_in,
                                 16, 1, 0, None) == -1
    assert L.sgmv_shrink_strided(a["y"], a["x"], h_in + 8, a["A"], a["ss"], a["sa"], 0, 0, h_in,
                                 16, 1, 0, None) == 0
    assert L.sgmv_expand_strided(a["y"], h_out + 2, a["x"], a["B"], a["ss"], a["sa"], 4, 0, 16,
                                 h_out, 1.0, 1, 0, None) == -2
    assert L.sgmv_expand_strided(a["y"], h_out + 8, a["x"], a["B"], a["ss"], a["sa"], 0, 0, 16,
                                 h_out, 1.0, 1, 0, None) == 0


def test_shrink_expand_validate_host_checks(L):
    a = OK_ARGS
    assert L.sgmv_shrink(None, a["x"], a["A"], a["ss"], a["sa"], 4, 0, 4096, 16, 1, None) == -1
    assert L.sgmv_shrink(a["y"], a["x"], a["A"], a["ss"], a["sa"], 4, 0, 4096, 24, 1, None) == -3
    assert L.sgmv_shrink(a["y"], a["x"], a["A"], a["ss"], a["sa"], 0, 0, 4096, 16, 1, None) == 0
    assert L.sgmv_expand(a["y"], None, a["B"], a["ss"], a["sa"], 4, 0, 16, 4096, 1.0, 1,
                         None) == -1
    assert L.sgmv_expand(a["y"], a["x"], a["B"], a["ss"], a["sa"], 4, 0, 16, 4090, 1.0, 1,
                         None) == -2
    assert L.sgmv_validate(None, a["sa"], 4, 8, 10, a["y"], None) == -1
    assert L.sgmv_validate(a["ss"], a["sa"], -1, 8, 10, a["y"], None) == -1
    assert L.sgmv_get_error(None, 0, None) == -1


def test_python_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    y = torch.zeros(2, 8, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA"):
        lora_apply(y, y, torch.zeros(1, dtype=torch.int64), torch.zeros(1, dtype=torch.int64),
                   torch.zeros(2, dtype=torch.int32), torch.zeros(1, dtype=torch.int32), 0, 16,
                   1.0)


class _FakeMatrix:
    """Stands in for a CUDA tensor in the binding's shape / stride checks (no device needed)."""

    def __init__(self, shape, stride, is_cuda=True):
        self.shape, self._stride, self.is_cuda = shape, stride, is_cuda

    def dim(self):
        return len(self.shape)

    def stride(self, i):
        return self._stride[i]


@pytest.mark.parametrize("shape,stride,ld", [
    ((5, 64), (64, 1), 64),      # dense
    ((5, 64), (192, 1), 192),    # the middle third of 3x-wide rows
    ((1, 64), (999, 1), 64),     # one row: its stride does not matter
    ((5, 1), (8, 7), 8),         # one column: its column stride does not matter
])
def test_binding_row_stride(shape, stride, ld):
    assert binding._rows(_FakeMatrix(shape, stride), "x") == ld


@pytest.mark.parametrize("m", [
    _FakeMatrix((5, 64), (1, 5)),          # column-major
    _FakeMatrix((5, 64), (32, 1)),         # rows overlap
    _FakeMatrix((5, 64, 2), (128, 2, 1)),  # not a matrix
    _FakeMatrix((5, 64), (64, 1), is_cuda=False),
])
def test_binding_rejects_unusable_layouts(m):
    with pytest.raises(ValueError):
        binding._rows(m, "x")


def test_plan_size_and_host_checks(L):
    """The plan's size formula (16 header words, group offsets and adapters, the row list) and
    the host checks of sgmv_plan and the planned calls (num_segments = 0: checks only)."""
    assert L.sgmv_plan_size(64, 64) == 4 * (16 + 2 * 64 + 1 + 64)
    assert L.sgmv_plan_size(0, 0) == 4 * 17
    assert L.sgmv_plan_size(-1, 5) == 0 and L.sgmv_plan_size(5, -1) == 0
    assert L.sgmv_plan_size(4097, 5) == 0
    a = OK_ARGS
    plan = P + 0x60000
    n = L.sgmv_plan_size(8, 100)
    assert L.sgmv_plan(a["ss"], a["sa"], 8, 100, plan, n - 4, None) == -1   # too small
    assert L.sgmv_plan(a["ss"], a["sa"], 8, 100, None, n, None) == -1
    assert L.sgmv_plan(a["ss"], a["sa"], 8, 100, plan + 4, n, None) == -2  # plan misaligned
    assert L.sgmv_plan(a["ss"], a["sa"], 4097, 100, plan, 1 << 30, None) == -3
    assert L.sgmv_plan(a["ss"], a["sa"], -1, 100, plan, n, None) == -1

    def planned(plan=plan, S=0, flags=0, r=16, ldx=4096, ldy=4096):
        return L.lora_apply_planned(a["y"], ldy, a["x"], ldx, a["A"], a["B"], plan, S, 0, 4096,
                                    4096, r, 1.0, 1, flags, None)
    assert planned() == 0
    assert planned(plan=None) == -1
    assert planned(plan=plan + 8) == -2
    assert planned(S=4097) == -3
    assert planned(r=12) == -3
    assert planned(flags=6) == -1
    assert planned(ldx=4088, S=4) == -1
    assert L.sgmv_shrink_planned(a["y"], a["x"], 4096, a["A"], None, 4, 0, 4096, 16, 1, 0,
                                 None) == -1
    assert L.sgmv_shrink_planned(a["y"], a["x"], 4096, a["A"], plan, 0, 0, 4096, 16, 1, 0,
                                 None) == 0
    assert L.sgmv_expand_planned(a["y"], 4096, a["x"], a["B"], plan, 4, 0, 16, 4090, 1.0, 1, 0,
                                 None) == -2
    assert L.sgmv_expand_planned(a["y"], 4096, a["x"], a["B"], plan, 0, 0, 16, 4096, 1.0, 1, 0,
                                 None) == 0


def test_multi_host_checks(L):
    a = OK_ARGS
    plan = P + 0x60000

    def proj(**kw):
        d = dict(y=a["y"], x=a["x"], A_ptrs=a["A"], B_ptrs=a["B"], ldy=4096, ldx=4096, h_in=4096,
                 h_out=4096, scale=1.0, reserved=0)
        d.update(kw)
        return binding.Projection(**d)

    def multi(projs, S=0, plan=plan, r=16, flags=0):
        arr = (binding.Projection * max(1, len(projs)))(*projs)
        return L.lora_apply_multi(arr, len(projs), plan, S, 0, r, 1, flags, None)
    assert multi([proj(), proj(h_out=1024, ldy=1024)]) == 0
    assert multi([]) == -1
    assert multi([proj()] * 5) == -3
    assert multi([proj(), proj(y=None)]) == -1
    assert multi([proj(), proj(h_out=1020, ldy=1020)]) == -2
    assert multi([proj(x=P + 0x10008)]) == -2
    assert multi([proj()], plan=None) == -1
    assert multi([proj()], r=24) == -3
    assert multi([proj()], flags=32) == -1


def test_pool_host_checks(L):
    """The adapter pool's size formula and the checks it makes before any CUDA call."""
    import ctypes
    assert L.sgmv_pool_slot_bytes(2, 4096, 4096, 16, 1) == 2 * (2 * 4096 * 16 * 2)
    assert L.sgmv_pool_slot_bytes(1, 100, 60, 8, 0) == 3328 + 2048  # each block up to 256 B
    assert L.sgmv_pool_slot_bytes(0, 4096, 4096, 16, 1) == 0
    assert L.sgmv_pool_slot_bytes(1, 4096, 4096, 16, 9) == 0
    h = ctypes.c_void_p()
    sb = L.sgmv_pool_slot_bytes(1, 256, 256, 16, 1)
    assert L.sgmv_pool_create(None, P, 4 * sb, 4, 8, 1, 256, 256, 16, 1) == -1
    assert L.sgmv_pool_create(ctypes.byref(h), None, 4 * sb, 4, 8, 1, 256, 256, 16, 1) == -1
    assert L.sgmv_pool_create(ctypes.byref(h), P, 4 * sb, 0, 8, 1, 256, 256, 16, 1) == -1
    assert L.sgmv_pool_create(ctypes.byref(h), P, 3 * sb, 4, 8, 1, 256, 256, 16, 1) == -1
    assert L.sgmv_pool_create(ctypes.byref(h), P + 16, 4 * sb, 4, 8, 1, 256, 256, 16, 1) == -2
    assert L.sgmv_pool_destroy(None) == -1
    assert L.sgmv_pool_register(None, 0, P, P) == -1
    assert L.sgmv_pool_acquire(None, None, 0, P, P, None, None, None) == -1
    assert L.sgmv_pool_release(None, None, 0, None) == -1
    assert L.sgmv_pool_stats(None, None, None, None) == -1


def test_base_host_checks(L):
    """lora_apply_base: argument checks that need no device (M = 0 returns OK, no launch)."""
    a = OK_ARGS
    W0, v = P + 0x70000, P + 0x80000

    def base(M=0, S=4, dt=1, r=16, h_in=4096, h_out=4096, ldx=4096, ldy=4096, ldw=4096,
             x=a["x"], w=W0, vw=v, flags=0):
        return L.lora_apply_base(a["y"], ldy, x, ldx, M, w, ldw, a["A"], a["B"], a["ss"],
                                 a["sa"], S, 0, h_in, h_out, r, 1.0, vw, dt, flags, None)
    assert base() == 0
    assert base(S=0, vw=None) == 0
    assert base(dt=0) == -3          # fp32: the tensor cores take 16-bit operands
    assert base(r=24) == -3
    assert base(M=-1) == -1
    assert base(w=None) == -1
    assert base(vw=None) == -1       # segments need the workspace
    assert base(ldw=4090) == -1
    assert base(ldw=4100) == -2
    assert base(h_out=4092, ldy=4092) == -2
    assert base(x=P + 0x10008) == -2
    assert base(vw=v + 8) == -2
    assert base(flags=32) == -1
    assert base(S=5000) == -3
