"""GPU parity of the strided entry points (lora_apply_strided, sgmv_shrink_strided,
sgmv_expand_strided), through the C ABI: x and y are column slices of wider matrices, as the
q / k / v parts of a fused projection output are.

Each case compares the slice with the fp64 oracle run on dense copies
(|y - y_ref| <= 1e-2 + 1e-2 |y_ref|), and checks that every element of the wide y outside the
slice is bit-for-bit unchanged.  The cases cover the CUDA-core and the tensor-core roles (TMA
row boxes and gathered rows), both launch geometries, and fp32 / fp16 / bf16.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from segmented_gather_gemm_sgmv_gb300 import workloads  # noqa: E402
from tests import harness  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    from segmented_gather_gemm_sgmv_gb300 import binding
    binding.lib()
    yield
    torch.cuda.synchronize()


def _table(lens, ids):
    ss = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return ss, np.asarray(ids, np.int32)


# long groups (tensor role when allowed; adapter 1 gathered from three segments), short groups,
# an empty segment, a segment with no adapter
LENS = [70, 1, 64, 40, 300, 0, 23, 90, 5, 40, 7]
IDS = [1, 4, 3, 2, 0, 2, 2, 1, 5, 1, -1]


def _wide(c, x_off, x_pad, y_off, y_pad, seed):
    """Wide x / y holding c.x / c.y0 at column offsets, with random values around them."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    M, h_in = c.x.shape
    h_out = c.y0.shape[1]
    X = torch.randn((M, x_off + h_in + x_pad), generator=g, device="cuda").to(c.x.dtype)
    Y = torch.randn((M, y_off + h_out + y_pad), generator=g, device="cuda").to(c.y0.dtype)
    X[:, x_off:x_off + h_in] = c.x
    Y[:, y_off:y_off + h_out] = c.y0
    return X, Y


@pytest.mark.parametrize("dtype,r,h_in,h_out", [
    ("bf16", 64, 512, 640),
    ("f16", 16, 200, 328),
    ("f32", 16, 264, 136),
])
@pytest.mark.parametrize("tensor_cores", ["always", "never"])
@pytest.mark.parametrize("long_batch", [False, True])
def test_lora_apply_on_column_slices(dtype, r, h_in, h_out, tensor_cores, long_batch):
    if dtype == "f32" and tensor_cores == "always":
        pytest.skip("no tensor role for fp32")
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    w = workloads.Workload("strided", h_in, h_out, r, dtype, 6, 2)
    ss, sa = _table(LENS, IDS)
    c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 3)
    x_off, y_off = 16, 8
    X, Y = _wide(c, x_off, 24, y_off, 40, seed=3)
    Y0 = Y.clone()
    x = X[:, x_off:x_off + h_in]
    y = Y[:, y_off:y_off + h_out]
    assert x.stride(0) != h_in and y.stride(0) != h_out
    layer = 1
    lora_apply(y, x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, layer, r, w.scale,
               tensor_cores=tensor_cores, long_batch=long_batch)
    ref = harness.oracle_apply(c, layer)
    harness.assert_close(y.float().cpu().numpy(), ref,
                         f"strided {dtype} r{r} {tensor_cores} long={long_batch}")
    outside = torch.ones_like(Y, dtype=torch.bool)
    outside[:, y_off:y_off + h_out] = False
    assert torch.equal(Y[outside], Y0[outside]), "elements outside the y slice were modified"
    assert torch.equal(X[:, x_off:x_off + h_in], c.x), "x was modified"


def test_lora_apply_strided_equals_dense_bitwise():
    """The same call on a slice and on a dense copy gives bit-identical rows (the row stride
    changes addresses only)."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    w = workloads.Workload("strided_eq", 1024, 1536, 16, "f16", 8, 1)
    rng = np.random.default_rng(11)
    ids = rng.permutation(8)
    ss, sa = _table([1, 3, 2, 70, 1, 4, 100, 2], ids)
    c = harness.make_case(w, ss, sa)
    X, Y = _wide(c, 8, 8, 16, 24, seed=5)
    y_dense = c.y0.clone()
    lora_apply(y_dense, c.x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, 0, w.r, w.scale)
    y = Y[:, 16:16 + w.h_out]
    lora_apply(y, X[:, 8:8 + w.h_in], c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, 0, w.r, w.scale)
    assert torch.equal(y, y_dense)


@pytest.mark.parametrize("tensor_cores", ["always", "never"])
def test_shrink_and_expand_on_column_slices(tensor_cores):
    import oracle
    from segmented_gather_gemm_sgmv_gb300 import sgmv_expand, sgmv_shrink
    r = 64
    w = workloads.Workload("strided_unfused", 512, 640, r, "bf16", 6, 2)
    ss, sa = _table(LENS, IDS)
    c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 3)
    layer = 1
    keys = harness.touched(sa, ss)
    A = harness.oracle_blocks(c.A, keys, layer)
    B = harness.oracle_blocks(c.B, keys, layer)
    X, Y = _wide(c, 24, 8, 8, 56, seed=7)
    Y0 = Y.clone()
    v = torch.full((c.M, r), -7.0, device="cuda")
    sgmv_shrink(v, X[:, 24:24 + w.h_in], c.A_ptrs, c.d_ss, c.d_sa, layer, r,
                tensor_cores=tensor_cores)
    v_ref = oracle.sgmv_shrink(np.full((c.M, r), -7.0), c.x.double().cpu().numpy(), A, ss, sa, 0)
    harness.assert_close(v.cpu().numpy(), v_ref, f"shrink {tensor_cores}", atol=1e-3, rtol=1e-3)
    y = Y[:, 8:8 + w.h_out]
    sgmv_expand(y, v, c.B_ptrs, c.d_ss, c.d_sa, layer, r, w.scale, tensor_cores=tensor_cores)
    y_ref = oracle.sgmv_expand(c.y0.double().cpu().numpy(), v.double().cpu().numpy(), B, ss, sa,
                               0, w.scale)
    harness.assert_close(y.float().cpu().numpy(), y_ref, f"expand {tensor_cores}")
    outside = torch.ones_like(Y, dtype=torch.bool)
    outside[:, 8:8 + w.h_out] = False
    assert torch.equal(Y[outside], Y0[outside]), "elements outside the y slice were modified"
