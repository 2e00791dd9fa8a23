"""GPU parity of lora_apply / sgmv_shrink / sgmv_expand launched with SGMV_LONG_BATCH (one
CTA per SM with the whole shared memory: deeper rings for both the CUDA-core and the tensor
roles), through the C ABI.

Each case is compared with the fp64 oracle (|y - y_ref| <= 1e-2 + 1e-2 |y_ref|).  Integer-valued
inputs make every summation order exact, so there the long-batch launch must equal the default
launch and the oracle bit for bit.
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


# long groups (tensor role when allowed), short groups, an empty segment, a segment with no
# adapter
LENS = [70, 1, 64, 40, 300, 0, 23, 90, 5, 40, 7]
IDS = [1, 4, 3, 2, 0, 2, 2, 1, 5, 1, -1]


@pytest.mark.parametrize("dtype,r,h_in,h_out", [
    ("bf16", 64, 512, 640),
    ("f16", 16, 200, 328),
    ("f32", 16, 264, 136),     # CUDA-core role only
])
@pytest.mark.parametrize("tensor_cores", ["auto", "always", "never"])
def test_long_batch_matches_oracle(dtype, r, h_in, h_out, tensor_cores):
    if dtype == "f32" and tensor_cores == "always":
        pytest.skip("no tensor role for fp32")
    w = workloads.Workload("long", h_in, h_out, r, dtype, 6, 2)
    ss, sa = _table(LENS, IDS)
    c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 3)
    for layer in (0, 1):
        y = harness.run_apply(c, layer, tensor_cores=tensor_cores, long_batch=True)
        harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, layer),
                             f"long batch {dtype} r{r} {tensor_cores} L{layer}")
        keep = harness.row_adapters(c.ss, c.sa, c.M) < 0
        idx = torch.as_tensor(np.nonzero(keep)[0], device="cuda")
        assert torch.equal(y[idx], c.y0[idx]), "rows without an adapter were modified"


def test_long_batch_decode_rows():
    """Many one-row segments (the CUDA-core groups of CTAs, E > 1, with the partial-sum
    exchange) under the long-batch geometry."""
    n = 96
    w = workloads.Workload("long_decode", 1024, 1536, 16, "f16", n, 1)
    rng = np.random.default_rng(5)
    ids = rng.permutation(n).astype(np.int32)
    ss, sa = _table([1] * n, ids)
    c = harness.make_case(w, ss, sa)
    y = harness.run_apply(c, 0, long_batch=True)
    harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, 0), "long decode")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("tensor_cores", ["always", "never"])
def test_long_batch_integer_exact(dtype, tensor_cores):
    """x, A, B in {-1,0,1} and h_in <= 256: both geometries and the oracle agree bit for bit."""
    dt = workloads.torch_dtype(dtype)
    r, h_in, h_out, n = 32, 256, 320, 6
    w = workloads.Workload("long_int", h_in, h_out, r, dtype, n, 1)
    ss, sa = _table(LENS, IDS)
    g = torch.Generator(device="cuda").manual_seed(22)
    A = torch.randint(-1, 2, (n, 1, h_in, r), generator=g, device="cuda").to(dt)
    B = torch.randint(-1, 2, (n, 1, r, h_out), generator=g, device="cuda").to(dt)
    c = harness.make_case(w, ss, sa, pool=(A, B))
    c.x = torch.randint(-1, 2, c.x.shape, generator=g, device="cuda").to(dt)
    c.y0 = torch.randint(-4, 5, c.y0.shape, generator=g, device="cuda").to(dt)
    y_long = harness.run_apply(c, 0, tensor_cores=tensor_cores, long_batch=True)
    y_pair = harness.run_apply(c, 0, tensor_cores=tensor_cores)
    ref = torch.as_tensor(harness.oracle_apply(c, 0)).to(dt)
    assert torch.equal(y_long.cpu(), ref), f"long batch not bit-exact ({dtype}, {tensor_cores})"
    assert torch.equal(y_long, y_pair)


def test_long_batch_unfused_forms():
    """sgmv_shrink / sgmv_expand with long_batch=True against the oracle."""
    import oracle
    from segmented_gather_gemm_sgmv_gb300 import sgmv_expand, sgmv_shrink
    r = 64
    w = workloads.Workload("long_unfused", 512, 640, r, "bf16", 6, 2)
    ss, sa = _table(LENS, IDS)
    c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 3)
    layer = 1
    keys = harness.touched(sa, ss)
    A = harness.oracle_blocks(c.A, keys, layer)
    B = harness.oracle_blocks(c.B, keys, layer)
    for mode in ("always", "never"):
        v = torch.full((c.M, r), -7.0, device="cuda")
        sgmv_shrink(v, c.x, c.A_ptrs, c.d_ss, c.d_sa, layer, r, tensor_cores=mode,
                    long_batch=True)
        v_ref = oracle.sgmv_shrink(np.full((c.M, r), -7.0), c.x.double().cpu().numpy(), A, ss,
                                   sa, 0)
        harness.assert_close(v.cpu().numpy(), v_ref, f"shrink {mode}", atol=1e-3, rtol=1e-3)
        y = c.y0.clone()
        sgmv_expand(y, v, c.B_ptrs, c.d_ss, c.d_sa, layer, r, w.scale, tensor_cores=mode,
                    long_batch=True)
        y_ref = oracle.sgmv_expand(c.y0.double().cpu().numpy(), v.double().cpu().numpy(), B, ss,
                                   sa, 0, w.scale)
        harness.assert_close(y.float().cpu().numpy(), y_ref, f"expand {mode}")


@pytest.mark.parametrize("dtype,r", [("bf16", 64), ("f16", 16)])
def test_long_batch_ring_reuse_across_shrink_and_expand(dtype, r):
    """More shrink chunks per cluster member than the ring has slots (h_in = 3072: 12 chunks
    per member over 8 slots), so every expand slot reuses a slot that held shrink data earlier
    in the same m-tile, and many n-tiles per member for both epilogue groups of the 416-thread
    kernel.  Fused and unfused forms against the oracle, every row."""
    import oracle
    from segmented_gather_gemm_sgmv_gb300 import sgmv_expand, sgmv_shrink
    w = workloads.Workload("long_reuse", 3072, 2560, r, dtype, 4, 1)
    ss, sa = _table([400, 200, 129, 300, 3], [0, 1, 2, 0, 3])
    c = harness.make_case(w, ss, sa)
    y = harness.run_apply(c, 0, tensor_cores="always", long_batch=True)
    harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, 0),
                         f"ring reuse {dtype} fused")
    keys = harness.touched(sa, ss)
    B = harness.oracle_blocks(c.B, keys, 0)
    v = torch.zeros((c.M, r), device="cuda")
    sgmv_shrink(v, c.x, c.A_ptrs, c.d_ss, c.d_sa, 0, r, tensor_cores="always", long_batch=True)
    y = c.y0.clone()
    sgmv_expand(y, v, c.B_ptrs, c.d_ss, c.d_sa, 0, r, w.scale, tensor_cores="always",
                long_batch=True)
    y_ref = oracle.sgmv_expand(c.y0.double().cpu().numpy(), v.double().cpu().numpy(), B, ss, sa,
                               0, w.scale)
    harness.assert_close(y.float().cpu().numpy(), y_ref, f"ring reuse {dtype} expand")
