"""GPU parity of the tensor-core role (tcgen05.mma) of lora_apply, through the C ABI.

With SGMV_TENSOR_CORES_ALWAYS, adapter groups of at least 64 rows run on the tensor cores
(fp16 / bf16, r >= 16); smaller groups stay on the CUDA cores.  The cases below mix both kinds in one call, span several
128-row m-tiles and 64-column n-tiles, and give h_in / h_out ragged tails (not multiples of
64), groups gathered from non-adjacent segments, and the 63 / 64-row boundary.  Every case is
compared with the fp64 oracle (|y - y_ref| <= 1e-2 + 1e-2 |y_ref|) and with the same call
forced onto the CUDA cores (SGMV_NO_TENSOR_CORES); integer-valued inputs are bit-exact.
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


# Long groups: adapter 1 (200 rows over three segments), adapter 3 (64 rows, the smallest
# tensor group), adapter 0 (300 rows: three m-tiles, ragged last one); short groups: adapter 2
# (63 rows over two segments), adapter 4 (1 row), adapter 5 (5 rows); one empty segment and
# one segment with no adapter.
MIXED_LENS = [70, 1, 64, 40, 300, 0, 23, 90, 5, 40, 7]
MIXED_IDS = [1, 4, 3, 2, 0, 2, 2, 1, 5, 1, -1]


@pytest.mark.parametrize("dtype,r,h_in,h_out", [
    ("bf16", 64, 512, 640),
    ("f16", 16, 200, 328),     # ragged K chunk and ragged n-tile
    ("bf16", 32, 1000, 136),
    ("f16", 64, 264, 4104),
    ("bf16", 64, 128, 200),    # two K chunks: two of the four split-K members shrink nothing
])
def test_mixed_groups_match_oracle_and_cuda_cores(dtype, r, h_in, h_out):
    w = workloads.Workload("tc_mixed", h_in, h_out, r, dtype, 6, 2)
    ss, sa = _table(MIXED_LENS, MIXED_IDS)
    c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 3)
    for layer in (0, 1):
        y_tc = harness.run_apply(c, layer, tensor_cores="always")
        y_cc = harness.run_apply(c, layer, tensor_cores="never")
        ref = harness.oracle_apply(c, layer)
        harness.assert_close(y_tc.float().cpu().numpy(), ref, f"tensor {dtype} r{r} L{layer}")
        harness.assert_close(y_cc.float().cpu().numpy(), ref, f"cuda-core {dtype} r{r} L{layer}")
        keep = harness.row_adapters(c.ss, c.sa, c.M) < 0
        idx = torch.as_tensor(np.nonzero(keep)[0], device="cuda")
        assert torch.equal(y_tc[idx], c.y0[idx]), "rows without an adapter were modified"


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_integer_exact_tensor_groups(dtype):
    """x, A, B in {-1,0,1}, h_in <= 256: v is an integer of magnitude <= 256, exact in the
    16-bit high part (low part 0), so the tensor path must equal the oracle bit for bit."""
    dt = workloads.torch_dtype(dtype)
    r, h_in, h_out, n = 32, 256, 320, 6
    w = workloads.Workload("tc_int", h_in, h_out, r, dtype, n, 1)
    ss, sa = _table(MIXED_LENS, MIXED_IDS)
    g = torch.Generator(device="cuda").manual_seed(21)
    A = torch.randint(-1, 2, (n, 1, h_in, r), generator=g, device="cuda").to(dt)
    B = torch.randint(-1, 2, (n, 1, r, h_out), generator=g, device="cuda").to(dt)
    c = harness.make_case(w, ss, sa, pool=(A, B))
    c.x = torch.randint(-1, 2, c.x.shape, generator=g, device="cuda").to(dt)
    c.y0 = torch.randint(-4, 5, c.y0.shape, generator=g, device="cuda").to(dt)
    y = harness.run_apply(c, 0, tensor_cores="always")
    ref = torch.as_tensor(harness.oracle_apply(c, 0)).to(dt)
    assert torch.equal(y.cpu(), ref), f"tensor path not bit-exact ({dtype})"


def test_adapter_tags_long_groups():
    """A_k[:,0] = (k+1) e_0, x[:,0] = 1, B_k row 0 = e_0: y[t,0] - y_in[t,0] = scale (k(t)+1)
    names the adapter of every row, including rows gathered into m-tiles across segments."""
    r, h, n = 16, 256, 8
    w = workloads.Workload("tc_tag", h, h, r, "bf16", n, 1)
    lens = [100, 30, 3, 130, 40, 1, 60, 70]
    ids = [0, 1, 2, 3, 1, 4, 1, 5]
    ss, sa = _table(lens, ids)
    A = torch.zeros((n, 1, h, r), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((n, 1, r, h), dtype=torch.bfloat16, device="cuda")
    for k in range(n):
        A[k, 0, 0, 0] = k + 1
    B[:, 0, 0, 0] = 1
    c = harness.make_case(w, ss, sa, pool=(A, B))
    c.x = torch.zeros_like(c.x)
    c.x[:, 0] = 1
    c.y0 = torch.zeros_like(c.y0)
    y = harness.run_apply(c, 0, tensor_cores="always")
    want = np.zeros(c.M)
    for i, k in enumerate(sa):
        want[ss[i]:ss[i + 1]] = w.scale * (k + 1)
    assert np.array_equal(y[:, 0].float().cpu().numpy(), want)
    assert torch.count_nonzero(y[:, 1:]) == 0


def test_guard_rows_around_tensor_groups():
    """NaN rows before, between and after long segments stay NaN (never read into a tile
    that is stored, never written)."""
    w = workloads.Workload("tc_guard", 384, 200, 64, "bf16", 3, 1)
    ss = np.array([5, 140, 150, 290], np.int32)
    sa = np.array([0, -1, 2], np.int32)
    c = harness.make_case(w, ss, sa, M=300)
    c.y0[:5] = float("nan")
    c.y0[140:150] = float("nan")
    c.y0[290:] = float("nan")
    y = harness.run_apply(c, 0, tensor_cores="always")
    assert torch.isnan(y[:5]).all() and torch.isnan(y[140:150]).all()
    assert torch.isnan(y[290:]).all()
    ref = harness.oracle_apply(c, 0)
    for lo, hi in ((5, 140), (150, 290)):
        harness.assert_close(y[lo:hi].float().cpu().numpy(), ref[lo:hi], f"rows {lo}:{hi}")


def test_many_tiles_deterministic():
    """Several (m-tile, n-tile) pairs per tensor CTA, ranges that cross m-tile boundaries (a
    CTA then computes two shrinks); two runs give identical bits."""
    w = workloads.Workload("tc_many", 512, 1024, 64, "f16", 4, 1)
    lens = [1500, 900, 2100, 700]
    ss, sa = _table(lens, [0, 1, 2, 3])
    c = harness.make_case(w, ss, sa)
    y1 = harness.run_apply(c, 0, tensor_cores="always")
    y2 = harness.run_apply(c, 0, tensor_cores="always")
    assert torch.equal(y1, y2)
    rng = np.random.default_rng(9)
    rows = set(rng.choice(c.M, 200, replace=False).tolist())
    for i in range(len(lens)):
        rows.update({int(ss[i]), int(ss[i + 1]) - 1})
        rows.update(int(t) for t in range(ss[i] + 127, ss[i + 1], 128))
    rows, ref = harness.oracle_apply(c, 0, rows=rows)
    harness.assert_close(y1[torch.as_tensor(rows, device="cuda")].float().cpu().numpy(), ref,
                         "many tiles")


def test_large_table_gathered_group():
    """A segment table large enough that fewer ring slots fit beside it (three), with one
    adapter's rows scattered over hundreds of single-row segments (one gathered m-tile, no
    consecutive rows) next to two 16-row segments and many short groups."""
    w = workloads.Workload("tc_table", 1024, 768, 64, "bf16", 64, 1)
    rng = np.random.default_rng(17)
    ids = rng.choice(64, size=600, p=np.r_[0.3, np.full(63, 0.7 / 63)]).astype(np.int32)
    lens = np.ones(602, np.int64)
    lens[:2] = 16
    ids = np.r_[[0, 5], ids].astype(np.int32)
    ss, sa = _table(lens, ids)
    c = harness.make_case(w, ss, sa)
    y = harness.run_apply(c, 0, tensor_cores="always")
    y_cc = harness.run_apply(c, 0, tensor_cores="never")
    ref = harness.oracle_apply(c, 0)
    harness.assert_close(y.float().cpu().numpy(), ref, "large table, tensor")
    harness.assert_close(y_cc.float().cpu().numpy(), ref, "large table, cuda cores")


@pytest.mark.parametrize("dtype,r,h_in,h_out", [("bf16", 64, 512, 640), ("f16", 16, 200, 328),
                                                ("bf16", 32, 1000, 136), ("f16", 32, 128, 72)])
def test_unfused_shrink_and_expand_on_tensor_cores(dtype, r, h_in, h_out):
    """sgmv_shrink_ex / sgmv_expand_ex with SGMV_TENSOR_CORES_ALWAYS: long groups run the
    tensor role's shrink-only (v rows to v_out) and expand-only (v rows from v_in) forms;
    compared with the oracle and with the CUDA-core forms of the same calls."""
    import oracle
    from segmented_gather_gemm_sgmv_gb300 import sgmv_expand, sgmv_shrink
    w = workloads.Workload("tc_unfused", h_in, h_out, r, dtype, 6, 2)
    ss, sa = _table(MIXED_LENS, MIXED_IDS)
    c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 3)
    layer = 1
    keys = harness.touched(sa, ss)
    A = harness.oracle_blocks(c.A, keys, layer)
    B = harness.oracle_blocks(c.B, keys, layer)
    vs = {}
    for mode in ("always", "never"):
        v = torch.full((c.M, r), -7.0, device="cuda")
        sgmv_shrink(v, c.x, c.A_ptrs, c.d_ss, c.d_sa, layer, r, tensor_cores=mode)
        vs[mode] = v
    v_ref = oracle.sgmv_shrink(np.full((c.M, r), -7.0), c.x.double().cpu().numpy(), A, ss, sa, 0)
    for mode, v in vs.items():
        harness.assert_close(v.cpu().numpy(), v_ref, f"shrink {mode}", atol=1e-3, rtol=1e-3)
    v = vs["never"]
    y_ref = oracle.sgmv_expand(c.y0.double().cpu().numpy(), v.double().cpu().numpy(), B, ss, sa,
                               0, w.scale)
    for mode in ("always", "never"):
        y = c.y0.clone()
        sgmv_expand(y, v, c.B_ptrs, c.d_ss, c.d_sa, layer, r, w.scale, tensor_cores=mode)
        harness.assert_close(y.float().cpu().numpy(), y_ref, f"expand {mode}")
