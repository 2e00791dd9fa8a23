"""GPU parity of lora_apply_base (the base projection with the LoRA term added in its epilogue)
against the fp64 oracle (oracle.base_lora): |y - y_ref| <= 1e-2 + 1e-2 |y_ref| elementwise.

Cases span several 128-row and 256-column tiles with ragged tails, an h_in that is not a
multiple of the 64-wide K stage, every rank, both 16-bit types, tiles holding several
adapters (and one adapter in non-adjacent segments), rows without an adapter and rows outside
every segment; the prefill shape (4096 -> 11008, r = 64, bf16) is checked at full size on
sampled rows against the oracle and on every row against an fp32 torch reference.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
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
    torch.cuda.empty_cache()


def make_base(w, ss, sa, seed, M=None, num_adapters=None, layers=None):
    """A case plus a base weight W0 [h_out, h_in] ~ U(+-1/sqrt(h_in))."""
    c = harness.make_case(w, ss, sa, seed=seed, M=M, num_adapters=num_adapters, layers=layers)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 77)
    bound = 1.0 / np.sqrt(w.h_in)
    W0 = ((torch.rand((w.h_out, w.h_in), generator=g, device="cuda") * 2 - 1) * bound).to(
        workloads.torch_dtype(w.dtype))
    return c, W0


def oracle_base(c, W0, layer, rows=None):
    keys = harness.touched(c.sa, c.ss)
    A = harness.oracle_blocks(c.A, keys, layer)
    B = harness.oracle_blocks(c.B, keys, layer)
    x = c.x.double().cpu().numpy()
    W = W0.double().cpu().numpy()
    if rows is None:
        return oracle.base_lora(x, W, A, B, c.ss, c.sa, 0, c.w.scale)
    # selected rows only: each as its own row of a smaller problem
    ra = harness.row_adapters(c.ss, c.sa, c.M)
    xs = x[rows]
    ss = np.arange(len(rows) + 1, dtype=np.int32)
    sa = ra[rows].astype(np.int32)
    return oracle.base_lora(xs, W, A, B, ss, sa, 0, c.w.scale)


def run_base(c, W0, layer, **kw):
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_base
    y = torch.full((c.M, c.w.h_out), float("nan"), dtype=c.x.dtype, device="cuda")
    lora_apply_base(y, c.x, W0, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, layer, c.w.r, c.w.scale,
                    **kw)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("r", [8, 16, 32, 64])
def test_matches_oracle_every_row(dtype, r):
    """300 rows (3 m-tiles, 44 in the last), h_in 200 (a partial K stage), h_out 328 (a
    partial n-tile); segments: two of adapter 1 around one of adapter 2 inside the first tile,
    an empty one, one without an adapter, a long one across a tile edge, and rows 290-299 in
    no segment."""
    w = workloads.Workload(f"base_{dtype}_{r}", 200, 328, r, dtype, 4, 2)
    ss = np.array([0, 10, 30, 45, 45, 60, 250, 290], np.int32)
    sa = np.array([1, 2, 1, 3, -1, 0, 2], np.int32)
    c, W0 = make_base(w, ss, sa, seed=3 + r, M=300)
    y = run_base(c, W0, 1)
    ref = oracle_base(c, W0, 1)
    harness.assert_close(y.float().cpu().numpy(), ref, f"lora_apply_base {dtype} r={r}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_no_segments_is_the_base_projection(dtype):
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_base
    w = workloads.Workload("base_only", 512, 768, 16, dtype, 1, 1)
    c, W0 = make_base(w, [0], np.zeros(0, np.int32), seed=5, M=200)
    y = torch.full((200, 768), float("nan"), dtype=c.x.dtype, device="cuda")
    lora_apply_base(y, c.x, W0, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, 0, 16, 1.0)
    torch.cuda.synchronize()
    ref = c.x.double().cpu().numpy() @ W0.double().cpu().numpy().T
    harness.assert_close(y.float().cpu().numpy(), ref, "base only")


def test_many_adapters_per_tile():
    """A decode-style table: 256 one-row segments over 24 adapters (repeats not adjacent), so
    every tile holds many LoRA rounds."""
    rng = np.random.default_rng(9)
    w = workloads.Workload("base_decode", 256, 512, 16, "bf16", 24, 1)
    ss = np.arange(257, dtype=np.int32)
    sa = rng.integers(-1, 24, size=256).astype(np.int32)
    c, W0 = make_base(w, ss, sa, seed=11)
    y = run_base(c, W0, 0)
    harness.assert_close(y.float().cpu().numpy(), oracle_base(c, W0, 0), "many adapters")


def test_strided_x_and_y():
    """x and y as column slices of wider matrices (row strides 3 h)."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_base
    w = workloads.Workload("base_strided", 256, 320, 32, "f16", 3, 1)
    ss = np.array([0, 70, 71, 200], np.int32)
    sa = np.array([2, 0, 1], np.int32)
    c, W0 = make_base(w, ss, sa, seed=13, M=210)
    X = torch.zeros((210, 3 * 256), dtype=c.x.dtype, device="cuda")
    X[:, 256:512] = c.x
    Y = torch.full((210, 3 * 320), 7.0, dtype=c.x.dtype, device="cuda")
    lora_apply_base(Y[:, 320:640], X[:, 256:512], W0, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, 0,
                    32, c.w.scale)
    torch.cuda.synchronize()
    harness.assert_close(Y[:, 320:640].float().cpu().numpy(), oracle_base(c, W0, 0), "strided")
    assert bool((Y[:, :320] == 7.0).all()) and bool((Y[:, 640:] == 7.0).all())


def test_prefill_shape_full_size():
    """prefill_mixed's shape (4096 -> 11008, r = 64, bf16, 8 segments of 128-1024 rows): 96
    sampled rows (tile edges, segment edges, random) against the oracle, and every row against
    x W0^T in fp32 (torch) plus the LoRA term of lora_apply (checked against the oracle
    elsewhere)."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    w = workloads.WORKLOADS["prefill_mixed"]
    ss, sa = workloads.make_segments(w.name, 0)
    c, W0 = make_base(w, ss, sa, seed=21)
    y = run_base(c, W0, 0)
    rng = np.random.default_rng(4)
    rows = set(int(t) for t in rng.integers(0, c.M, size=48))
    for i in range(len(sa)):
        rows.update([int(ss[i]), int(ss[i + 1]) - 1])
    rows.update(t for t in range(127, c.M, 128))
    rows.update([c.M - 1])
    rows = np.array(sorted(rows))[:96]
    ref = oracle_base(c, W0, 0, rows=rows)
    harness.assert_close(y[torch.as_tensor(rows, device="cuda")].float().cpu().numpy(), ref,
                         "prefill shape, sampled rows")
    base = (c.x.float() @ W0.float().T).to(c.x.dtype)
    lora_apply(base, c.x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, 0, w.r, w.scale)
    torch.cuda.synchronize()
    yf, bf = y.float(), base.float()
    bad = (yf - bf).abs() > 2e-2 + 2e-2 * bf.abs()
    assert not bool(bad.any()), f"{int(bad.sum())} elements differ from x W0^T + lora_apply"


def test_wait_timeout_reports_and_recovers():
    """A stall injected into every CTA runs out the (shortened) wait bound: the call reports
    SGMV_ETIMEOUT and writes nothing; the next call is correct."""
    from segmented_gather_gemm_sgmv_gb300 import sgmv_get_error, sgmv_set_wait_limit
    w = workloads.Workload("base_timeout", 256, 512, 16, "bf16", 2, 1)
    ss = np.array([0, 100, 200], np.int32)
    sa = np.array([0, 1], np.int32)
    c, W0 = make_base(w, ss, sa, seed=31, M=256)
    assert sgmv_get_error(clear=True) == 0
    sgmv_set_wait_limit(2_000_000, inject_stall=True)
    try:
        y = run_base(c, W0, 0)
    finally:
        sgmv_set_wait_limit(0)
    assert sgmv_get_error(clear=True) == -5
    assert bool(torch.isnan(y.float()).all()), "a call that gave up wrote y"
    y = run_base(c, W0, 0)
    assert sgmv_get_error(clear=True) == 0
    harness.assert_close(y.float().cpu().numpy(), oracle_base(c, W0, 0), "after a timeout")
