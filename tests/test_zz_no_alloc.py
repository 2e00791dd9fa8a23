"""lora_apply_static_plan, the entry point that allocates no device memory, against lora_apply.

lora_apply_static_plan builds the adapter grouping into a fixed array inside the library and
applies it.  These tests call it through the C-ABI (the ctypes binding) twice in a row on one
stream with different segment tables and layers, so the second call runs on the array that the
first one filled, and compare every row with lora_apply on the same inputs:
|y - y_ref| <= 1e-2 + 1e-2 |y_ref| elementwise.  The file name puts it last in collection: it
must pass on its own in a fresh process (the first call sets the array up) and after the rest.
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
    torch.cuda.empty_cache()


def assert_close(y, ref, what):
    y, ref = y.float(), ref.float()
    bad = (y - ref).abs() > harness.ATOL + harness.RTOL * ref.abs()
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} elements out of tolerance"


def shuffled_table(ss, sa, seed):
    """The same rows and adapters with the segments in another order (same row ranges)."""
    rng = np.random.default_rng(seed)
    sa = np.asarray(sa, np.int32).copy()
    rng.shuffle(sa)
    return np.asarray(ss, np.int32), sa


@pytest.mark.parametrize("name,layers,long_batch", [
    ("decode_zipf", (0, 3), False),
    ("decode_distinct", (31, 0), False),
    ("prefill_mixed", (0, 0), True),
])
def test_two_calls_in_a_row_match_lora_apply(name, layers, long_batch):
    from segmented_gather_gemm_sgmv_gb300 import lora_apply, lora_apply_static_plan
    w = workloads.WORKLOADS[name]
    ss1, sa1 = workloads.make_segments(name, 0)
    ss2, sa2 = shuffled_table(ss1, sa1, 7)
    if name == "decode_zipf":
        sa2[::5] = -1  # some segments without an adapter in the second call
    n_layers = max(layers) + 1
    c = harness.make_case(w, ss1, sa1, layers=n_layers)
    tables = [(c.d_ss, c.d_sa),
              (torch.as_tensor(ss2, device="cuda"), torch.as_tensor(sa2, device="cuda"))]
    M = c.M
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    outs, refs = [], []
    with torch.cuda.stream(stream):
        for (d_ss, d_sa), layer in zip(tables, layers):
            y = c.y0.clone()
            lora_apply_static_plan(y, c.x, c.A_ptrs, c.B_ptrs, d_ss, d_sa, M, layer, w.r,
                                   w.scale, stream=stream, long_batch=long_batch)
            outs.append(y)
        for (d_ss, d_sa), layer in zip(tables, layers):
            y = c.y0.clone()
            lora_apply(y, c.x, c.A_ptrs, c.B_ptrs, d_ss, d_sa, layer, w.r, w.scale,
                       stream=stream, long_batch=long_batch)
            refs.append(y)
    torch.cuda.synchronize()
    from segmented_gather_gemm_sgmv_gb300 import sgmv_get_error
    assert sgmv_get_error(clear=True) == 0
    for i, (y, ref) in enumerate(zip(outs, refs)):
        assert_close(y, ref, f"{name} call {i + 1}")
    # rows without an adapter in the second table keep the base output bit for bit
    rows = harness.row_adapters(ss2, sa2, M)
    keep = torch.as_tensor(np.nonzero(rows < 0)[0], device="cuda")
    if keep.numel():
        assert torch.equal(outs[1][keep], c.y0[keep])


def test_limits_and_flags_are_refused_before_any_launch():
    from segmented_gather_gemm_sgmv_gb300 import binding
    w = workloads.WORKLOADS["tiny"]
    c = harness.make_case(w, [0, 3, 9], [1, 2])
    y = c.y0.clone()
    L = binding.lib()
    stream = torch.cuda.current_stream().cuda_stream

    def call(max_rows, flags, S=2, ss=c.d_ss, sa=c.d_sa):
        return L.lora_apply_static_plan(
            y.data_ptr(), y.shape[1], c.x.data_ptr(), c.x.shape[1], c.A_ptrs.data_ptr(),
            c.B_ptrs.data_ptr(), ss.data_ptr(), sa.data_ptr(), S, max_rows, 0, w.h_in, w.h_out,
            w.r, 1.0, binding._dtype_code(c.x), flags, stream)

    assert call(binding.SGMV_STATIC_PLAN_MAX_ROWS + 1, 0) == binding.SGMV_EUNSUPPORTED
    big_ss = torch.zeros(binding.SGMV_MAX_SEGMENTS + 2, dtype=torch.int32, device="cuda")
    big_sa = torch.full((binding.SGMV_MAX_SEGMENTS + 1,), -1, dtype=torch.int32, device="cuda")
    assert call(16, 0, binding.SGMV_MAX_SEGMENTS + 1, big_ss, big_sa) == \
        binding.SGMV_EUNSUPPORTED
    assert call(16, binding.SGMV_OVERLAP_PRIOR) == binding.SGMV_EINVAL
    assert call(-1, 0) == binding.SGMV_EINVAL
    torch.cuda.synchronize()
    assert torch.equal(y, c.y0)
    # the largest accepted capacity runs and matches lora_apply
    assert call(binding.SGMV_STATIC_PLAN_MAX_ROWS, 0) == binding.SGMV_OK
    ref = c.y0.clone()
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    lora_apply(ref, c.x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, 0, w.r, 1.0)
    torch.cuda.synchronize()
    assert_close(y, ref, "tiny at the largest capacity")


def test_rows_beyond_capacity_report_and_leave_y():
    """A table with more rows than max_rows: the plan reports the overflow, the apply call
    writes nothing and the library's error word says SGMV_EPLAN."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_static_plan, sgmv_get_error
    w = workloads.WORKLOADS["tiny"]
    c = harness.make_case(w, [0, 3, 9], [1, 2])
    assert sgmv_get_error(clear=True) == 0
    y = c.y0.clone()
    lora_apply_static_plan(y, c.x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, 4, 0, w.r, 1.0)
    torch.cuda.synchronize()
    assert sgmv_get_error(clear=True) == -6
    assert torch.equal(y, c.y0)
