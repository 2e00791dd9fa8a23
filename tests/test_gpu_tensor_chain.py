"""GPU parity of the tensor role in chained launches (SGMV_OVERLAP_PRIOR), through the C ABI.

With the flag, the tensor role's loaders build their first row table and issue the weight
copies of each loader warp's first ring slot before the kernel waits for the previous kernel
of the stream, and copy that slot's activations (x or y rows) only after the wait.  These cases
make every call depend on the one before it -- it reads, as x, the y the previous call wrote, or
(unfused) the expand reads the v the shrink just wrote -- so an activation copied before the
wait would show as a wrong row.  Shapes include first m-tiles with fewer ring slots than loader
warps (h_in of two 64-column chunks), ragged chunks, both launch geometries, and expand-only
launches whose contiguous (m-tile, n-tile) ranges cross m-tiles.  Every call is compared with
the fp64 oracle given that call's actual inputs: |y - y_ref| <= 1e-2 + 1e-2 |y_ref|.
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


def _table(lens, ids):
    ss = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return ss, np.asarray(ids, np.int32)


# Three tensor groups (300 rows over two segments, 130, 64) and two CUDA-core groups (9, 1),
# one segment without an adapter.
CHAIN_LENS = [200, 9, 130, 64, 100, 1, 12]
CHAIN_IDS = [0, 3, 1, 2, 0, 4, -1]


@pytest.mark.parametrize("dtype,r,h,long_batch", [
    ("bf16", 64, 128, False),   # two K chunks: members with one shrink slot or none
    ("f16", 16, 256, True),
    ("bf16", 32, 1000, False),  # ragged K chunk and n-tile
    ("f16", 64, 2048, True),
])
def test_tensor_chain_reads_previous_output(dtype, r, h, long_batch):
    """Call i reads as x the y that call i - 1 wrote (h_in = h_out)."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    w = workloads.Workload("tc_chain", h, h, r, dtype, 5, 4)
    ss, sa = _table(CHAIN_LENS, CHAIN_IDS)
    c = harness.make_case(w, ss, sa, seed=7)
    n = 4
    y_init = [c.y0 * (0.5 + 0.25 * i) for i in range(n)]
    ys = [y.clone() for y in y_init]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())  # inputs made on the default stream
    with torch.cuda.stream(stream):
        x = c.x
        for i in range(n):
            lora_apply(ys[i], x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, i % w.layers, w.r,
                       w.scale, stream=stream, overlap_prior=True, tensor_cores="always",
                       long_batch=long_batch)
            x = ys[i]
    torch.cuda.synchronize()
    x = c.x
    for i in range(n):
        ref = harness.oracle_apply(c, i % w.layers, y_in=y_init[i], x=x)
        harness.assert_close(ys[i].float().cpu().numpy(), ref, f"call {i}")
        x = ys[i]


@pytest.mark.parametrize("dtype,r,h_in,h_out,long_batch", [
    ("bf16", 64, 1024, 4096, True),    # 10 m-tiles x 64 n-tiles over 144-152 expand units
    ("bf16", 64, 1024, 4096, False),
    ("f16", 16, 2048, 2048, False),
    ("f16", 32, 200, 4104, True),      # ragged K chunk and a ragged last n-tile
])
def test_tensor_shrink_then_expand_chain(dtype, r, h_in, h_out, long_batch):
    """sgmv_shrink writes v, then sgmv_expand (launched as its programmatic dependent) reads
    it: the expand's loaders prefetch B before the wait, and its epilogue reads v after."""
    from segmented_gather_gemm_sgmv_gb300 import sgmv_expand, sgmv_shrink
    w = workloads.Workload("tc_unfused", h_in, h_out, r, dtype, 5, 2)
    lens = [600, 300, 70, 10, 5, 200]
    ids = [0, 1, 2, 3, -1, 4]
    ss, sa = _table(lens, ids)
    c = harness.make_case(w, ss, sa, seed=11)
    layer = 1
    v = torch.full((c.M, r), float("nan"), dtype=torch.float32, device="cuda")
    y = c.y0.clone()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    kw = dict(stream=stream, overlap_prior=True, tensor_cores="always", long_batch=long_batch)
    with torch.cuda.stream(stream):
        for _ in range(2):  # the second pair follows a kernel of its own kind
            v.fill_(float("nan"))
            y.copy_(c.y0)
            sgmv_shrink(v, c.x, c.A_ptrs, c.d_ss, c.d_sa, layer, r, **kw)
            sgmv_expand(y, v, c.B_ptrs, c.d_ss, c.d_sa, layer, r, w.scale, **kw)
    torch.cuda.synchronize()
    keys = harness.touched(c.sa, c.ss)
    A = harness.oracle_blocks(c.A, keys, layer)
    B = harness.oracle_blocks(c.B, keys, layer)
    rows = harness.row_adapters(c.ss, c.sa, c.M) >= 0
    v_ref = oracle.sgmv_shrink(np.zeros((c.M, r)), c.x.double().cpu().numpy(), A, c.ss, c.sa, 0)
    v_gpu = v.double().cpu().numpy()
    harness.assert_close(v_gpu[rows], v_ref[rows], "v")
    # the expand given the library's own v (its rounding is not the expand's concern)
    y_ref = oracle.sgmv_expand(c.y0.double().cpu().numpy(), np.where(rows[:, None], v_gpu, 0.0),
                               B, c.ss, c.sa, 0, w.scale)
    harness.assert_close(y.float().cpu().numpy(), y_ref, "y")
    keep = torch.as_tensor(np.nonzero(~rows)[0], device="cuda")
    assert torch.equal(y[keep], c.y0[keep]), "rows without an adapter were modified"
