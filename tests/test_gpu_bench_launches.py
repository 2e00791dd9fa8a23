"""GPU parity of exactly the launches that bench.py times, at the workloads' full sizes.

bench.py replays a CUDA graph of back-to-back lora_apply calls, each on its own x / y buffer set
and layer, launched with SGMV_OVERLAP_PRIOR (each kernel may stream weights while the previous
one runs), and adds SGMV_LONG_BATCH for the workloads that hold prefill segments.  These tests
capture the same kind of graph (same flags, same workload tables, same pools) and compare EVERY
row of every call with the fp64 oracle: |y - y_ref| <= 1e-2 + 1e-2 |y_ref| elementwise.
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


def run_chain(c, layers, long_batch, seed=40, dense_grid=False):
    """Back-to-back calls in one CUDA graph, as bench.py times them: call i works on its own
    (x_i, y_i) at layers[i], with SGMV_OVERLAP_PRIOR (+ SGMV_LONG_BATCH).  Returns the inputs and
    outputs of every call."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    sets = [workloads.make_activations(c.w, c.M, "cuda", seed=seed + i) for i in range(len(layers))]
    ys = [y0.clone() for _, y0 in sets]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())  # inputs made on the default stream

    def chain():
        for (x, _), y, layer in zip(sets, ys, layers):
            lora_apply(y, x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, layer, c.w.r, c.w.scale,
                       stream=stream, overlap_prior=True, long_batch=long_batch,
                       dense_grid=dense_grid)

    with torch.cuda.stream(stream):
        chain()  # uncaptured first calls set the kernels' attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        chain()
    for (_, y0), y in zip(sets, ys):
        y.copy_(y0)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    return sets, ys


def check_chain(c, layers, sets, ys, what):
    for i, ((x, y0), y, layer) in enumerate(zip(sets, ys, layers)):
        ref = harness.oracle_apply(c, layer, y_in=y0, x=x)
        harness.assert_close(y.float().cpu().numpy(), ref, f"{what} call {i} (layer {layer})")
        rows = harness.row_adapters(c.ss, c.sa, c.M)
        keep = torch.as_tensor(np.nonzero(rows < 0)[0], device=y.device)
        if keep.numel():
            assert torch.equal(y[keep], y0[keep]), f"{what}: rows without an adapter changed"


def test_decode_distinct_overlap_chain_full_size():
    """The headline launch: decode_distinct (h=4096, r=16, fp16, 64 one-token segments, 64
    adapters x 32 layers), chained with SGMV_OVERLAP_PRIOR, first and last layers."""
    w = workloads.WORKLOADS["decode_distinct"]
    ss, sa = workloads.make_segments(w.name, 0)
    c = harness.make_case(w, ss, sa)
    layers = [0, 31, 0, 31]
    sets, ys = run_chain(c, layers, long_batch=False)
    check_chain(c, layers, sets, ys, w.name)


# decode_zipf and decode_uniform are timed with SGMV_DENSE_GRID (two CTAs of a call per SM: many
# rows over many adapter groups); decode_same without it.  Both forms are checked for all three.
@pytest.mark.parametrize("dense", [False, True])
@pytest.mark.parametrize("name", ["decode_zipf", "decode_uniform", "decode_same"])
def test_decode_skewed_overlap_chain_full_size(name, dense):
    w = workloads.WORKLOADS[name]
    ss, sa = workloads.make_segments(name, 0)
    c = harness.make_case(w, ss, sa)
    layers = [0, 15, 7]
    sets, ys = run_chain(c, layers, long_batch=False, dense_grid=dense)
    check_chain(c, layers, sets, ys, f"{name} dense={dense}")


def test_prefill_mixed_long_batch_every_row():
    """prefill_mixed (4096 -> 11008, r=64, bf16, 8 segments of 128..1024 rows) in the timed
    launch: SGMV_LONG_BATCH (one CTA per SM, the 416-thread kernel for <= 64 segments) with
    SGMV_OVERLAP_PRIOR; every one of the ~3450 rows of both calls against the oracle."""
    w = workloads.WORKLOADS["prefill_mixed"]
    ss, sa = workloads.make_segments(w.name, 0)
    c = harness.make_case(w, ss, sa)
    layers = [0, 0]
    sets, ys = run_chain(c, layers, long_batch=True)
    check_chain(c, layers, sets, ys, w.name + " long batch")


def test_prefill_mixed_default_geometry_every_row():
    w = workloads.WORKLOADS["prefill_mixed"]
    ss, sa = workloads.make_segments(w.name, 0)
    c = harness.make_case(w, ss, sa)
    y = harness.run_apply(c, 0)
    harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, 0),
                         w.name + " default geometry")


def test_mixed_70b_long_batch_layers():
    """mixed_70b (h=8192, r=64, bf16; 2 x 16 prefill rows + 480 decode rows, unsorted Zipf ids
    over 256 adapters x 80 layers, 43 GB pool) in the timed launch (SGMV_LONG_BATCH +
    SGMV_OVERLAP_PRIOR), layers 0, 40 and 79, every row."""
    w = workloads.WORKLOADS["mixed_70b"]
    ss, sa = workloads.make_segments(w.name, 0)
    c = harness.make_case(w, ss, sa)
    layers = [0, 40, 79]
    sets, ys = run_chain(c, layers, long_batch=True)
    check_chain(c, layers, sets, ys, w.name + " long batch")
    del c, sets, ys
    torch.cuda.empty_cache()


@pytest.mark.parametrize("long_batch", [True, False])
def test_prefill_mixed_unfused_pair_every_row(long_batch):
    """The bench's unfused leg at full size: sgmv_shrink into v, then sgmv_expand from it, both
    with SGMV_OVERLAP_PRIOR on one stream (the expand reads the v the shrink just wrote).  The
    shrink-only routing sends every prefill group (142-891 rows, rank 64) to the tensor role.
    v is compared with the oracle's shrink, y with the oracle's expand of the library's v."""
    import oracle
    from segmented_gather_gemm_sgmv_gb300 import sgmv_expand, sgmv_shrink
    w = workloads.WORKLOADS["prefill_mixed"]
    ss, sa = workloads.make_segments(w.name, 0)
    c = harness.make_case(w, ss, sa, seed=5)
    v = torch.full((c.M, w.r), float("nan"), dtype=torch.float32, device="cuda")
    y = c.y0.clone()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    kw = dict(stream=stream, overlap_prior=True, long_batch=long_batch)
    with torch.cuda.stream(stream):
        sgmv_shrink(v, c.x, c.A_ptrs, c.d_ss, c.d_sa, 0, w.r, **kw)
        sgmv_expand(y, v, c.B_ptrs, c.d_ss, c.d_sa, 0, w.r, w.scale, **kw)
    torch.cuda.synchronize()
    keys = harness.touched(c.sa, c.ss)
    rows = harness.row_adapters(c.ss, c.sa, c.M) >= 0
    v_gpu = v.double().cpu().numpy()
    v_ref = oracle.sgmv_shrink(np.zeros((c.M, w.r)), c.x.double().cpu().numpy(),
                               harness.oracle_blocks(c.A, keys, 0), c.ss, c.sa, 0)
    harness.assert_close(v_gpu[rows], v_ref[rows], "v")
    y_ref = oracle.sgmv_expand(c.y0.double().cpu().numpy(), np.where(rows[:, None], v_gpu, 0.0),
                               harness.oracle_blocks(c.B, keys, 0), c.ss, c.sa, 0, w.scale)
    harness.assert_close(y.float().cpu().numpy(), y_ref, "y")
