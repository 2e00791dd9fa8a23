"""GPU parity of plans (sgmv_plan) and the calls that read them: lora_apply_planned,
sgmv_shrink_planned, sgmv_expand_planned and the one-launch multi-projection lora_apply_multi.

- The plan itself (the adapter grouping) is integer work: compared bit for bit with the
  oracle's grouping.
- A planned call visits the same rows in the same order as the unplanned one, so with the same
  launch flags the two agree bit for bit; both are checked against the fp64 oracle
  (|y - y_ref| <= 1e-2 + 1e-2 |y_ref|).
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


def _plan(c, max_rows=None):
    from segmented_gather_gemm_sgmv_gb300 import sgmv_plan
    return sgmv_plan(c.d_ss, c.d_sa, c.M if max_rows is None else max_rows)


def _check_plan(plan, ss, sa, max_rows):
    want = oracle.plan(ss, sa, max_rows)
    got = plan.groups()
    assert (want is None) == (got is None)
    if want is not None:
        for w, g, name in zip(want, got, ("group starts", "group adapters", "rows")):
            assert np.array_equal(w, g), name


@pytest.mark.parametrize("name", ["tiny", "decode_distinct", "decode_zipf", "decode_uniform",
                                  "decode_same", "prefill_mixed", "mixed_70b"])
def test_plan_matches_oracle_grouping(name):
    from segmented_gather_gemm_sgmv_gb300 import sgmv_plan
    ss, sa = workloads.make_segments(name, 0)
    M = int(ss[-1])
    plan = sgmv_plan(torch.as_tensor(ss, device="cuda"), torch.as_tensor(sa, device="cuda"), M)
    _check_plan(plan, ss, sa, M)


def test_plan_random_tables_and_capacity():
    """Unsorted repeated adapters, empty segments, negative ids, tables up to the segment limit
    and a row capacity one short of the table (an invalid plan)."""
    from segmented_gather_gemm_sgmv_gb300 import binding, sgmv_plan
    rng = np.random.default_rng(7)
    for trial in range(30):
        S = int(rng.choice([1, 2, 31, 32, 33, 200, 1000, binding.SGMV_MAX_SEGMENTS]))
        ss, sa = workloads.random_segments(rng, S, int(rng.integers(1, 40)),
                                           int(rng.integers(1, 3 * S + 2)), p_empty=0.2,
                                           first=int(rng.integers(0, 5)))
        sa = np.where(rng.random(S) < 0.1, -1, sa).astype(np.int32)
        rows = int(sum(ss[i + 1] - ss[i] for i in range(S) if sa[i] >= 0))
        cap = rows if trial % 5 else max(rows - 1, 0)
        plan = sgmv_plan(torch.as_tensor(ss, device="cuda"), torch.as_tensor(sa, device="cuda"),
                         cap)
        _check_plan(plan, ss, sa, cap)


def test_planned_calls_equal_unplanned_and_oracle():
    """Mixed groups (long ones on the tensor cores, short ones on the CUDA cores), unsorted
    repeated adapters, empty segments, rows without an adapter: planned == unplanned bitwise,
    and both match the oracle, for the fused and the unfused forms, in both geometries."""
    from segmented_gather_gemm_sgmv_gb300 import (lora_apply, lora_apply_planned, sgmv_expand,
                                                  sgmv_expand_planned, sgmv_shrink,
                                                  sgmv_shrink_planned)
    lens = [70, 1, 64, 40, 300, 0, 23, 90, 5, 40, 7, 2, 1]
    ids = [1, 4, 3, 2, 0, 2, 2, 1, 5, 1, -1, 4, 0]
    ss = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sa = np.asarray(ids, np.int32)
    for dtype, r, h_in, h_out in (("bf16", 64, 512, 640), ("f16", 16, 1024, 768),
                                  ("f32", 32, 264, 136)):
        w = workloads.Workload("planned", h_in, h_out, r, dtype, 6, 3)
        c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 2)
        plan = _plan(c)
        for long_batch in (False, True):
            for tc in (("auto", "always") if dtype != "f32" else ("auto",)):
                y0 = harness.run_apply(c, 2, tensor_cores=tc, long_batch=long_batch)
                y1 = c.y0.clone()
                lora_apply_planned(y1, c.x, c.A_ptrs, c.B_ptrs, plan, 2, r, w.scale,
                                   tensor_cores=tc, long_batch=long_batch)
                assert torch.equal(y0, y1), (dtype, long_batch, tc)
                harness.assert_close(y1.float().cpu().numpy(), harness.oracle_apply(c, 2),
                                     f"planned {dtype} {tc} long={long_batch}")
                v0 = torch.zeros((c.M, r), device="cuda")
                v1 = torch.zeros((c.M, r), device="cuda")
                sgmv_shrink(v0, c.x, c.A_ptrs, c.d_ss, c.d_sa, 1, r, tensor_cores=tc,
                            long_batch=long_batch)
                sgmv_shrink_planned(v1, c.x, c.A_ptrs, plan, 1, r, tensor_cores=tc,
                                    long_batch=long_batch)
                assert torch.equal(v0, v1)
                ya, yb = c.y0.clone(), c.y0.clone()
                sgmv_expand(ya, v0, c.B_ptrs, c.d_ss, c.d_sa, 1, r, w.scale, tensor_cores=tc,
                            long_batch=long_batch)
                sgmv_expand_planned(yb, v1, c.B_ptrs, plan, 1, r, w.scale, tensor_cores=tc,
                                    long_batch=long_batch)
                assert torch.equal(ya, yb)
        keys = harness.touched(sa, ss)
        v_ref = oracle.sgmv_shrink(np.zeros((c.M, r)), c.x.double().cpu().numpy(),
                                   harness.oracle_blocks(c.A, keys, 1), ss, sa, 0)
        harness.assert_close(v1.cpu().numpy(), v_ref, f"planned shrink {dtype}", atol=1e-3,
                             rtol=1e-3)


def test_planned_layer_sweep_decode_distinct():
    """One plan reused by a CUDA graph of all 32 layers of decode_distinct (SGMV_OVERLAP_PRIOR,
    each call on its own x / y), every layer against the oracle."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_planned
    w = workloads.WORKLOADS["decode_distinct"]
    ss, sa = workloads.make_segments(w.name, 0)
    c = harness.make_case(w, ss, sa)
    plan = _plan(c)
    torch.cuda.synchronize()
    sets = [workloads.make_activations(w, c.M, "cuda", seed=70 + i) for i in range(w.layers)]
    ys = [y0.clone() for _, y0 in sets]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())  # inputs made on the default stream

    def sweep():
        for i, ((x, _), y) in enumerate(zip(sets, ys)):
            lora_apply_planned(y, x, c.A_ptrs, c.B_ptrs, plan, i, w.r, w.scale, stream=stream,
                               overlap_prior=True)

    with torch.cuda.stream(stream):
        sweep()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sweep()
    for (_, y0), y in zip(sets, ys):
        y.copy_(y0)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    for i, ((x, y0), y) in enumerate(zip(sets, ys)):
        harness.assert_close(y.float().cpu().numpy(),
                             harness.oracle_apply(c, i, y_in=y0, x=x), f"layer {i}")


def test_planned_prefill_and_70b():
    """The long-batch workloads through a plan: prefill_mixed every row, and mixed_70b (482
    unsorted segments: groups gathered from non-adjacent segments) at its first and last
    layers, every row."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_planned
    for name, layers in (("prefill_mixed", (0,)), ("mixed_70b", (0, 79))):
        w = workloads.WORKLOADS[name]
        ss, sa = workloads.make_segments(name, 0)
        c = harness.make_case(w, ss, sa)
        plan = _plan(c)
        for layer in layers:
            y = c.y0.clone()
            lora_apply_planned(y, c.x, c.A_ptrs, c.B_ptrs, plan, layer, w.r, w.scale,
                               long_batch=True, overlap_prior=True)
            harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, layer),
                                 f"{name} planned layer {layer}")
        del c, plan
        torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype,r,long_batch,dense", [("f16", 16, False, False),
                                                      ("bf16", 64, True, False),
                                                      ("f32", 8, False, False),
                                                      ("f16", 16, False, True),
                                                      ("bf16", 32, False, True)])
def test_multi_projection_one_launch(dtype, r, long_batch, dense):
    """q / k / v-like projections (h_out 1024, 256, 256; k and v on column slices of one fused
    output) and a gate-like one (h_out 2048) in one lora_apply_multi launch, each against the
    oracle.  (Each projection runs on a share of the grid, so the CUDA-core role may split its
    K sums differently from a solo call: equal within rounding, not bit for bit.)"""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_multi, lora_apply_planned
    rng = np.random.default_rng(31)
    ss, sa = workloads.random_segments(rng, 40, 6, 12, p_empty=0.1)
    sa[3] = -1
    ss[-1] = ss[-2] + 200  # one long segment: tensor-core groups where allowed
    M = int(ss[-1])
    shapes = [(512, 1024), (512, 256), (512, 256), (512, 2048)]
    cases = []
    for q, (h_in, h_out) in enumerate(shapes):
        w = workloads.Workload(f"proj{q}", h_in, h_out, r, dtype, 12, 2, alpha=8.0 + q)
        cases.append(harness.make_case(w, ss, sa, seed=10 * q, M=M))
    x = cases[0].x  # q, k, v and gate read the same activations
    kv = torch.zeros((M, 512), dtype=x.dtype, device="cuda")
    ys = [cases[0].y0.clone(), kv[:, 0:256], kv[:, 256:512], cases[3].y0.clone()]
    ys[1].copy_(cases[1].y0)
    ys[2].copy_(cases[2].y0)
    plan = _plan(cases[0], M)
    lora_apply_multi([(y, x, c.A_ptrs, c.B_ptrs, c.w.scale) for y, c in zip(ys, cases)], plan, 1,
                     r, long_batch=long_batch, dense_grid=dense)
    for q, (y, c) in enumerate(zip(ys, cases)):
        harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, 1, x=x),
                             f"multi projection {q}")
        solo = c.y0.clone()
        lora_apply_planned(solo, x, c.A_ptrs, c.B_ptrs, plan, 1, r, c.w.scale,
                           long_batch=long_batch)
        harness.assert_close(y.float().cpu().numpy(), solo.float().cpu().numpy(),
                             f"multi vs solo projection {q}")


def test_invalid_plans_report_and_leave_y():
    """A plan built with too small a row capacity, and a plan passed with the wrong
    num_segments, make the call return without writing y and set SGMV_EPLAN."""
    from segmented_gather_gemm_sgmv_gb300 import (lora_apply_planned, sgmv_get_error,
                                                  sgmv_plan)
    w = workloads.Workload("badplan", 256, 256, 16, "f16", 4, 1)
    ss, sa = np.array([0, 3, 4, 9], np.int32), np.array([0, 2, 1], np.int32)
    c = harness.make_case(w, ss, sa)
    assert sgmv_get_error(clear=True) == 0
    small = sgmv_plan(c.d_ss, c.d_sa, c.M - 1)
    y = c.y0.clone()
    lora_apply_planned(y, c.x, c.A_ptrs, c.B_ptrs, small, 0, w.r, w.scale)
    assert sgmv_get_error(clear=True) == -6
    assert torch.equal(y, c.y0)
    good = sgmv_plan(c.d_ss, c.d_sa, c.M)
    good.num_segments += 1  # a capacity that does not match the plan
    lora_apply_planned(y, c.x, c.A_ptrs, c.B_ptrs, good, 0, w.r, w.scale)
    assert sgmv_get_error(clear=True) == -6
    assert torch.equal(y, c.y0)
    good.num_segments -= 1
    lora_apply_planned(y, c.x, c.A_ptrs, c.B_ptrs, good, 0, w.r, w.scale)
    harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, 0), "valid plan")
    assert sgmv_get_error(clear=True) == 0
