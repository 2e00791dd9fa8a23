"""Seeded randomized GPU parity sweep of lora_apply through the C ABI.

Each case draws a dtype, a rank, hidden sizes (multiples of 8, often not of 64), a segment
table mixing one-row decode segments, empty segments, segments with no adapter (-1) and long
segments whose adapters repeat across non-adjacent segments (tensor-core groups), and the
launch options (tensor-core routing, long-batch geometry, two CTAs per SM, programmatic
overlap, column-slice views).  Every output row is compared with the fp64 oracle
(|y - y_ref| <= 1e-2 + 1e-2 |y_ref|); rows without an adapter and the elements outside a
slice must be bit-for-bit unchanged.  The draws are fixed by the seed, so a failure is
reproducible by its case index.  SGMV_FUZZ_CASES sets the number of cases (default 100).
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from segmented_gather_gemm_sgmv_gb300 import workloads  # noqa: E402
from tests import harness  # noqa: E402

pytestmark = pytest.mark.gpu

N_CASES = int(os.environ.get("SGMV_FUZZ_CASES", "100"))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    from segmented_gather_gemm_sgmv_gb300 import binding
    binding.lib()
    yield
    torch.cuda.synchronize()


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    dtype = ["f16", "bf16", "f32"][rng.integers(0, 3)]
    r = int(rng.choice([8, 16, 32, 64]))
    h_in = int(8 * rng.integers(4, 80))
    h_out = int(8 * rng.integers(4, 80))
    if rng.random() < 0.12:  # now and then a model-sized projection
        h_in = int(rng.choice([4096, 8192]))
        h_out = int(rng.choice([4096, 11008]))
    n_adapters = int(rng.integers(2, 9))
    lens, ids = [], []
    for _ in range(int(rng.integers(1, 24))):
        kind = rng.random()
        if kind < 0.45:
            lens.append(1)
        elif kind < 0.6:
            lens.append(int(rng.integers(2, 9)))
        elif kind < 0.68:
            lens.append(0)
        else:
            lens.append(int(rng.integers(20, 200)))
        ids.append(-1 if rng.random() < 0.08 else int(rng.integers(0, n_adapters)))
    opts = dict(tensor_cores=["auto", "always", "never"][rng.integers(0, 3)],
                long_batch=bool(rng.random() < 0.3), overlap_prior=bool(rng.random() < 0.5))
    if dtype == "f32" and opts["tensor_cores"] == "always":
        opts["tensor_cores"] = "auto"
    strided = bool(rng.random() < 0.35)
    return dtype, r, h_in, h_out, n_adapters, lens, ids, opts, strided


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_matches_oracle(i):
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    dtype, r, h_in, h_out, n_adapters, lens, ids, opts, strided = _draw(i)
    ss = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sa = np.asarray(ids, np.int32)
    w = workloads.Workload("fuzz", h_in, h_out, r, dtype, n_adapters, 2)
    c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 2, seed=i)
    layer = i % 2
    what = f"case {i}: {dtype} r{r} {h_in}->{h_out} lens={lens} ids={ids} {opts} strided={strided}"
    if strided:
        X = torch.zeros((c.M, h_in + 24), dtype=c.x.dtype, device="cuda")
        Y = torch.full((c.M, h_out + 40), 3.0, dtype=c.y0.dtype, device="cuda")
        X[:, 8:8 + h_in] = c.x
        Y[:, 16:16 + h_out] = c.y0
        Y0 = Y.clone()
        x, y = X[:, 8:8 + h_in], Y[:, 16:16 + h_out]
    else:
        x, y = c.x, c.y0.clone()
    # SGMV_DENSE_GRID (two CTAs of the call per SM) on a third of the cases, drawn apart so
    # that the other draws stay as they were
    opts = dict(opts, dense_grid=bool(np.random.default_rng(777 + i).random() < 0.3))
    what += f" dense={opts['dense_grid']}"
    lora_apply(y, x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, layer, r, w.scale, **opts)
    torch.cuda.synchronize()
    harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, layer), what)
    keep = harness.row_adapters(c.ss, c.sa, c.M) < 0
    idx = torch.as_tensor(np.nonzero(keep)[0], device="cuda")
    assert torch.equal(y[idx], c.y0[idx]), f"{what}: rows without an adapter were modified"
    if strided:
        outside = torch.ones_like(Y, dtype=torch.bool)
        outside[:, 16:16 + h_out] = False
        assert torch.equal(Y[outside], Y0[outside]), f"{what}: elements outside the slice changed"


@pytest.mark.parametrize("i", range(N_CASES // 2))
def test_random_unfused_case_matches_oracle(i):
    """sgmv_shrink then sgmv_expand on the same draws: v against the oracle's shrink, y against
    the oracle's expand of the library's v."""
    import oracle
    from segmented_gather_gemm_sgmv_gb300 import sgmv_expand, sgmv_shrink
    dtype, r, h_in, h_out, n_adapters, lens, ids, opts, strided = _draw(5000 + i)
    ss = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sa = np.asarray(ids, np.int32)
    w = workloads.Workload("fuzz_unfused", h_in, h_out, r, dtype, n_adapters, 2)
    c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 2, seed=i)
    layer = 1 - i % 2
    what = f"unfused case {i}: {dtype} r{r} {h_in}->{h_out} lens={lens} ids={ids} {opts}"
    keys = harness.touched(sa, ss)
    A = harness.oracle_blocks(c.A, keys, layer)
    B = harness.oracle_blocks(c.B, keys, layer)
    kw = dict(tensor_cores=opts["tensor_cores"], long_batch=opts["long_batch"])
    v = torch.full((c.M, r), -7.0, device="cuda")
    sgmv_shrink(v, c.x, c.A_ptrs, c.d_ss, c.d_sa, layer, r, **kw)
    v_ref = oracle.sgmv_shrink(np.full((c.M, r), -7.0), c.x.double().cpu().numpy(), A, ss, sa, 0)
    harness.assert_close(v.cpu().numpy(), v_ref, what + " shrink", atol=1e-3, rtol=1e-3)
    y = c.y0.clone()
    sgmv_expand(y, v, c.B_ptrs, c.d_ss, c.d_sa, layer, r, w.scale, **kw)
    y_ref = oracle.sgmv_expand(c.y0.double().cpu().numpy(), v.double().cpu().numpy(), B, ss, sa,
                               0, w.scale)
    harness.assert_close(y.float().cpu().numpy(), y_ref, what + " expand")


@pytest.mark.parametrize("i", range(N_CASES // 3))
def test_random_planned_case_matches_oracle(i):
    """The same draws through a plan (sgmv_plan, then lora_apply_planned with the draw's
    options): the row capacity is the row count exactly, and every row is checked."""
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_planned, sgmv_plan
    dtype, r, h_in, h_out, n_adapters, lens, ids, opts, strided = _draw(9000 + i)
    ss = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sa = np.asarray(ids, np.int32)
    w = workloads.Workload("fuzz_planned", h_in, h_out, r, dtype, n_adapters, 2)
    c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 2, seed=i)
    layer = i % 2
    what = f"planned case {i}: {dtype} r{r} {h_in}->{h_out} lens={lens} ids={ids} {opts}"
    plan = sgmv_plan(c.d_ss, c.d_sa, max(1, int(ss[-1])))
    y = c.y0.clone()
    opts = dict(opts, dense_grid=bool(np.random.default_rng(888 + i).random() < 0.5))
    what += f" dense={opts['dense_grid']}"
    lora_apply_planned(y, c.x, c.A_ptrs, c.B_ptrs, plan, layer, r, w.scale, **opts)
    torch.cuda.synchronize()
    harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, layer), what)
    keep = harness.row_adapters(c.ss, c.sa, c.M) < 0
    idx = torch.as_tensor(np.nonzero(keep)[0], device="cuda")
    assert torch.equal(y[idx], c.y0[idx]), f"{what}: rows without an adapter were modified"


@pytest.mark.parametrize("i", range(N_CASES // 4))
def test_random_base_case_matches_oracle(i):
    """lora_apply_base (base projection + LoRA term, written) on the draws' tables, 16-bit
    types and hidden sizes up to 640, against oracle.base_lora on every row."""
    import oracle
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_base
    dtype, r, h_in, h_out, n_adapters, lens, ids, opts, strided = _draw(12000 + i)
    rng = np.random.default_rng(77 + i)
    dtype = "bf16" if dtype == "f32" else dtype
    h_in, h_out = int(8 * rng.integers(4, 81)), int(8 * rng.integers(4, 81))
    ss = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sa = np.asarray(ids, np.int32)
    w = workloads.Workload("fuzz_base", h_in, h_out, r, dtype, n_adapters, 2)
    M = int(ss[-1]) + int(rng.integers(0, 40))  # rows after the last segment: base only
    c = harness.make_case(w, ss, sa, M=max(M, 1), seed=i)
    layer = i % 2
    g = torch.Generator(device="cuda")
    g.manual_seed(300 + i)
    W0 = ((torch.rand((h_out, h_in), generator=g, device="cuda") * 2 - 1) /
          np.sqrt(h_in)).to(c.x.dtype)
    y = torch.full((c.M, h_out), float("nan"), dtype=c.x.dtype, device="cuda")
    tc = "never" if opts["tensor_cores"] == "never" else "auto"
    lora_apply_base(y, c.x, W0, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, layer, r, w.scale,
                    tensor_cores=tc, overlap_prior=opts["overlap_prior"],
                    long_batch=opts["long_batch"])
    torch.cuda.synchronize()
    keys = harness.touched(sa, ss)
    A = harness.oracle_blocks(c.A, keys, layer)
    B = harness.oracle_blocks(c.B, keys, layer)
    ref = oracle.base_lora(c.x.double().cpu().numpy(), W0.double().cpu().numpy(), A, B, ss, sa,
                           0, w.scale)
    harness.assert_close(y.float().cpu().numpy(), ref,
                         f"base case {i}: {dtype} r{r} {h_in}->{h_out} M={c.M} lens={lens} "
                         f"ids={ids} {opts}")
