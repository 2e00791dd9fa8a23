"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on seeded inputs.

Named workloads at their full sizes (sampled rows where the oracle would be slow), custom
cases spanning several tiles and ragged tails, and the edge cases of the segment table.
Values: |y - y_ref| <= 1e-2 + 1e-2 |y_ref| elementwise; indices: bit-exact.
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


def _check_untouched(c, y):
    rows = harness.row_adapters(c.ss, c.sa, c.M)
    keep = torch.as_tensor(np.nonzero(rows < 0)[0], device=y.device)
    if keep.numel():
        assert torch.equal(y[keep], c.y0[keep]), "rows without an adapter were modified"


# ---------------------------------------------------------------- named workloads ----
def test_tiny_fp32():
    w = workloads.WORKLOADS["tiny"]
    for seed in range(4):
        ss, sa = workloads.make_segments("tiny", seed)
        c = harness.make_case(w, ss, sa, seed=seed)
        y = harness.run_apply(c, 0)
        ref = harness.oracle_apply(c, 0)
        harness.assert_close(y.cpu().numpy(), ref, f"tiny seed {seed}")
        harness.assert_close(y.cpu().numpy(), ref, f"tiny seed {seed} (fp32 bound)", atol=1e-4,
                             rtol=1e-5)


def test_decode_distinct_layers():
    w = workloads.WORKLOADS["decode_distinct"]
    ss, sa = workloads.make_segments(w.name, 0)
    c = harness.make_case(w, ss, sa)
    for layer in (0, 15, 31):
        y = harness.run_apply(c, layer)
        harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, layer),
                             f"{w.name} layer {layer}")


@pytest.mark.parametrize("name", ["decode_zipf", "decode_uniform", "decode_same"])
def test_decode_skewed(name):
    w = workloads.WORKLOADS[name]
    ss, sa = workloads.make_segments(name, 0)
    c = harness.make_case(w, ss, sa)
    for layer in (0, 8, 15):
        y = harness.run_apply(c, layer)
        harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, layer),
                             f"{name} layer {layer}")


def test_prefill_mixed_sampled():
    w = workloads.WORKLOADS["prefill_mixed"]
    ss, sa = workloads.make_segments(w.name, 0)
    c = harness.make_case(w, ss, sa)
    y = harness.run_apply(c, 0)
    rng = np.random.default_rng(5)
    rows = set(rng.choice(c.M, size=160, replace=False).tolist())
    for i in range(len(sa)):  # first and last rows of every segment, and 128-row tile edges
        rows.update({int(ss[i]), int(ss[i + 1]) - 1})
        rows.update(int(t) for t in range(ss[i] + 127, ss[i + 1], 128))
        rows.update(int(t) for t in range(ss[i] + 128, ss[i + 1], 128))
    rows, ref = harness.oracle_apply(c, 0, rows=rows)
    harness.assert_close(y[torch.as_tensor(rows, device=y.device)].float().cpu().numpy(), ref,
                         w.name)
    assert torch.isfinite(y.float()).all()


def test_mixed_70b_full_pool():
    w = workloads.WORKLOADS["mixed_70b"]
    ss, sa = workloads.make_segments(w.name, 0)
    c = harness.make_case(w, ss, sa)
    for layer in (0, 79):
        y = harness.run_apply(c, layer)
        harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, layer),
                             f"{w.name} layer {layer}")
    del c
    torch.cuda.empty_cache()


# ------------------------------------------------------------ shrink / expand ----
@pytest.mark.parametrize("dtype,r,h_in,h_out", [("f32", 8, 256, 256), ("f16", 16, 1024, 768),
                                                ("bf16", 64, 512, 1376), ("bf16", 32, 264, 136)])
def test_shrink_expand_and_fused(dtype, r, h_in, h_out):
    import oracle
    w = workloads.Workload("custom", h_in, h_out, r, dtype, 6, 3)
    rng = np.random.default_rng(7)
    ss, sa = workloads.random_segments(rng, 40, 12, 6, p_empty=0.15, first=3)
    c = harness.make_case(w, ss, sa, M=int(ss[-1]) + 5)
    from segmented_gather_gemm_sgmv_gb300 import sgmv_expand, sgmv_shrink
    layer = 2
    v = torch.full((c.M, r), -7.0, device="cuda")
    sgmv_shrink(v, c.x, c.A_ptrs, c.d_ss, c.d_sa, layer, r)
    keys = harness.touched(sa, ss)
    A = harness.oracle_blocks(c.A, keys, layer)
    B = harness.oracle_blocks(c.B, keys, layer)
    v_ref = oracle.sgmv_shrink(np.full((c.M, r), -7.0), c.x.double().cpu().numpy(), A, ss, sa, 0)
    harness.assert_close(v.cpu().numpy(), v_ref, "shrink", atol=1e-3, rtol=1e-3)
    y = c.y0.clone()
    sgmv_expand(y, v, c.B_ptrs, c.d_ss, c.d_sa, layer, r, w.scale)
    y_ref = oracle.sgmv_expand(c.y0.double().cpu().numpy(), v.double().cpu().numpy(), B, ss, sa,
                               0, w.scale)
    harness.assert_close(y.float().cpu().numpy(), y_ref, "expand")
    yf = harness.run_apply(c, layer)
    ref = harness.oracle_apply(c, layer)
    harness.assert_close(yf.float().cpu().numpy(), ref, "fused")
    harness.assert_close(y.float().cpu().numpy(), yf.float().cpu().numpy(),
                         "fused vs shrink+expand")
    _check_untouched(c, yf)


# ------------------------------------------------------------- index exactness ----
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_integer_exact(dtype):
    """x, A, B in {-1,0,1} with h_in <= 256: every partial sum is an exact integer, so a row
    processed twice, skipped or given the wrong adapter shows up bit-exactly."""
    dt = workloads.torch_dtype(dtype)
    r, h_in, h_out, n, L = 16, 256, 384, 9, 2
    w = workloads.Workload("int", h_in, h_out, r, dtype, n, L)
    rng = np.random.default_rng(11)
    ss, sa = workloads.random_segments(rng, 60, 20, n, p_empty=0.1)
    g = torch.Generator(device="cuda").manual_seed(3)
    A = torch.randint(-1, 2, (n, L, h_in, r), generator=g, device="cuda").to(dt)
    B = torch.randint(-1, 2, (n, L, r, h_out), generator=g, device="cuda").to(dt)
    c = harness.make_case(w, ss, sa, pool=(A, B))
    c.x = torch.randint(-1, 2, c.x.shape, generator=g, device="cuda").to(dt)
    c.y0 = torch.randint(-4, 5, c.y0.shape, generator=g, device="cuda").to(dt)
    for scale in (1.0, 2.0):
        c.w = dataclasses_replace(w, alpha=scale * r)
        for layer in (0, 1):
            y = harness.run_apply(c, layer)
            ref = harness.oracle_apply(c, layer)
            ref_t = torch.as_tensor(ref).to(dt)
            assert torch.equal(y.cpu(), ref_t), f"not bit-exact ({dtype}, scale {scale})"


def dataclasses_replace(w, **kw):
    import dataclasses
    return dataclasses.replace(w, **kw)


def test_adapter_tags():
    """A_k[:,0] = (k+1) e_0 and x[:,0] = 1 make v_0 = k+1; B_k row 0 = e_0, so
    y[t,0] - y_in[t,0] = scale (k(t)+1) names the adapter each row used."""
    r, h, n = 16, 512, 40
    w = workloads.Workload("tag", h, h, r, "bf16", n, 1)
    rng = np.random.default_rng(13)
    ss, sa = workloads.random_segments(rng, 200, 6, n, p_empty=0.05)
    A = torch.zeros((n, 1, h, r), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((n, 1, r, h), dtype=torch.bfloat16, device="cuda")
    for k in range(n):
        A[k, 0, 0, 0] = k + 1
    B[:, 0, 0, 0] = 1
    c = harness.make_case(w, ss, sa, pool=(A, B))
    c.x = torch.zeros_like(c.x)
    c.x[:, 0] = 1
    c.y0 = torch.zeros_like(c.y0)
    y = harness.run_apply(c, 0)
    want = np.zeros(c.M)
    for i, k in enumerate(sa):
        want[ss[i]:ss[i + 1]] = w.scale * (k + 1)
    assert np.array_equal(y[:, 0].float().cpu().numpy(), want)
    assert torch.count_nonzero(y[:, 1:]) == 0


def test_guard_rows_and_empty_segments():
    """NaN guard rows around the segments, empty segments and no-adapter segments stay
    bitwise untouched."""
    w = workloads.Workload("guard", 1024, 512, 32, "f16", 5, 1)
    ss = np.array([4, 9, 9, 30, 30, 31, 60], np.int32)
    sa = np.array([1, 3, -1, 0, 2, 1], np.int32)
    c = harness.make_case(w, ss, sa, M=68)
    c.y0[:4] = float("nan")
    c.y0[60:] = float("nan")
    y = harness.run_apply(c, 0)
    assert torch.isnan(y[:4]).all() and torch.isnan(y[60:]).all()
    assert torch.equal(y[9:30], c.y0[9:30])
    ref = harness.oracle_apply(c, 0)
    harness.assert_close(y[4:60].float().cpu().numpy(), ref[4:60], "guarded")


def test_no_segments_is_noop():
    w = workloads.Workload("empty", 256, 256, 16, "f16", 2, 1)
    c = harness.make_case(w, np.array([0, 1], np.int32), np.array([0], np.int32), M=4)
    y = c.y0.clone()
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    lora_apply(y, c.x, c.A_ptrs, c.B_ptrs, c.d_ss[:1], c.d_sa[:0], 0, 16, 1.0)
    assert torch.equal(y, c.y0)


@pytest.mark.parametrize("dtype,r", [("f16", 16), ("bf16", 64), ("f32", 32)])
def test_long_segments_and_repeats(dtype, r):
    """Segments longer than 1024 rows, ragged tails, and one adapter owning many
    non-adjacent segments (its rows are gathered into one group)."""
    w = workloads.Workload("long", 512, 640, r, dtype, 4, 1)
    lens = [1100, 1, 37, 1, 1, 300, 1, 9, 1030, 3]
    ids = [2, 0, 2, 1, 2, 3, 0, 2, 1, 2]
    ss = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    c = harness.make_case(w, ss, np.array(ids, np.int32))
    y = harness.run_apply(c, 0)
    rng = np.random.default_rng(3)
    rows = set(rng.choice(c.M, 300, replace=False).tolist())
    for i in range(len(ids)):
        rows.update({int(ss[i]), int(ss[i + 1]) - 1})
    rows, ref = harness.oracle_apply(c, 0, rows=rows)
    harness.assert_close(y[torch.as_tensor(rows, device="cuda")].float().cpu().numpy(), ref,
                         f"long {dtype}")


def test_deterministic():
    w = workloads.WORKLOADS["decode_zipf"]
    ss, sa = workloads.make_segments(w.name, 1)
    c = harness.make_case(w, ss, sa, num_adapters=128, layers=2)
    sa = np.minimum(sa, 127).astype(np.int32)
    c.sa, c.d_sa = sa, torch.as_tensor(sa, device="cuda")
    y1 = harness.run_apply(c, 1)
    y2 = harness.run_apply(c, 1)
    assert torch.equal(y1, y2)


# -------------------------------------------------------------------- validation ----
def test_validate_matches_oracle():
    import oracle
    from segmented_gather_gemm_sgmv_gb300 import sgmv_validate
    cases = [([0, 2, 2, 5], [0, 3, 1], 4, 5), ([0, 3, 2, 5], [0, 1, 1], 4, 5),
             ([-1, 2, 5], [0, 1], 4, 5), ([0, 2, 6], [0, 1], 4, 5), ([0, 2, 5], [0, 4], 4, 5),
             ([0, 2, 5], [-1, 3], 4, 5), ([0], [], 4, 0), ([1, 0, 9], [7, 0], 4, 5)]
    rng = np.random.default_rng(1)
    for _ in range(20):
        ss, sa = workloads.random_segments(rng, int(rng.integers(1, 700)), 5, 50)
        if rng.random() < 0.5:
            j = int(rng.integers(0, len(sa)))
            sa[j] = 50 + int(rng.integers(0, 3))
        if rng.random() < 0.5:
            j = int(rng.integers(1, len(ss)))
            ss[j] = ss[j - 1] - 1
        cases.append((ss.tolist(), sa.tolist(), 50, int(max(ss[-1], 0)) - int(rng.integers(0, 2))))
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for ss, sa, n, M in cases:
        d_ss = torch.tensor(ss, dtype=torch.int32, device="cuda")
        d_sa = torch.tensor(sa, dtype=torch.int32, device="cuda")
        sgmv_validate(d_ss, d_sa, n, M, d_err)
        assert int(d_err.item()) == oracle.validate(ss, sa, n, M), (ss[:8], sa[:8])


def test_bad_arguments_raise():
    from segmented_gather_gemm_sgmv_gb300 import SgmvError, lora_apply
    w = workloads.Workload("bad", 256, 256, 16, "f16", 2, 1)
    c = harness.make_case(w, np.array([0, 2], np.int32), np.array([1], np.int32))
    with pytest.raises(SgmvError) as e:
        lora_apply(c.y0.clone(), c.x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, 0, 12, 1.0)
    assert e.value.status == -3
    with pytest.raises(SgmvError) as e:
        lora_apply(c.y0.clone(), c.x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, -1, 16, 1.0)
    assert e.value.status == -1
    with pytest.raises(ValueError):
        lora_apply(c.y0.cpu(), c.x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, 0, 16, 1.0)


# ---------------------------------------------------------------- bounded waits ----
def test_wait_timeout_reports_and_recovers():
    """A wait on a barrier that nothing completes runs out after the configured bound; the
    kernel returns, the error word reads SGMV_ETIMEOUT, and the next call is correct."""
    from segmented_gather_gemm_sgmv_gb300 import sgmv_get_error, sgmv_set_wait_limit
    w = workloads.Workload("stall", 512, 512, 16, "f16", 3, 1)
    ss, sa = np.array([0, 3, 4, 9], np.int32), np.array([0, 2, 1], np.int32)
    c = harness.make_case(w, ss, sa)
    assert sgmv_get_error(clear=True) == 0
    sgmv_set_wait_limit(2_000_000, inject_stall=True)  # 2 ms
    try:
        y = harness.run_apply(c, 0)
        torch.cuda.synchronize()
    finally:
        sgmv_set_wait_limit(0, inject_stall=False)
    assert sgmv_get_error(clear=True) == -5
    assert torch.equal(y, c.y0), "a timed-out call must not write y"
    y = harness.run_apply(c, 0)
    harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, 0), "after timeout")
    assert sgmv_get_error(clear=True) == 0


# ------------------------------------------------------------- overlapped launches ----
@pytest.mark.parametrize("use_graph", [False, True])
def test_overlap_prior_chain(use_graph):
    """Back-to-back lora_apply_ex(SGMV_OVERLAP_PRIOR) calls where each call reads, as x, the y
    the previous call wrote: the prefetch may overlap the previous kernel, the activations may
    not.  Checked against the oracle applied in sequence."""
    import oracle
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    w = workloads.Workload("chain", 1024, 1024, 16, "f16", 24, 6)
    rng = np.random.default_rng(21)
    ss, sa = workloads.random_segments(rng, 40, 3, 24)
    c = harness.make_case(w, ss, sa)
    n = 6
    ys = [c.y0.clone() * 0.5 for _ in range(n)]
    x0 = c.x.clone()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())  # inputs made on the default stream

    def chain():
        x = x0
        for i in range(n):
            lora_apply(ys[i], x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, i, w.r, w.scale,
                       stream=stream, overlap_prior=True)
            x = ys[i]

    if use_graph:
        with torch.cuda.stream(stream):
            chain()  # uncaptured first calls set kernel attributes
        torch.cuda.synchronize()
        for i in range(n):
            ys[i].copy_(c.y0 * 0.5)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            chain()
        for i in range(n):
            ys[i].copy_(c.y0 * 0.5)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
    else:
        with torch.cuda.stream(stream):
            chain()
    torch.cuda.synchronize()
    keys = harness.touched(sa, ss)
    x = x0.double().cpu().numpy()
    for i in range(n):
        A = harness.oracle_blocks(c.A, keys, i)
        B = harness.oracle_blocks(c.B, keys, i)
        y_in = (c.y0 * 0.5).double().cpu().numpy()
        ref = oracle.lora_apply(y_in, x, A, B, ss, sa, 0, w.scale)
        harness.assert_close(ys[i].float().cpu().numpy(), ref, f"chain step {i}")
        x = ys[i].double().cpu().numpy()  # the next call reads what this one wrote


def test_max_segments():
    """num_segments = SGMV_MAX_SEGMENTS (4096 one-token segments; the large-table geometry)."""
    from segmented_gather_gemm_sgmv_gb300 import SgmvError, binding
    w = workloads.Workload("maxseg", 512, 256, 16, "bf16", 64, 1)
    rng = np.random.default_rng(9)
    S = binding.SGMV_MAX_SEGMENTS
    ss = np.arange(S + 1, dtype=np.int32)
    sa = rng.integers(-1, 64, size=S).astype(np.int32)
    c = harness.make_case(w, ss, sa)
    y = harness.run_apply(c, 0)
    harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, 0), "max segments")
    _check_untouched(c, y)
    ss2 = np.arange(S + 2, dtype=np.int32)
    sa2 = np.zeros(S + 1, np.int32)
    with pytest.raises(SgmvError) as e:
        from segmented_gather_gemm_sgmv_gb300 import lora_apply
        lora_apply(c.y0.clone(), c.x, c.A_ptrs, c.B_ptrs,
                   torch.as_tensor(ss2, device="cuda"), torch.as_tensor(sa2, device="cuda"), 0,
                   w.r, w.scale)
    assert e.value.status == -3


def test_tensor_role_wait_timeout_reports_and_recovers():
    """The bounded-wait path of the tensor-core role: long adapter groups (>= 64 rows, forced
    onto tcgen05), a barrier that nothing completes, a short bound.  The error word reads
    SGMV_ETIMEOUT, y is untouched, and the next call matches the oracle."""
    from segmented_gather_gemm_sgmv_gb300 import sgmv_get_error, sgmv_set_wait_limit
    for dtype, r, h_in, h_out in (("bf16", 64, 512, 640), ("f16", 16, 1024, 768)):
        w = workloads.Workload("stall_tc", h_in, h_out, r, dtype, 3, 2)
        ss = np.array([0, 150, 170, 420, 425], np.int32)
        sa = np.array([0, 2, 1, 0], np.int32)
        c = harness.make_case(w, ss, sa)
        assert sgmv_get_error(clear=True) == 0
        for long_batch in (False, True):
            sgmv_set_wait_limit(2_000_000, inject_stall=True)  # 2 ms
            try:
                y = harness.run_apply(c, 1, tensor_cores="always", long_batch=long_batch)
                torch.cuda.synchronize()
            finally:
                sgmv_set_wait_limit(0, inject_stall=False)
            assert sgmv_get_error(clear=True) == -5
            assert torch.equal(y, c.y0), "a timed-out call must not write y"
            y = harness.run_apply(c, 1, tensor_cores="always", long_batch=long_batch)
            harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, 1),
                                 f"{dtype} r={r} after timeout (long_batch={long_batch})")
            assert sgmv_get_error(clear=True) == 0


def test_validate_pointers_matches_oracle():
    """The pointer check flags null and misaligned weight pointers of the adapters a table
    uses, exactly as the oracle does.  The bad tables go to the validator only, never to a
    compute call."""
    import oracle
    from segmented_gather_gemm_sgmv_gb300 import sgmv_validate_pointers
    rng = np.random.default_rng(3)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for trial in range(30):
        n = int(rng.integers(1, 40))
        ss, sa = workloads.random_segments(rng, int(rng.integers(0, 300)), 4, n, p_empty=0.2)
        sa = np.where(rng.random(len(sa)) < 0.1, -1, sa).astype(np.int32)
        if len(sa) and rng.random() < 0.3:
            sa[int(rng.integers(0, len(sa)))] = n + 2  # past the pool: skipped here
        A = (0x7f0000000000 + 4096 * np.arange(n, dtype=np.uint64)).astype(np.uint64)
        B = (0x7f1000000000 + 4096 * np.arange(n, dtype=np.uint64)).astype(np.uint64)
        for arr in (A, B):
            for j in rng.choice(n, size=int(rng.integers(0, 3)), replace=True):
                arr[j] = 0 if rng.random() < 0.5 else arr[j] + np.uint64(8 * rng.integers(1, 2))
        use_a, use_b = [(True, True), (True, False), (False, True)][trial % 3]
        dA = torch.as_tensor(A.view(np.int64), device="cuda") if use_a else None
        dB = torch.as_tensor(B.view(np.int64), device="cuda") if use_b else None
        d_ss = torch.as_tensor(ss, device="cuda")
        d_sa = torch.as_tensor(sa, device="cuda")
        sgmv_validate_pointers(dA, dB, d_ss, d_sa, d_err)
        want = oracle.validate_pointers(A if use_a else None, B if use_b else None, ss, sa, n)
        assert int(d_err.item()) == want, (trial, int(d_err.item()), want)
