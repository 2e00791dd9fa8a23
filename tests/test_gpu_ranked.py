"""GPU parity of lora_apply_ranked: a rank and a scale of its own for every adapter, adapters
of ranks 8..64 in one call, on the CUDA cores and the tensor cores, with the segment table or a
plan, against the fp64 oracle (|y - y_ref| <= 1e-2 + 1e-2 |y_ref|; integer-valued inputs bit for
bit)."""
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


class RankedPool:
    """Adapter k of rank ranks[k]: its own [L][h_in][r_k] and [L][r_k][h_out] blocks."""

    def __init__(self, ranks, h_in, h_out, L, dtype, seed, integer=False):
        dt = workloads.torch_dtype(dtype)
        g = torch.Generator(device="cuda").manual_seed(seed)
        self.A, self.B = [], []
        for r in ranks:
            if integer:
                a = torch.randint(-1, 2, (L, h_in, r), generator=g, device="cuda").to(dt)
                b = torch.randint(-1, 2, (L, r, h_out), generator=g, device="cuda").to(dt)
            else:
                a = ((torch.rand((L, h_in, r), generator=g, device="cuda") * 2 - 1)
                     / np.sqrt(h_in)).to(dt)
                b = (torch.randn((L, r, h_out), generator=g, device="cuda") / np.sqrt(r)).to(dt)
            self.A.append(a)
            self.B.append(b)
        self.A_ptrs = torch.tensor([a.data_ptr() for a in self.A], dtype=torch.int64,
                                   device="cuda")
        self.B_ptrs = torch.tensor([b.data_ptr() for b in self.B], dtype=torch.int64,
                                   device="cuda")

    def blocks(self, layer, keys):
        A = [a[layer:layer + 1].double().cpu().numpy() if k in keys else None
             for k, a in enumerate(self.A)]
        B = [b[layer:layer + 1].double().cpu().numpy() if k in keys else None
             for k, b in enumerate(self.B)]
        return A, B


def _run(pool, ranks, scales, x, y0, ss, sa, layer, r_max, plan=None, **kw):
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_ranked
    y = y0.clone()
    d_rank = torch.tensor(ranks, dtype=torch.int32, device="cuda")
    d_scale = torch.tensor(scales, dtype=torch.float32, device="cuda")
    if plan is None:
        lora_apply_ranked(y, x, pool.A_ptrs, pool.B_ptrs, d_rank, d_scale, layer, r_max,
                          seg_starts=torch.as_tensor(ss, device="cuda"),
                          seg_adapter=torch.as_tensor(sa, device="cuda"), **kw)
    else:
        lora_apply_ranked(y, x, pool.A_ptrs, pool.B_ptrs, d_rank, d_scale, layer, r_max,
                          plan=plan, **kw)
    return y


def _ref(pool, ranks, scales, x, y0, ss, sa, layer):
    keys = harness.touched(sa, ss)
    A, B = pool.blocks(layer, keys)
    return oracle.lora_apply_ranked(y0.double().cpu().numpy(), x.double().cpu().numpy(), A, B,
                                    ranks, scales, ss, sa, 0)


# decode rows (CUDA-core items) and long groups (tensor role where allowed), ranks mixed
LENS = [1, 1, 200, 3, 90, 1, 2, 0, 130, 4]
IDS = [0, 1, 2, 3, 4, 5, 0, 6, 7, 2]


@pytest.mark.parametrize("dtype,r_max,ranks", [
    ("bf16", 64, [8, 16, 64, 32, 16, 64, 8, 48, 24]),
    ("f16", 32, [16, 8, 32, 24, 16, 32, 8, 8, 24]),
    ("f32", 64, [8, 64, 40, 16, 56, 8, 32, 24, 8]),
])
@pytest.mark.parametrize("tensor_cores", ["auto", "always", "never"])
@pytest.mark.parametrize("long_batch", [False, True])
def test_mixed_ranks_match_oracle(dtype, r_max, ranks, tensor_cores, long_batch):
    if dtype == "f32" and tensor_cores == "always":
        pytest.skip("no tensor role for fp32")
    h_in, h_out, L = 512, 640, 2
    ss = np.concatenate([[0], np.cumsum(LENS)]).astype(np.int32)
    sa = np.asarray(IDS, np.int32)
    pool = RankedPool(ranks, h_in, h_out, L, dtype, seed=3)
    scales = [16.0 / r for r in ranks]
    w = workloads.Workload("ranked", h_in, h_out, r_max, dtype, len(ranks), L)
    x, y0 = workloads.make_activations(w, int(ss[-1]) + 2, "cuda", seed=9)
    y = _run(pool, ranks, scales, x, y0, ss, sa, 1, r_max, tensor_cores=tensor_cores,
             long_batch=long_batch)
    harness.assert_close(y.float().cpu().numpy(), _ref(pool, ranks, scales, x, y0, ss, sa, 1),
                         f"ranked {dtype} {tensor_cores} long={long_batch}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("tensor_cores", ["always", "never"])
def test_mixed_ranks_integer_exact(dtype, tensor_cores):
    """x, A, B in {-1, 0, 1}, h_in <= 256, integer scales: every partial sum is exact, so both
    roles equal the oracle bit for bit -- a wrong rank, stride or layer offset shows."""
    h_in, h_out, L = 256, 320, 2
    ranks = [8, 64, 16, 32, 24, 64, 8, 40, 16]
    ss = np.concatenate([[0], np.cumsum(LENS)]).astype(np.int32)
    sa = np.asarray(IDS, np.int32)
    pool = RankedPool(ranks, h_in, h_out, L, dtype, seed=5, integer=True)
    scales = [1.0, 2.0, 1.0, 1.0, 2.0, 1.0, 1.0, 2.0, 1.0]
    dt = workloads.torch_dtype(dtype)
    g = torch.Generator(device="cuda").manual_seed(6)
    M = int(ss[-1])
    x = torch.randint(-1, 2, (M, h_in), generator=g, device="cuda").to(dt)
    y0 = torch.randint(-4, 5, (M, h_out), generator=g, device="cuda").to(dt)
    y = _run(pool, ranks, scales, x, y0, ss, sa, 1, 64, tensor_cores=tensor_cores)
    ref = torch.as_tensor(_ref(pool, ranks, scales, x, y0, ss, sa, 1)).to(dt)
    assert torch.equal(y.cpu(), ref)


def test_uniform_ranks_equal_lora_apply_bitwise():
    """Every rank = r_max and every scale = scale: the ranked call is lora_apply bit for bit
    (CUDA-core and tensor-core groups)."""
    w = workloads.Workload("uniform", 512, 640, 32, "bf16", 8, 2)
    ss = np.concatenate([[0], np.cumsum(LENS)]).astype(np.int32)
    sa = np.asarray(IDS, np.int32)
    c = harness.make_case(w, ss, sa)
    from segmented_gather_gemm_sgmv_gb300 import lora_apply_ranked
    for tc in ("auto", "always", "never"):
        y0 = harness.run_apply(c, 1, tensor_cores=tc)
        y1 = c.y0.clone()
        lora_apply_ranked(y1, c.x, c.A_ptrs, c.B_ptrs,
                          torch.full((8,), 32, dtype=torch.int32, device="cuda"),
                          torch.full((8,), w.scale, dtype=torch.float32, device="cuda"), 1, 32,
                          seg_starts=c.d_ss, seg_adapter=c.d_sa, tensor_cores=tc)
        assert torch.equal(y0, y1), tc


def test_ranked_with_plan_and_invalid_rank():
    """The plan form matches the table form bit for bit; an adapter whose rank entry is not a
    multiple of 8 in [8, r_max] is skipped (its rows unchanged bit for bit)."""
    from segmented_gather_gemm_sgmv_gb300 import sgmv_plan
    ranks = [8, 16, 64, 32, 16, 64, 8, 48, 24]
    h_in, h_out, L = 512, 640, 2
    ss = np.concatenate([[0], np.cumsum(LENS)]).astype(np.int32)
    sa = np.asarray(IDS, np.int32)
    pool = RankedPool(ranks, h_in, h_out, L, "bf16", seed=4)
    scales = [16.0 / r for r in ranks]
    w = workloads.Workload("ranked_plan", h_in, h_out, 64, "bf16", len(ranks), L)
    M = int(ss[-1])
    x, y0 = workloads.make_activations(w, M, "cuda", seed=12)
    plan = sgmv_plan(torch.as_tensor(ss, device="cuda"), torch.as_tensor(sa, device="cuda"), M)
    for tc in ("auto", "always", "never"):
        a = _run(pool, ranks, scales, x, y0, ss, sa, 0, 64, tensor_cores=tc)
        b = _run(pool, ranks, scales, x, y0, ss, sa, 0, 64, plan=plan, tensor_cores=tc)
        assert torch.equal(a, b), tc
    bad = list(ranks)
    bad[2] = 12   # adapter 2 (the 200-row and the 4-row segments): not a multiple of 8
    bad[4] = 128  # adapter 4: above r_max
    y = _run(pool, bad, scales, x, y0, ss, sa, 0, 64)
    rows = harness.row_adapters(ss, sa, M)
    skip = torch.as_tensor(np.nonzero((rows == 2) | (rows == 4))[0], device="cuda")
    assert torch.equal(y[skip], y0[skip])
    good = [k for k in range(len(ranks)) if k not in (2, 4)]
    sa_good = np.where(np.isin(sa, good), sa, -1).astype(np.int32)
    harness.assert_close(y.float().cpu().numpy(),
                         _ref(pool, ranks, scales, x, y0, ss, sa_good, 0), "valid adapters")
