"""GPU parity for adapter groups of 16 to 511 rows, the band between one-token decode rows and
prefill tiles, on both routes: the library's own rule (these groups stay on the CUDA cores at
these shapes) and SGMV_TENSOR_CORES_ALWAYS (groups of 64 rows and more on tcgen05, so 63 and
64 sit on either side of the tile threshold and 127/255/511 leave a ragged last m-tile).

Each table puts the group's rows in three segments that are not adjacent (another adapter's
rows and a row without an adapter sit between them) plus single-row segments of other
adapters, and every row is compared with the fp64 oracle:
|y - y_ref| <= 1e-2 + 1e-2 |y_ref|; rows without an adapter stay bit-identical.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from segmented_gather_gemm_sgmv_gb300 import workloads  # noqa: E402
from tests import harness  # noqa: E402

pytestmark = pytest.mark.gpu

SIZES = [16, 63, 64, 127, 255, 256, 511]


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


def group_table(n, seed):
    """Adapter 3 owns n rows in three pieces; adapters 0-2 and 4-5 own single rows between
    and after them; one row has no adapter."""
    rng = np.random.default_rng(seed)
    a = int(rng.integers(1, max(2, n // 2)))
    b = int(rng.integers(1, max(2, n - a)))
    pieces = [a, b, n - a - b]
    lens, ids = [], []
    for j, p in enumerate(pieces):
        if p > 0:
            lens.append(p)
            ids.append(3)
        lens += [1, 1]
        ids += [j % 3, -1 if j == 1 else 4 + (j % 2)]
    starts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return starts, np.asarray(ids, np.int32)


@pytest.mark.parametrize("tc", ["auto", "always"])
@pytest.mark.parametrize("dtype,r", [("f16", 16), ("bf16", 16), ("f16", 64), ("bf16", 64)])
@pytest.mark.parametrize("n", SIZES)
def test_group_of_n_rows(n, dtype, r, tc):
    from segmented_gather_gemm_sgmv_gb300 import lora_apply
    w = workloads.Workload(f"group_{n}", 512, 640, r, dtype, 6, 2)
    ss, sa = group_table(n, seed=n + r)
    c = harness.make_case(w, ss, sa, seed=n)
    y = c.y0.clone()
    lora_apply(y, c.x, c.A_ptrs, c.B_ptrs, c.d_ss, c.d_sa, 1, r, w.scale, tensor_cores=tc)
    torch.cuda.synchronize()
    harness.assert_close(y.float().cpu().numpy(), harness.oracle_apply(c, 1),
                         f"group of {n} rows, {dtype}, r={r}, tensor cores {tc}")
    rows = harness.row_adapters(c.ss, c.sa, c.M)
    keep = torch.as_tensor(np.nonzero(rows < 0)[0], device="cuda")
    if keep.numel():
        assert torch.equal(y[keep], c.y0[keep])
