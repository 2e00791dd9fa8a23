"""GPU tests of the adapter pool (sgmv_pool_*): adapters copied host -> device on demand into a
fixed number of slots, least-recently-used eviction of slots no unreleased batch reads, copies
on their own stream overlapped with the compute of the batch before; every batch's lora_apply
result against the fp64 oracle over the full adapter set."""
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


W = workloads.Workload("paged", 512, 384, 16, "f16", 16, 3)


def _host_adapters(n, seed):
    """n adapters' [L][h_in][r] / [L][r][h_out] blocks in pinned host memory."""
    A, B = workloads.make_pool(W, "cuda", seed=seed, num_adapters=n)
    hA = [A[k].cpu().contiguous().pin_memory() for k in range(n)]
    hB = [B[k].cpu().contiguous().pin_memory() for k in range(n)]
    return A, B, hA, hB


def _oracle_batch(A, B, x, y0, ss, sa, layer):
    import oracle
    keys = harness.touched(sa, ss)
    Ab = harness.oracle_blocks(A, keys, layer)
    Bb = harness.oracle_blocks(B, keys, layer)
    return oracle.lora_apply(y0.double().cpu().numpy(), x.double().cpu().numpy(), Ab, Bb, ss, sa,
                             0, W.scale)


def test_paged_batches_match_oracle_and_evict_lru():
    """Twelve batches drawn from 16 adapters through a 6-slot pool: each batch acquires, runs,
    releases; results against the oracle; the pool copies exactly the adapters it lacks."""
    from segmented_gather_gemm_sgmv_gb300 import AdapterPool, lora_apply
    n = 16
    A, B, hA, hB = _host_adapters(n, seed=1)
    pool = AdapterPool(6, n, W.layers, W.h_in, W.h_out, W.r, torch.float16)
    for k in range(n):
        pool.register(k, hA[k], hB[k])
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    rng = np.random.default_rng(3)
    resident = []  # LRU order, as the pool keeps it
    for b in range(12):
        ids = rng.choice(n, size=int(rng.integers(1, 7)), replace=False)
        ss, sa = workloads.random_segments(rng, 10, 3, 1)
        sa = rng.choice(ids, size=10).astype(np.int32)
        sa[0] = -1
        c = harness.make_case(W, ss, sa, pool=(A, B), seed=b)
        copied = pool.acquire(sa, copy_s, comp_s)
        want = list(dict.fromkeys(int(k) for k in sa if k >= 0))  # first-use order
        hits = [k for k in want if k in resident]
        misses = [k for k in want if k not in resident]
        assert copied == len(misses), (b, copied, misses)
        # the pool's LRU order after the batch: the others (oldest evicted first), then the
        # batch's hits, then its misses
        others = [k for k in resident if k not in hits]
        evicted = max(0, len(others) + len(want) - 6)
        resident = others[evicted:] + hits + misses
        y = c.y0.clone()
        comp_s.wait_stream(torch.cuda.current_stream())  # x, y made on the default stream
        with torch.cuda.stream(comp_s):
            lora_apply(y, c.x, pool.A_ptrs, pool.B_ptrs, c.d_ss, c.d_sa, b % W.layers, W.r,
                       W.scale, stream=comp_s)
        pool.release(sa, comp_s)
        comp_s.synchronize()
        harness.assert_close(y.float().cpu().numpy(),
                             _oracle_batch(A, B, c.x, c.y0, ss, sa, b % W.layers), f"batch {b}")
    st = pool.stats()
    assert st["resident"] == 6 and st["misses"] >= 6
    pool.close()


def test_overlapped_batches_without_host_waits():
    """Batch i+1's acquire (and its copies) is enqueued while batch i still computes: no host
    synchronisation between batches; every batch's output checked at the end."""
    from segmented_gather_gemm_sgmv_gb300 import AdapterPool, lora_apply
    n = 12
    A, B, hA, hB = _host_adapters(n, seed=2)
    pool = AdapterPool(8, n, W.layers, W.h_in, W.h_out, W.r, torch.float16)
    for k in range(n):
        pool.register(k, hA[k], hB[k])
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    rng = np.random.default_rng(8)
    runs = []
    for b in range(10):
        ids = rng.choice(n, size=4, replace=False)
        ss = np.arange(0, 4 * 24 + 1, 24, dtype=np.int32)
        sa = ids.astype(np.int32)
        c = harness.make_case(W, ss, sa, pool=(A, B), seed=40 + b)
        try:
            pool.acquire(sa, copy_s, comp_s)
        except Exception as e:  # too few idle slots while earlier batches still run
            assert "SGMV_ENOSPACE" in str(e)
            comp_s.synchronize()
            pool.acquire(sa, copy_s, comp_s)
        y = c.y0.clone()
        comp_s.wait_stream(torch.cuda.current_stream())  # x, y made on the default stream
        lora_apply(y, c.x, pool.A_ptrs, pool.B_ptrs, c.d_ss, c.d_sa, 1, W.r, W.scale,
                   stream=comp_s)
        pool.release(sa, comp_s)
        runs.append((c, ss, sa, y))
    torch.cuda.synchronize()
    for b, (c, ss, sa, y) in enumerate(runs):
        harness.assert_close(y.float().cpu().numpy(), _oracle_batch(A, B, c.x, c.y0, ss, sa, 1),
                             f"overlapped batch {b}")
    pool.close()


def test_pins_space_and_reregistration():
    """Pinned (acquired, unreleased) slots are never evicted: a batch that needs more slots
    than are free fails with SGMV_ENOSPACE and changes nothing; re-registering a pinned adapter
    fails with SGMV_EBUSY; after release both succeed and the new weights are copied."""
    from segmented_gather_gemm_sgmv_gb300 import AdapterPool, SgmvError, lora_apply
    n = 8
    A, B, hA, hB = _host_adapters(n, seed=4)
    pool = AdapterPool(4, n, W.layers, W.h_in, W.h_out, W.r, torch.float16)
    for k in range(n):
        pool.register(k, hA[k], hB[k])
    s = torch.cuda.current_stream()
    assert pool.acquire([0, 1, 2], s, s) == 3
    with pytest.raises(SgmvError) as e:
        pool.acquire([3, 4], s, s)           # one free slot
    assert e.value.status == -7
    with pytest.raises(SgmvError) as e:
        pool.acquire(list(range(5)), s, s)   # more adapters than slots
    assert e.value.status == -7
    assert pool.acquire([3], s, s) == 1      # the one free slot
    with pytest.raises(SgmvError) as e:
        pool.register(1, hB[1], hA[1])
    assert e.value.status == -8
    pool.release([0, 1, 2, 3], s)
    torch.cuda.synchronize()
    # new weights for adapter 1 (negated): the next acquire copies them
    nA, nB = (-A[1]).cpu().contiguous().pin_memory(), B[1].cpu().contiguous().pin_memory()
    pool.register(1, nA, nB)
    assert pool.acquire([1, 4, 5], s, s) == 3
    ss, sa = np.array([0, 3, 5, 9], np.int32), np.array([1, 4, 5], np.int32)
    A2 = A.clone()
    A2[1] = -A[1]
    c = harness.make_case(W, ss, sa, pool=(A2, B), seed=7)
    y = c.y0.clone()
    lora_apply(y, c.x, pool.A_ptrs, pool.B_ptrs, c.d_ss, c.d_sa, 2, W.r, W.scale)
    pool.release(sa, s)
    harness.assert_close(y.float().cpu().numpy(), _oracle_batch(A2, B, c.x, c.y0, ss, sa, 2),
                         "after re-registration")
    pool.close()
