"""Pins that tie the fp64 oracle to things other than itself.

Each check takes an oracle binding (``oracle.OracleLib``) and raises AssertionError when the
oracle disagrees with what "Punica Guide: Multi-Tenant LoRA Serving with SGMV" and plain linear
algebra fix.  The pins (closed forms, numpy matmuls on a separate code path, invariants, brute
force, a hand-worked example) are chosen so that a plausible slip anywhere in the oracle -- a
dropped term, a wrong sign, scale or index, a transposed operand, a wrong layer or adapter --
trips at least one of them; tests/test_oracle_mutations.py plants such slips to prove it.

Sources: section "The Heterogeneous Batching Bottleneck" (y_i = x_i W0 + (alpha/r) x_i A B,
A: d_in x r, B: r x d_out); section "The SGMV Mathematical Formulation" (segments, pointer
array of adapters); section "Step-by-Step Implementation" (per-row loop x[i] @ A[id] @ B[id]).
"""
from __future__ import annotations

import json
import os

import numpy as np

from segmented_gather_gemm_sgmv_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
RTOL = 1e-12


def _close(a, b, rtol=RTOL, what=""):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= rtol * scale, f"{what}: max abs err {err:.3e} > {rtol * scale:.3e}"


def random_problem(seed, S=7, max_len=5, n_adapters=4, L=3, h_in=24, h_out=40, r=4,
                   p_empty=0.0):
    rng = np.random.default_rng(seed)
    ss, sa = workloads.random_segments(rng, S, max_len, n_adapters, p_empty=p_empty)
    M = int(ss[-1])
    x = rng.standard_normal((M, h_in))
    y = rng.standard_normal((M, h_out))
    A = [rng.uniform(-1, 1, (L, h_in, r)) for _ in range(n_adapters)]
    B = [rng.standard_normal((L, r, h_out)) for _ in range(n_adapters)]
    return dict(ss=ss, sa=sa, x=x, y=y, A=A, B=B, L=L, h_in=h_in, h_out=h_out, r=r, M=M)


def check_hand_example(o):
    """The hand-worked example in tests/golden/hand_example.json, exactly."""
    g = json.load(open(os.path.join(GOLDEN, "hand_example.json")))
    A = [np.asarray(a, np.float64)[None] for a in g["A"]]
    B = [np.asarray(b, np.float64)[None] for b in g["B"]]
    y = o.lora_apply(g["y_in"], g["x"], A, B, g["seg_starts"], g["seg_adapter"], 0, g["scale"])
    assert np.array_equal(y, np.asarray(g["y_expected"], np.float64)), y
    v = o.sgmv_shrink(np.zeros((3, 1)), g["x"], A, g["seg_starts"], g["seg_adapter"], 0)
    assert np.array_equal(v, np.asarray(g["v_expected"], np.float64)), v


def check_merged_weights(o):
    """x W0 + s x A B == x (W0 + s A B): the LoRA term merged into the base weight."""
    p = random_problem(11, h_in=20, h_out=36, r=3)
    rng = np.random.default_rng(12)
    W0 = rng.standard_normal((p["h_in"], p["h_out"]))
    s, layer = 0.75, 2
    y_base = p["x"] @ W0
    got = o.lora_apply(y_base, p["x"], p["A"], p["B"], p["ss"], p["sa"], layer, s)
    want = np.empty_like(got)
    for i, k in enumerate(p["sa"]):
        lo, hi = p["ss"][i], p["ss"][i + 1]
        Wk = W0 + s * (p["A"][k][layer] @ p["B"][k][layer])
        want[lo:hi] = p["x"][lo:hi] @ Wk
    _close(got, want, what="merged weights")


def check_per_request_gemv(o):
    """SGMV equals one independent GEMV chain per request (row), each with its own adapter."""
    p = random_problem(21, S=9, max_len=4, n_adapters=5, L=4, h_in=16, h_out=28, r=6)
    s, layer = 1.5, 3
    got = o.lora_apply(p["y"], p["x"], p["A"], p["B"], p["ss"], p["sa"], layer, s)
    want = p["y"].copy()
    for i, k in enumerate(p["sa"]):
        for t in range(p["ss"][i], p["ss"][i + 1]):
            want[t] = p["y"][t] + s * (p["x"][t:t + 1] @ p["A"][k][layer] @ p["B"][k][layer])[0]
    _close(got, want, what="per-request GEMV")


def check_single_adapter_dense(o):
    """All segments on one adapter == one dense GEMM y + s (X A) B over the rows."""
    rng = np.random.default_rng(31)
    ss = np.array([0, 3, 3, 8, 13], np.int32)
    sa = np.array([2, 2, 2, 2], np.int32)
    h_in, h_out, r, L = 32, 20, 8, 2
    x = rng.standard_normal((13, h_in))
    y = rng.standard_normal((13, h_out))
    A = [rng.uniform(-1, 1, (L, h_in, r)) for _ in range(3)]
    B = [rng.standard_normal((L, r, h_out)) for _ in range(3)]
    got = o.lora_apply(y, x, A, B, ss, sa, 1, 0.5)
    _close(got, y + 0.5 * ((x @ A[2][1]) @ B[2][1]), what="single adapter dense")


def check_zero_adapter(o):
    """A zero A or a zero B leaves the rows of that adapter bitwise unchanged."""
    p = random_problem(41, S=10, n_adapters=3)
    p["A"][1] = np.zeros_like(p["A"][1])
    p["B"][2] = np.zeros_like(p["B"][2])
    got = o.lora_apply(p["y"], p["x"], p["A"], p["B"], p["ss"], p["sa"], 0, 2.0)
    touched_other = False
    for i, k in enumerate(p["sa"]):
        lo, hi = p["ss"][i], p["ss"][i + 1]
        if k in (1, 2):
            assert np.array_equal(got[lo:hi], p["y"][lo:hi]), f"zero adapter {k} changed y"
        elif hi > lo:
            touched_other = touched_other or not np.array_equal(got[lo:hi], p["y"][lo:hi])
    assert touched_other, "adapter 0 rows should change"


def check_permutation(o):
    """Permuting segments together with their rows permutes the output identically."""
    p = random_problem(51, S=8, max_len=4)
    rng = np.random.default_rng(52)
    perm = rng.permutation(len(p["sa"]))
    rows, starts = [], [0]
    for i in perm:
        rows.extend(range(p["ss"][i], p["ss"][i + 1]))
        starts.append(starts[-1] + p["ss"][i + 1] - p["ss"][i])
    rows = np.asarray(rows, np.int64)
    got = o.lora_apply(p["y"], p["x"], p["A"], p["B"], p["ss"], p["sa"], 1, 1.25)
    got_p = o.lora_apply(p["y"][rows], p["x"][rows], p["A"], p["B"], np.asarray(starts),
                         p["sa"][perm], 1, 1.25)
    assert np.array_equal(got[rows], got_p), "permutation changed the result"


def check_brute_force(o):
    """Pure-Python triple loop on tiny inputs (and the 'tiny' workload's segment table)."""
    for seed in range(3):
        p = random_problem(61 + seed, S=4, max_len=3, n_adapters=3, L=2, h_in=5, h_out=6, r=2,
                           p_empty=0.2)
        s, layer = 0.5 + seed, seed % 2
        want = [list(map(float, row)) for row in p["y"]]
        for i, k in enumerate(p["sa"]):
            for t in range(int(p["ss"][i]), int(p["ss"][i + 1])):
                for n in range(p["h_out"]):
                    acc = 0.0
                    for c in range(p["r"]):
                        vc = 0.0
                        for j in range(p["h_in"]):
                            vc += p["x"][t][j] * p["A"][k][layer][j][c]
                        acc += vc * p["B"][k][layer][c][n]
                    want[t][n] += s * acc
        got = o.lora_apply(p["y"], p["x"], p["A"], p["B"], p["ss"], p["sa"], layer, s)
        _close(got, np.asarray(want), what=f"brute force {seed}")
    ss, sa = workloads.make_segments("tiny", 0)
    rng = np.random.default_rng(65)
    M = int(ss[-1])
    x, y = rng.standard_normal((M, 3)), rng.standard_normal((M, 2))
    A = [rng.standard_normal((1, 3, 2)) for _ in range(4)]
    B = [rng.standard_normal((1, 2, 2)) for _ in range(4)]
    want = y.copy()
    for i, k in enumerate(sa):
        for t in range(ss[i], ss[i + 1]):
            for n in range(2):
                want[t, n] += 2.0 * sum(sum(x[t, j] * A[k][0][j, c] for j in range(3))
                                        * B[k][0][c, n] for c in range(2))
    _close(o.lora_apply(y, x, A, B, ss, sa, 0, 2.0), want, what="tiny table brute force")


def check_layer_selection(o):
    """layer_idx picks the [h_in][r] / [r][h_out] slice of each adapter's stacked block."""
    p = random_problem(71, S=6, L=5, h_in=12, h_out=10, r=3)
    for layer in (0, 2, 4):
        got = o.lora_apply(p["y"], p["x"], p["A"], p["B"], p["ss"], p["sa"], layer, 1.0)
        A1 = [a[layer:layer + 1] for a in p["A"]]
        B1 = [b[layer:layer + 1] for b in p["B"]]
        one = o.lora_apply(p["y"], p["x"], A1, B1, p["ss"], p["sa"], 0, 1.0)
        assert np.array_equal(got, one), f"layer {layer} != single-layer block"
        want = p["y"].copy()
        for i, k in enumerate(p["sa"]):
            lo, hi = p["ss"][i], p["ss"][i + 1]
            want[lo:hi] += p["x"][lo:hi] @ p["A"][k][layer] @ p["B"][k][layer]
        _close(got, want, what=f"layer {layer}")


def check_shrink_expand(o):
    """shrink == x A_k, expand == y + s v B_k (numpy), and expand(shrink) == lora_apply."""
    p = random_problem(81, S=7, h_in=18, h_out=14, r=5)
    s, layer = 0.25, 1
    v0 = np.full((p["M"], p["r"]), 7.0)
    v = o.sgmv_shrink(v0, p["x"], p["A"], p["ss"], p["sa"], layer)
    v_want = v0.copy()
    for i, k in enumerate(p["sa"]):
        lo, hi = p["ss"][i], p["ss"][i + 1]
        v_want[lo:hi] = p["x"][lo:hi] @ p["A"][k][layer]
    _close(v, v_want, what="shrink")
    y = o.sgmv_expand(p["y"], v, p["B"], p["ss"], p["sa"], layer, s)
    y_want = p["y"].copy()
    for i, k in enumerate(p["sa"]):
        lo, hi = p["ss"][i], p["ss"][i + 1]
        y_want[lo:hi] += s * (v_want[lo:hi] @ p["B"][k][layer])
    _close(y, y_want, what="expand")
    fused = o.lora_apply(p["y"], p["x"], p["A"], p["B"], p["ss"], p["sa"], layer, s)
    _close(fused, y, what="fused == expand(shrink)")


def check_untouched_rows(o):
    """Rows outside every segment, in empty segments or with a negative id stay bitwise."""
    rng = np.random.default_rng(91)
    ss = np.array([2, 4, 4, 7, 9], np.int32)      # rows 0,1 and 9,10 outside; seg 1 empty
    sa = np.array([0, 1, -1, 1], np.int32)        # seg 2 (rows 4..6) carries no adapter
    x, y = rng.standard_normal((11, 6)), rng.standard_normal((11, 5))
    A = [rng.standard_normal((1, 6, 2)) for _ in range(2)]
    B = [rng.standard_normal((1, 2, 5)) for _ in range(2)]
    got = o.lora_apply(y, x, A, B, ss, sa, 0, 1.0)
    for t in (0, 1, 4, 5, 6, 9, 10):
        assert np.array_equal(got[t], y[t]), f"row {t} should be untouched"
    for t in (2, 3, 7, 8):
        assert not np.array_equal(got[t], y[t]), f"row {t} should change"


def check_validate(o):
    """The table check flags exactly the documented defects."""
    ok = o.validate([0, 2, 2, 5], [0, 3, 1], 4, 5)
    assert ok == 0, ok
    assert o.validate([0, 3, 2, 5], [0, 1, 1], 4, 5) == 1          # decreasing offsets
    assert o.validate([-1, 2, 5], [0, 1], 4, 5) == 2               # negative first offset
    assert o.validate([0, 2, 6], [0, 1], 4, 5) == 4                # past the last row
    assert o.validate([0, 2, 5], [0, 4], 4, 5) == 8                # id out of the pool
    assert o.validate([0, 2, 5], [-1, 3], 4, 5) == 0               # negative id = no adapter
    assert o.validate([0], [], 4, 0) == 0                          # no segments
    assert o.validate([1, 0, 9], [7, 0], 4, 5) == 1 | 4 | 8


def check_validate_pointers(o):
    """The pointer check flags exactly a null or non-16-byte-aligned address of an adapter that
    a non-empty segment uses, and looks at nothing else."""
    good = [0x1000, 0x2010, 0x3020, 0x4030]
    ss, sa = [0, 2, 2, 5], [0, 3, 1]
    assert o.validate_pointers(good, good, ss, sa, 4) == 0
    # segment 1 is empty, so adapter 3's pointers are never used
    assert o.validate_pointers([0x1000, 0x2010, 0x3020, 0], good, ss, sa, 4) == 0
    assert o.validate_pointers([0x1000, 0, 0x3020, 0x4030], good, ss, sa, 4) == 16   # A[1] null
    assert o.validate_pointers(good, [0x1000, 0x2018, 0, 0], ss, sa, 4) == 32        # B[1] odd
    assert o.validate_pointers(good, [0x1008, 0x2010, 0x3020, 0x4031], ss, sa, 4) == 32  # B[0]
    # adapter 1 sits in an empty segment and adapter 2 in none: their pointers are not used
    assert o.validate_pointers([0x1000, 0, 0x3001, 0x4030], good, [0, 2, 2, 5], [0, 1, 3], 4) == 0
    # a negative id carries no adapter; an id past the pool is reported by validate(), not here
    assert o.validate_pointers([0x1000, 0x2010, 0x3020, 0x4030], good, [0, 1, 2], [-1, 9], 4) == 0
    assert o.validate_pointers([8, 16], [0, 32], [0, 1, 2], [0, 1], 2) == 16 | 32
    assert o.validate_pointers(None, [0, 32], [0, 1, 2], [0, 1], 2) == 32       # A not checked
    assert o.validate_pointers([8, 16], None, [0, 1, 2], [0, 1], 2) == 16       # B not checked
    assert o.validate_pointers(good, good, [0], [], 4) == 0                      # no segments


def check_plan(o):
    """The grouping: hand-worked tables, and on random tables the invariants that fix it --
    every row of a non-empty segment with an adapter listed exactly once, under its adapter,
    groups in order of first appearance, rows of a group in segment order then row order."""
    # segment 0 (rows 0,1) and segment 3 (rows 3..6) use adapter 5, segment 1 (row 2) adapter 1,
    # segment 2 is empty, segment 4 has no adapter
    gs, ga, rows = o.plan([0, 2, 3, 3, 7, 8], [5, 1, 4, 5, -1], 100)
    assert ga.tolist() == [5, 1] and gs.tolist() == [0, 6, 7]
    assert rows.tolist() == [0, 1, 3, 4, 5, 6, 2]
    assert o.plan([0, 2, 3, 3, 7, 8], [5, 1, 4, 5, -1], 6) is None      # 7 rows > 6
    gs, ga, rows = o.plan([0], [], 0)
    assert gs.tolist() == [0] and len(ga) == 0 and len(rows) == 0
    gs, ga, rows = o.plan([4, 9], [0], 5)                               # rows need not start at 0
    assert ga.tolist() == [0] and rows.tolist() == [4, 5, 6, 7, 8]
    rng = np.random.default_rng(11)
    for _ in range(40):
        S = int(rng.integers(1, 60))
        lens = rng.integers(0, 5, size=S)
        ss = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        sa = rng.integers(-1, 8, size=S).astype(np.int32)
        gs, ga, rows = o.plan(ss, sa, int(ss[-1]))
        want = sorted(t for i in range(S) if sa[i] >= 0 for t in range(ss[i], ss[i + 1]))
        assert sorted(rows.tolist()) == want                            # each row exactly once
        firsts = []
        for i in range(S):
            if sa[i] >= 0 and lens[i] > 0 and sa[i] not in firsts:
                firsts.append(int(sa[i]))
        assert ga.tolist() == firsts                                    # order of first use
        for g, k in enumerate(ga):
            expect = [t for i in range(S) if sa[i] == k for t in range(ss[i], ss[i + 1])]
            assert rows[gs[g]:gs[g + 1]].tolist() == expect


def check_ranked(o):
    """Per-adapter rank and scale, pinned three ways: a hand-worked two-adapter case; per-row
    GEMV chains through numpy with each adapter's own shapes (a library matmul, not this
    loop); and zero-padding -- an adapter of rank r_k gives exactly what the same weights
    padded with zero columns of A and zero rows of B to a larger rank give."""
    # hand-worked: h_in = h_out = 2; adapter 0 of rank 1, adapter 1 of rank 2
    x = np.array([[1.0, 2.0], [3.0, -1.0], [0.5, 0.5]])
    y = np.array([[10.0, 20.0], [30.0, 40.0], [50.0, 60.0]])
    A0 = np.array([[[1.0], [1.0]]])               # (1, 2, 1): v = x0 + x1
    B0 = np.array([[[2.0, -1.0]]])                # (1, 1, 2)
    A1 = np.array([[[1.0, 0.0], [0.0, 1.0]]])     # identity
    B1 = np.array([[[1.0, 1.0], [0.0, 1.0]]])
    got = o.lora_apply_ranked(y, x, [A0, A1], [B0, B1], [1, 2], [0.5, 2.0], [0, 1, 3], [0, 1], 0)
    # row 0, adapter 0: v = 3 -> 0.5 * [6, -3] = [3, -1.5]
    # rows 1, 2, adapter 1: v = x -> v B1 = [x0, x0 + x1] -> *2
    want = np.array([[13.0, 18.5], [36.0, 44.0], [51.0, 62.0]])
    assert np.array_equal(got, want), got
    rng = np.random.default_rng(19)
    h_in, h_out, L = 24, 40, 2
    ranks = [8, 16, 24, 8, 32]
    A = [rng.standard_normal((L, h_in, r)) for r in ranks]
    B = [rng.standard_normal((L, r, h_out)) for r in ranks]
    scale = rng.uniform(0.1, 3.0, size=len(ranks))
    ss = np.array([0, 3, 4, 9, 9, 12], np.int32)
    sa = np.array([2, 0, 4, 1, 2], np.int32)
    x = rng.standard_normal((12, h_in))
    y = rng.standard_normal((12, h_out))
    got = o.lora_apply_ranked(y, x, A, B, ranks, scale, ss, sa, 1)
    want = y.copy()
    for i, k in enumerate(sa):
        for t in range(ss[i], ss[i + 1]):
            want[t] += scale[k] * (x[t:t + 1] @ A[k][1] @ B[k][1])[0]
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    # zero padding to rank 32 through the uniform-rank entry point, one adapter at a time
    for k in range(len(ranks)):
        Ap = np.zeros((L, h_in, 32))
        Bp = np.zeros((L, 32, h_out))
        Ap[:, :, :ranks[k]] = A[k]
        Bp[:, :ranks[k], :] = B[k]
        one = o.lora_apply_ranked(y, x, [A[k]], [B[k]], [ranks[k]], [scale[k]], [0, 12], [0], 1)
        pad = o.lora_apply(y, x, [Ap], [Bp], [0, 12], [0], 1, scale[k])
        assert np.allclose(one, pad, rtol=1e-12, atol=1e-12)


def check_base_lora(o):
    """The base projection plus the LoRA term, written into y, pinned four ways: the
    hand-worked case in tests/golden/base_lora_hand.json; merged weights through numpy (each
    row times W0^T + s A_k B_k of its own adapter, base only for rows without one); W0 = 0
    reduces it to the already pinned lora_apply on a zero y; and zero adapters reduce it to a
    numpy matmul x W0^T."""
    g = json.load(open(os.path.join(GOLDEN, "base_lora_hand.json")))
    A = [np.asarray(a, np.float64)[None] for a in g["A"]]
    B = [np.asarray(b, np.float64)[None] for b in g["B"]]
    y = o.base_lora(g["x"], g["W0"], A, B, g["seg_starts"], g["seg_adapter"], 0, g["scale"])
    assert np.array_equal(y, np.asarray(g["y_expected"], np.float64)), y
    rng = np.random.default_rng(23)
    p = random_problem(29, S=6, h_in=20, h_out=28, r=3, n_adapters=3)
    M = p["M"] + 3  # three rows after the last segment
    x = rng.standard_normal((M, p["h_in"]))
    W0 = rng.standard_normal((p["h_out"], p["h_in"]))
    sa = p["sa"].copy()
    sa[1] = -1
    s, layer = 0.6, 1
    got = o.base_lora(x, W0, p["A"], p["B"], p["ss"], sa, layer, s)
    want = x @ W0.T
    for i, k in enumerate(sa):
        lo, hi = p["ss"][i], p["ss"][i + 1]
        if k >= 0:
            want[lo:hi] = x[lo:hi] @ (W0.T + s * (p["A"][k][layer] @ p["B"][k][layer]))
    _close(got, want, what="base + LoRA, merged weights")
    zero_w = o.base_lora(x, np.zeros_like(W0), p["A"], p["B"], p["ss"], sa, layer, s)
    _close(zero_w, o.lora_apply(np.zeros((M, p["h_out"])), x, p["A"], p["B"], p["ss"], sa,
                                layer, s), what="W0 = 0")
    zero_a = o.base_lora(x, W0, [np.zeros_like(a) for a in p["A"]], p["B"], p["ss"], sa, layer,
                         s)
    _close(zero_a, x @ W0.T, what="zero adapters")


ALL_CHECKS = [check_hand_example, check_merged_weights, check_per_request_gemv,
              check_single_adapter_dense, check_zero_adapter, check_permutation,
              check_brute_force, check_layer_selection, check_shrink_expand,
              check_untouched_rows, check_validate, check_validate_pointers, check_plan,
              check_ranked, check_base_lora]
