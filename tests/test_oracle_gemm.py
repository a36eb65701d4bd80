"""Pins for the oracle's three grouped GEMM forms.

The oracle's numpy matmul is held to a pure-Python triple loop on tiny shapes
(1e-12 relative), and the layout rules to hand-placed one-hot rows, so a
transposed operand, a wrong segment offset or a dropped expert fails here.
"""
import numpy as np
import pytest

from oracle import gemm as og
from oracle import plan as op

pytestmark = pytest.mark.cpu


def triple_loop(a_rows, b_e):
    t, K = len(a_rows), len(a_rows[0]) if len(a_rows) else 0
    N = len(b_e)
    out = [[0.0] * N for _ in range(t)]
    for r in range(t):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += float(a_rows[r][k]) * float(b_e[n][k])
            out[r][n] = s
    return np.array(out).reshape(t, N)


def close(a, b, rel=1e-12):
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    return np.max(np.abs(a - b)) <= rel * scale if a.size else True


@pytest.mark.parametrize("counts,align", [([3, 0, 5, 1], 4), ([0, 0, 2], 2), ([7], 8), ([1, 1, 1, 1, 1], 1)])
def test_contiguous_vs_triple_loop(counts, align):
    rng = np.random.default_rng(1)
    E, N, K = len(counts), 5, 6
    p = op.plan(counts, align)
    rows_cap = p.P + 3
    A = rng.standard_normal((rows_cap, K))
    B = rng.standard_normal((E, N, K))
    R, written = og.contiguous(A, B, counts, align)
    for e, t in enumerate(counts):
        o = p.offsets[e]
        assert og.contiguous_segment(counts, align, e) == (o, o + t)
        assert written[o:o + t].all()
        assert close(R[o:o + t], triple_loop(A[o:o + t].tolist(), B[e].tolist()))
        # rows between this segment's end and the next aligned start stay untouched
        assert not written[o + t:p.offsets[e + 1]].any()
        assert np.isnan(R[o + t:p.offsets[e + 1]]).all()
    assert not written[p.P:].any()


def test_contiguous_one_hot_rows_pick_weight_columns():
    """Row r of expert e set to the unit vector e_k returns column k of B[e]."""
    counts, align = [2, 3], 4
    E, N, K = 2, 7, 5
    rng = np.random.default_rng(2)
    B = rng.standard_normal((E, N, K))
    A = np.zeros((8, K))
    picks = {0: (0, 3), 1: (0, 1), 4: (1, 0), 5: (1, 4), 6: (1, 2)}
    for r, (_, k) in picks.items():
        A[r, k] = 1.0
    R, written = og.contiguous(A, B, counts, align)
    for r, (e, k) in picks.items():
        assert np.array_equal(R[r], B[e][:, k])
    assert not written[2:4].any() and not written[7]


def test_contiguous_capacity_error():
    with pytest.raises(ValueError):
        og.contiguous(np.zeros((15, 2)), np.zeros((2, 3, 2)), [9, 1], 8)


def test_masked_vs_triple_loop():
    rng = np.random.default_rng(3)
    E, M, N, K = 4, 6, 3, 5
    valid = [0, 6, 2, 1]
    A = rng.standard_normal((E, M, K))
    B = rng.standard_normal((E, N, K))
    R, written = og.masked(A, B, valid)
    for e, v in enumerate(valid):
        assert written[e, :v].all() and not written[e, v:].any()
        assert close(R[e, :v], triple_loop(A[e, :v].tolist(), B[e].tolist()))
        assert np.isnan(R[e, v:]).all()
    with pytest.raises(ValueError):
        og.masked(A, B, [0, 7, 0, 0])


def test_masked_one_hot():
    E, M, N, K = 2, 3, 4, 3
    B = np.arange(E * N * K, dtype=float).reshape(E, N, K)
    A = np.zeros((E, M, K))
    A[1, 1, 2] = 1.0
    R, _ = og.masked(A, B, [0, 2])
    assert np.array_equal(R[1, 1], B[1][:, 2])
    assert np.array_equal(R[1, 0], np.zeros(N))


def test_kgrouped_vs_outer_product_sum():
    """dW[e][n][k] = sum over expert e's tokens t of dY[t][n] * X[t][k]."""
    rng = np.random.default_rng(4)
    counts = [3, 0, 4, 1]
    T_cap, N, K = 10, 3, 2
    dY = rng.standard_normal((T_cap, N))
    X = rng.standard_normal((T_cap, K))
    dW = og.kgrouped(dY, X, counts)
    t0 = 0
    for e, t in enumerate(counts):
        ref = np.zeros((N, K))
        for tok in range(t0, t0 + t):
            for n in range(N):
                for k in range(K):
                    ref[n, k] += dY[tok, n] * X[tok, k]
        assert close(dW[e], ref)
        t0 += t
    assert np.array_equal(dW[1], np.zeros((N, K)))
    with pytest.raises(ValueError):
        og.kgrouped(dY, X, [6, 6])


def test_kgrouped_one_hot_tokens():
    """A single token with unit vectors makes dW[e] a single 1 at (n, k)."""
    dY = np.zeros((3, 4))
    X = np.zeros((3, 5))
    dY[2, 1] = 1.0
    X[2, 3] = 1.0
    dW = og.kgrouped(dY, X, [2, 1])
    assert dW[1, 1, 3] == 1.0 and dW[1].sum() == 1.0 and dW[0].sum() == 0.0
