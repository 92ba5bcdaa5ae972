"""Pins of the product-key top-k oracle (oracle/product_key.py) against brute force over every
slot, hand-worked tie cases of the pages' rule and finite differences (no GPU)."""

import itertools
import zlib

import numpy as np
import pytest

from oracle import product_key as pk


def brute_scores(row, factors, dtype):
    """Score and lin of every slot, by the definition: float32 sums in factor order, each
    partial sum rounded to bfloat16 before the next factor for bfloat16 input and F > 2."""
    offs = np.concatenate([[0], np.cumsum(factors)[:-1]])
    F = len(factors)
    scores, lins = [], []
    for cs in itertools.product(*(range(f) for f in factors)):
        s = np.float32(row[offs[0] + cs[0]])
        for f in range(1, F):
            if dtype == "bf16" and F > 2 and f > 1:
                s = pk.bf16_round(np.array([s]))[0]
            s = np.float32(s + np.float32(row[offs[f] + cs[f]]))
        lin = 0
        for f in range(F):
            lin = lin * factors[f] + cs[f]
        scores.append(s)
        lins.append(lin)
    return np.array(scores, np.float32), np.array(lins, np.int64)


def as_compare(x):
    """The comparison value of a float32 score: NaN as -inf (zeros compare equal here)."""
    x = np.asarray(x, np.float64)
    return np.where(np.isnan(x), -np.inf, x)


def make_row(rng, factors, dtype, ties):
    n = sum(factors)
    x = rng.integers(-3, 4, n).astype(np.float32) if ties else rng.standard_normal(n).astype(np.float32)
    return pk.bf16_round(x) if dtype == "bf16" else x


@pytest.mark.parametrize("factors", [(7,), (5, 6), (4, 3, 5), (3, 4, 2, 3), (1, 9), (6, 1, 1)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("k", [1, 4, 13, 256])
def test_topk_is_an_exact_topk(factors, dtype, ties, k):
    """The selected scores are the kk largest of all slots (as a multiset), every selected
    slot's output is its own score, and lin is strictly ascending."""
    rng = np.random.default_rng(zlib.crc32(repr((factors, dtype, ties, k)).encode()))
    raw = np.stack([make_row(rng, factors, dtype, ties) for _ in range(3)])
    val, lin = pk.product_key_topk(raw, factors, k, dtype)
    kk = min(k, int(np.prod(factors)))
    assert val.shape == lin.shape == (3, kk)
    for r in range(3):
        scores, lins = brute_scores(raw[r], factors, dtype)
        best = np.sort(as_compare(scores))[::-1][:kk]
        assert np.all(np.diff(lin[r]) > 0)
        by_lin = dict(zip(lins.tolist(), scores.tolist()))
        got = np.array([by_lin[int(l)] for l in lin[r]], np.float32)
        np.testing.assert_array_equal(np.sort(as_compare(got))[::-1], best)
        expect_val = pk.bf16_round(got) if dtype == "bf16" else got
        np.testing.assert_array_equal(val[r], expect_val)


def test_tie_rule_hand_worked():
    """Two factors of four equal values, k = 2 (worked by hand from the pages' rule):
    each factor ranks columns 3, 2, 1, 0; the pairs (i + 1)(j + 1) <= 2 are (0,0), (0,1),
    (1,0), all tied, so the larger i + j wins, then the larger i: (1,0) then (0,1), i.e. slots
    (2, 3) and (3, 2), lin 11 and 14."""
    val, lin = pk.product_key_topk(np.ones((1, 8), np.float32), (4, 4), 2)
    np.testing.assert_array_equal(lin, [[11, 14]])
    np.testing.assert_array_equal(val, [[2.0, 2.0]])


def test_signed_zero_and_nan_rule():
    """+0 ranks above -0 and equal values go to the larger column; NaN counts as -inf."""
    _, lin = pk.product_key_topk(np.array([[0.0, -0.0, -0.0, 0.0]], np.float32), (4,), 2)
    np.testing.assert_array_equal(lin, [[0, 3]])
    val, lin = pk.product_key_topk(np.array([[np.nan, -np.inf, 1.0]], np.float32), (3,), 2)
    np.testing.assert_array_equal(lin, [[1, 2]])
    np.testing.assert_array_equal(val, [[-np.inf, 1.0]])


def test_backward_by_finite_differences():
    """val is a sum of raw columns for a fixed selection: the gradient of <g, val> by central
    differences (no ties, so the selection does not move) equals the oracle's backward."""
    factors, k = (5, 4, 3), 7
    rng = np.random.default_rng(99)
    raw = rng.standard_normal((2, sum(factors))).astype(np.float64)
    g = rng.standard_normal((2, k))
    _, lin = pk.product_key_topk(raw.astype(np.float32), factors, k)
    grad = pk.product_key_topk_backward(lin, g, factors)

    def loss(x):
        val, lin2 = pk.product_key_topk(x.astype(np.float32), factors, k)
        assert np.array_equal(lin2, lin)
        return float((val.astype(np.float64) * g).sum())

    h = 1e-3
    for r in range(2):
        for c in range(sum(factors)):
            xp, xm = raw.copy(), raw.copy()
            xp[r, c] += h
            xm[r, c] -= h
            fd = (loss(xp) - loss(xm)) / (2 * h)
            assert abs(fd - grad[r, c]) <= 1e-3 * max(1.0, abs(fd)), (r, c, fd, grad[r, c])


def test_tie_rule_larger_i_and_stage_ranks_hand_worked():
    """k = 3 over two factors of four equal values: the pairs (i+1)(j+1) <= 3 are (0,0),
    (0,1), (0,2), (1,0), (2,0); by i + j, then i: (2,0), (0,2), (1,0) are kept, i.e. slots
    (1,3), (3,1), (2,3): lin 7, 13, 11. (The larger-i rule picks (1,0) over (0,1), lin 11 not 14.)
    Three factors of two equal values, k = 2: stage 1 keeps (1,0) then (0,1), ranks 0 and 1 of
    the partial slots (0,1) and (1,0) (partial lin 1 and 2); stage 2 keeps (1,0) = partial lin
    2 with column 1, lin 5, and (0,1) = partial lin 1 with column 0, lin 2."""
    _, lin = pk.product_key_topk(np.ones((1, 8), np.float32), (4, 4), 3)
    np.testing.assert_array_equal(lin, [[7, 11, 13]])
    _, lin = pk.product_key_topk(np.ones((1, 6), np.float32), (2, 2, 2), 2)
    np.testing.assert_array_equal(lin, [[2, 5]])
