"""Exact top-k over product-key slots, as the selection rule of the pages states it
(sparse-delta-memory 2.0.0, product_key_topk.py: the ``product_key_topk`` docstring).

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle``): plain numpy, one row at a time.

A row of ``raw`` holds F >= 1 factors side by side (``factors`` = their widths). Slot
(c_0, ..., c_{F-1}) scores the float32 sum of its factor values, added in factor order; with
bfloat16 input and F > 2 each partial sum is rounded to bfloat16 before the next factor is
added. Its index is lin = (..(c_0 * factors[1] + c_1) * ..) * factors[F-1] + c_{F-1}.

Selection (the pages' rule, in their order):
  * scores compare as float32 numbers, -0 below +0, NaN counted as -inf;
  * each factor is ranked by value, the larger column first on ties;
  * stage 0 keeps the first min(k, factors[0]) ranks of factor 0;
  * stage f = 1..F-1 takes the previous stage's ranked list (n = its length) and the first
    m = min(k, factors[f]) ranks of factor f, and keeps the best c = min(k, n m) of the pairs
    (i, j), i < n, j < m, with (i + 1)(j + 1) <= c: higher score first, exact ties to the larger
    i + j, then the larger i. The kept pairs, in that order, are the next stage's ranks.
Output: the kept slots sorted by lin ascending, with val = the score rounded to the input dtype.

Reading (the pages leave it open): with bfloat16 input and F > 2, the score a stage f < F-1
compares is the bfloat16-rounded partial sum it passes on (rounding is monotone, so the
exactness argument of the rule holds for those values); the last stage compares the float32
sum.

Backward: the gradient of val reaches raw at each factor column of each selected slot (the
rounding of partial sums passes it unchanged), added in output order.
"""

from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 (round to nearest even) -> float32, on the bit pattern."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _order_desc(score: np.ndarray, *tiebreaks: np.ndarray) -> np.ndarray:
    """Indices sorting by score descending (NaN as -inf, -0 below +0), then by each tie-break
    array descending."""
    s = np.asarray(score, np.float32)
    val = np.where(np.isnan(s), -np.inf, s).astype(np.float64)
    pos_zero = ((s == 0) & ~np.signbit(s)).astype(np.int64)    # +0 above -0
    keys = [-np.asarray(t, np.int64) for t in reversed(tiebreaks)] + [-pos_zero, -val]
    return np.lexsort(keys)


def product_key_topk(raw: np.ndarray, factors: Sequence[int], k: int,
                     dtype: str = "f32") -> Tuple[np.ndarray, np.ndarray]:
    """(val [rows, kk] float32 (values of ``dtype``), lin [rows, kk] int64) for raw [rows,
    sum(factors)] holding the stored values (bfloat16 inputs as their float32 values)."""
    factors = tuple(int(f) for f in factors)
    F = len(factors)
    if F < 1 or min(factors) < 1 or not 1 <= k <= 256:
        raise ValueError("need F >= 1 factors of >= 1 column and 1 <= k <= 256")
    raw = np.asarray(raw, np.float32)
    rows = raw.reshape(-1, raw.shape[-1])
    if rows.shape[1] != sum(factors):
        raise ValueError("raw's last dimension must be sum(factors)")
    kk = min(k, int(np.prod(factors, dtype=np.int64)))
    offs = np.concatenate([[0], np.cumsum(factors)[:-1]]).astype(np.int64)
    round_partial = dtype == "bf16" and F > 2
    vals = np.zeros((rows.shape[0], kk), np.float32)
    lins = np.zeros((rows.shape[0], kk), np.int64)
    for r, row in enumerate(rows):
        ranks = []
        for f in range(F):
            v = row[offs[f]:offs[f] + factors[f]]
            cols = np.arange(factors[f])
            ranks.append(_order_desc(v, cols))              # larger column first on ties
        n = min(k, factors[0])
        score = row[offs[0] + ranks[0][:n]].astype(np.float32)
        lin = ranks[0][:n].astype(np.int64)
        for f in range(1, F):
            m = min(k, factors[f])
            c = min(k, n * m)
            ii, jj = np.meshgrid(np.arange(n), np.arange(m), indexing="ij")
            keep = (ii + 1) * (jj + 1) <= c
            ii, jj = ii[keep], jj[keep]
            fcol = ranks[f][jj]
            s = (score[ii] + row[offs[f] + fcol]).astype(np.float32)
            if round_partial and f < F - 1:
                s = bf16_round(s)
            order = _order_desc(s, ii + jj, ii)[:c]
            score, lin = s[order], lin[ii[order]] * factors[f] + fcol[order]
            n = c
        out = np.argsort(lin, kind="stable")
        lins[r] = lin[out]
        vals[r] = bf16_round(score[out]) if dtype == "bf16" else score[out]
    shape = raw.shape[:-1] + (kk,)
    return vals.reshape(shape), lins.reshape(shape)


def product_key_topk_backward(lin: np.ndarray, grad_val: np.ndarray,
                              factors: Sequence[int]) -> np.ndarray:
    """d(loss)/d(raw) [rows, sum(factors)] in float64: each output's gradient added to the raw
    column of every factor of its slot, outputs in order."""
    factors = tuple(int(f) for f in factors)
    offs = np.concatenate([[0], np.cumsum(factors)[:-1]]).astype(np.int64)
    lin2 = np.asarray(lin, np.int64).reshape(-1, np.shape(lin)[-1])
    g2 = np.asarray(grad_val, np.float64).reshape(lin2.shape)
    out = np.zeros((lin2.shape[0], sum(factors)), np.float64)
    for r in range(lin2.shape[0]):
        for t in range(lin2.shape[1]):
            rest = int(lin2[r, t])
            for f in range(len(factors) - 1, -1, -1):
                out[r, offs[f] + rest % factors[f]] += g2[r, t]
                rest //= factors[f]
    return out.reshape(np.shape(lin)[:-1] + (sum(factors),))
