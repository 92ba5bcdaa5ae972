"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Every check here uses code other than the oracle's own arithmetic: dense linear algebra,
closed forms, a hand-worked example, brute-force grouping and finite differences.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
import sdm_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(P=2, T=23, S=9, D=3, W=3, R=2, seed=0, ragged=True, zipf=True):
    wl = si.Workload("t", P, T, 8, S, D, W, R, "f32", "zipf1.1" if zipf else "uniform", ragged,
                     seed)
    x = oracle.from_stored(si.generate(wl), "f32")
    return wl, x


def args(x):
    return (x["bank"], x["ws"], x["k"], x["g"], x["beta"], x["v"], x["rs"], x["q"], x["valid"])


def rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


# ---------------------------------------------------------------------------------------
# sequential oracle
# ---------------------------------------------------------------------------------------

def dense_brute_force(bank, ws, k, g, beta, v, rs, q, valid):
    """B <- (I - beta K K^T) E B + beta K v^T, o = Q^T B: the token step as dense S x S maps
    (E = diag(exp(g)) on the written rows, K and Q the weight vectors over slots)."""
    P, T, W = ws.shape
    S = bank.shape[0] // P
    B = bank.reshape(P, S, -1).copy()
    out = np.zeros((P, T, B.shape[2]))
    for p in range(P):
        for t in range(valid[p]):
            E = np.eye(S)
            K = np.zeros(S)
            Q = np.zeros(S)
            for j in range(W):
                E[ws[p, t, j], ws[p, t, j]] = math.exp(g[p, t, j])
                K[ws[p, t, j]] += k[p, t, j]
            for i in range(rs.shape[2]):
                Q[rs[p, t, i]] += q[p, t, i]
            B[p] = (np.eye(S) - beta[p, t] * np.outer(K, K)) @ E @ B[p] + beta[p, t] * np.outer(K, v[p, t])
            out[p, t] = Q @ B[p]
    return out, B.reshape(P * S, -1)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_sequential_matches_dense_brute_force(seed):
    _, x = rand_case(seed=seed)
    o, B = oracle.sequential(*args(x))
    o2, B2 = dense_brute_force(*args(x))
    assert rel(o, o2) < 1e-12
    assert rel(B, B2) < 1e-12


def test_hand_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "hand_example.json")))
    T, W, R = ex["T"], ex["W"], ex["R"]
    g = np.where(np.array(ex["log_decay_is_ln_half"]), math.log(0.5), 0.0)
    o, B = oracle.sequential(np.array(ex["bank0"], float), np.array(ex["write_slots"])[None],
                             np.array(ex["write_w"], float)[None], g[None],
                             np.array(ex["beta"], float)[None], np.array(ex["v"], float)[None],
                             np.array(ex["read_slots"])[None], np.array(ex["read_w"], float)[None],
                             np.array([T]))
    np.testing.assert_allclose(o[0], np.array(ex["readings"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(B, np.array(ex["bank_final"]), rtol=0, atol=1e-12)
    # the chunked form reaches the same numbers at every chunk size
    for C in (1, 2, 3):
        oc, Bc, _ = oracle.chunked(C, np.array(ex["bank0"], float), np.array(ex["write_slots"])[None],
                                   np.array(ex["write_w"], float)[None], g[None],
                                   np.array(ex["beta"], float)[None], np.array(ex["v"], float)[None],
                                   np.array(ex["read_slots"])[None],
                                   np.array(ex["read_w"], float)[None], np.array([T]))
        np.testing.assert_allclose(oc[0], np.array(ex["readings"]), rtol=0, atol=1e-12)
        np.testing.assert_allclose(Bc, np.array(ex["bank_final"]), rtol=0, atol=1e-12)


def test_scalar_delta_rule_closed_form():
    """W = R = 1 on one slot, weight 1, g = 0: B_t = (1 - beta) B_{t-1} + beta v, so with
    constant beta and v, B_t - v = (1 - beta)^t (B_0 - v) and o_t = B_t."""
    T, D, beta, S = 40, 4, 0.3, 5
    rng = np.random.default_rng(3)
    bank = rng.standard_normal((S, D))
    v = rng.standard_normal(D)
    ws = np.full((1, T, 1), 2)
    o, B = oracle.sequential(bank, ws, np.ones((1, T, 1)), np.zeros((1, T, 1)),
                             np.full((1, T), beta), np.tile(v, (1, T, 1)), ws, np.ones((1, T, 1)))
    for t in range(T):
        expect = v + (1 - beta) ** (t + 1) * (bank[2] - v)
        np.testing.assert_allclose(o[0, t], expect, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(np.delete(B, 2, 0), np.delete(bank, 2, 0))


def test_beta_one_overwrites():
    """beta = 1, one write slot of weight 1: the written row becomes v (d + (v - d))."""
    T, D, S = 10, 3, 6
    rng = np.random.default_rng(4)
    bank = rng.standard_normal((S, D))
    ws = rng.integers(0, S, (1, T, 1))
    v = rng.standard_normal((1, T, D))
    g = -rng.random((1, T, 1))
    o, B = oracle.sequential(bank, ws, np.ones((1, T, 1)), g, np.ones((1, T)), v, ws,
                             np.ones((1, T, 1)))
    np.testing.assert_allclose(o[0], v[0], rtol=1e-13, atol=1e-13)


def test_pure_decay():
    """beta = 0: B_T[s] = exp(sum of g over the writes of s) B_0[s]; unwritten rows keep."""
    wl, x = rand_case(P=1, T=30, S=12, W=3, ragged=False, zipf=False, seed=5)
    x["beta"] = np.zeros_like(x["beta"])
    o, B = oracle.sequential(*args(x))
    gsum = np.zeros(12)
    for t in range(30):
        for j in range(3):
            gsum[x["ws"][0, t, j]] += x["g"][0, t, j]
    np.testing.assert_allclose(B, np.exp(gsum)[:, None] * x["bank"], rtol=1e-13, atol=1e-15)


def test_padding_tokens_touch_nothing():
    wl, x = rand_case(P=3, T=20, seed=6, ragged=False)
    x["valid"] = np.array([0, 7, 20], np.int32)
    o, B = oracle.sequential(*args(x))
    assert not o[0].any() and not o[1, 7:].any()
    np.testing.assert_array_equal(B[:wl.S], x["bank"][:wl.S])
    # garbage in the padding entries changes nothing
    y = dict(x)
    for key in ("k", "g", "v", "q"):
        y[key] = x[key].copy()
    y["k"][1, 7:] = 123.0
    y["v"][1, 7:] = -9.0
    o2, B2 = oracle.sequential(*args(y))
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(B, B2)


def test_rejects_repeated_write_slot():
    _, x = rand_case(P=1, T=5, S=9, W=3, ragged=False, seed=7)
    x["ws"] = x["ws"].copy()
    x["ws"][0, 2, 1] = x["ws"][0, 2, 0]
    with pytest.raises(ValueError):
        oracle.sequential(*args(x))
    x["ws"][0, 2, 1] = 9          # out of range
    with pytest.raises(ValueError):
        oracle.sequential(*args(x))


# ---------------------------------------------------------------------------------------
# chunked form
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("C", [1, 2, 3, 5, 8, 16, 23, 64])
def test_chunked_equals_sequential(C):
    """The chunked form reproduces the token loop (memory_ops.py SDMWriteRead docstring)."""
    _, x = rand_case(P=3, T=23, S=7, D=4, W=3, R=3, seed=11)
    o, B = oracle.sequential(*args(x))
    oc, Bc, _ = oracle.chunked(C, *args(x))
    assert rel(oc, o) < 1e-12
    assert rel(Bc, B) < 1e-12


def test_chunked_equals_sequential_workload0():
    wl = si.WORKLOADS[0]
    x = oracle.from_stored(si.generate(wl), wl.dtype)
    o, B = oracle.sequential(*args(x))
    for C in (16, 32, 64, 128, 256):
        oc, Bc, _ = oracle.chunked(C, *args(x))
        assert rel(oc, o) < 1e-10 and rel(Bc, B) < 1e-10


def test_phase1_intermediates_and_solve():
    _, x = rand_case(P=1, T=16, S=5, D=3, W=3, R=2, ragged=False, seed=12)
    C = 16
    _, _, d = oracle.chunked(C, *args(x), debug=(0, 0))
    A, QK, X, QX = d["A"], d["QK"], d["X"], d["QX"]
    assert not np.triu(A).any(), "A is strictly lower triangular"
    assert not np.triu(QK, 1).any(), "QK is lower triangular (diagonal included)"
    assert np.count_nonzero(A) > 10
    L = np.tril(x["beta"][0][:, None] * A, -1)
    np.testing.assert_allclose(X @ (np.eye(C) + L), np.eye(C), atol=1e-12)
    np.testing.assert_allclose(np.diag(X), 1.0)
    np.testing.assert_allclose(QX, QK @ X, atol=1e-12)
    # Lw: running sum of g over the writes of a slot, by brute force
    ws, g = x["ws"][0], x["g"][0]
    for t in range(C):
        for j in range(3):
            s = ws[t, j]
            expect = sum(g[u, jj] for u in range(t + 1) for jj in range(3) if ws[u, jj] == s)
            assert abs(d["lw"][t, j] - expect) < 1e-14
        for i in range(2):
            s = x["rs"][0][t, i]
            expect = sum(g[u, jj] for u in range(t + 1) for jj in range(3) if ws[u, jj] == s)
            assert abs(d["lr"][t, i] - expect) < 1e-14


def test_solve_padded_chunk_and_no_repeats():
    # ragged chunk: rows past the valid tokens are identity rows; the leading block of X is
    # the inverse of the leading block of I + L
    _, x = rand_case(P=1, T=16, S=4, D=2, W=2, R=2, ragged=False, seed=13)
    x["valid"] = np.array([11], np.int32)
    _, _, d = oracle.chunked(16, *args(x), debug=(0, 0))
    n = 11
    L = np.tril(x["beta"][0][:n, None] * d["A"][:n, :n], -1)
    np.testing.assert_allclose(d["X"][:n, :n], np.linalg.inv(np.eye(n) + L), atol=1e-12)
    np.testing.assert_array_equal(d["X"][n:], np.eye(16)[n:])
    # no slot repeats inside the chunk: A = 0 and X = I
    _, y = rand_case(P=1, T=8, S=100000, D=2, W=2, R=2, ragged=False, zipf=False, seed=14)
    assert len(set(y["ws"][0].reshape(-1).tolist())) == 16
    _, _, d2 = oracle.chunked(8, *args(y), debug=(0, 0))
    assert not d2["A"].any()
    np.testing.assert_array_equal(d2["X"], np.eye(8))


# ---------------------------------------------------------------------------------------
# dedup plan
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1])
def test_plan_matches_brute_force_grouping(seed):
    rng = np.random.default_rng(seed)
    n, width = 9, 4
    slots = np.stack([rng.choice(6, width, replace=False) for _ in range(n)])
    pl = oracle.plan(slots)
    entries = [(int(slots[e // width, e % width]), e) for e in range(n * width)]
    order = sorted(entries)            # by (slot, entry)
    assert pl["perm"].tolist() == [e for _, e in order]
    for pos, (s, e) in enumerate(order):
        members = [ee for ss, ee in entries if ss == s]
        assert pl["group_start"][pos] == (e == min(members))
        assert pl["owner"][pos] == (e == max(members))
        assert pl["only"][pos] == (len(members) == 1)
    assert pl["groups"] == len(set(slots.reshape(-1).tolist()))


# ---------------------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("with_final", [False, True])
def test_backward_finite_differences_and_restore(with_final):
    """Loss = <dO, readings> (+ <G, final bank>): every gradient against central
    differences of the token loop."""
    _, x = rand_case(P=2, T=9, S=5, D=3, W=2, R=2, seed=21, ragged=False)
    x["valid"] = np.array([9, 6], np.int32)
    rng = np.random.default_rng(22)
    dO = rng.standard_normal((2, 9, 3))
    G = rng.standard_normal((10, 3)) if with_final else None
    gr = oracle.backward(*args(x), dO, grad_final_bank=G)
    np.testing.assert_array_equal(gr["restored_bank"], x["bank"])

    def loss(y):
        o, B = oracle.sequential(*args(y))
        return float((o * dO).sum()) + (float((B * G).sum()) if with_final else 0.0)

    h = 1e-6
    for key, gkey in (("bank", "grad_bank"), ("v", "grad_v"), ("beta", "grad_beta"),
                      ("k", "grad_write_w"), ("g", "grad_log_decay"), ("q", "grad_read_w")):
        base = x[key]
        flat_idx = rng.choice(base.size, min(base.size, 12), replace=False)
        for fi in flat_idx:
            yp, ym = dict(x), dict(x)
            yp[key] = base.copy()
            ym[key] = base.copy()
            yp[key].reshape(-1)[fi] += h
            ym[key].reshape(-1)[fi] -= h
            fd = (loss(yp) - loss(ym)) / (2 * h)
            an = gr[gkey].reshape(-1)[fi]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (key, fi, fd, an)


# ---------------------------------------------------------------------------------------
# reverse mode from a stored snapshot (memory_ops.py sdm_write_read: snapshot_quant)
# ---------------------------------------------------------------------------------------

GRAD_KEYS = ("grad_bank", "grad_v", "grad_beta", "grad_write_w", "grad_log_decay",
             "grad_read_w")


def bf16_of_f32(x):
    """bfloat16 rounding (to nearest even) of the float32 value of x, by torch's conversion."""
    import torch

    return torch.from_numpy(np.asarray(x, np.float64)).float().bfloat16().double().numpy()


def fp8_of_f32(x):
    """float8_e4m3fn rounding (to nearest even) of the float32 value of x, by torch's
    conversion (finite inputs inside the format's range)."""
    import torch

    return torch.from_numpy(np.asarray(x, np.float64)).float().to(torch.float8_e4m3fn).double().numpy()


@pytest.mark.parametrize("C", [1, 3, 8, 64])
@pytest.mark.parametrize("with_final", [False, True])
def test_backward_snapshot_none_is_the_reverse_mode(C, with_final):
    """With an unrounded snapshot the chunked reverse pass is the token loop's reverse mode,
    bit for bit, at any chunk size (rows written in several chunks, ragged valid tokens)."""
    _, x = rand_case(P=2, T=23, S=7, D=3, W=3, R=2, seed=41)
    rng = np.random.default_rng(42)
    dO = rng.standard_normal((2, 23, 3))
    G = rng.standard_normal((14, 3)) if with_final else None
    ref = oracle.backward(*args(x), dO, grad_final_bank=G)
    got = oracle.backward_snapshot(*args(x), dO, chunk_size=C, snapshot="none", grad_final_bank=G)
    for key in GRAD_KEYS + ("restored_bank",):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)


def test_backward_snapshot_bf16_restores_rounded_initial_rows():
    """A bfloat16 snapshot leaves every row some valid token writes at bf16(its initial
    value), and every other row untouched, whatever the chunking."""
    _, x = rand_case(P=2, T=37, S=11, D=4, W=3, R=2, seed=43)
    dO = np.random.default_rng(44).standard_normal((2, 37, 4))
    written = np.zeros(2 * 11, bool)
    for p in range(2):
        for t in range(x["valid"][p]):
            written[p * 11 + x["ws"][p, t]] = True
    expect = x["bank"].copy()
    expect[written] = bf16_of_f32(x["bank"][written])
    for C in (4, 16):
        got = oracle.backward_snapshot(*args(x), dO, chunk_size=C, snapshot="bf16")
        np.testing.assert_array_equal(got["restored_bank"], expect)


@pytest.mark.parametrize("mode", ["bf16", "fp8"])
def test_backward_snapshot_is_the_reverse_mode_of_the_rounded_bank(mode):
    """When no chunk touches a row that an earlier chunk wrote, every chunk starts from the
    rounded initial values of the rows it writes (and of later chunks' rows it reads), so
    the bf16- or fp8-snapshot backward equals the exact reverse mode run on the bank whose
    written rows are rounded beforehand (torch's conversion)."""
    rnd = bf16_of_f32 if mode == "bf16" else fp8_of_f32
    P, T, C, S, D, W, R = 2, 24, 6, 40, 3, 2, 3
    Nt = T // C
    K = S // (Nt + 1)                      # chunk c writes slots [cK, (c+1)K); the top K stay unwritten
    rng = np.random.default_rng(45)
    ws = np.zeros((P, T, W), np.int32)
    rs = np.zeros((P, T, R), np.int32)
    for p in range(P):
        for t in range(T):
            c = t // C
            ws[p, t] = c * K + rng.choice(K, W, replace=False)
            rs[p, t] = rng.integers(c * K, S, R)          # its own range, later ones, unwritten
    x = {"bank": rng.standard_normal((P * S, D)) * 0.5, "ws": ws,
         "k": rng.uniform(0.1, 0.9, (P, T, W)), "g": -0.1 * rng.uniform(0, 1, (P, T, W)),
         "beta": rng.uniform(0.2, 0.9, (P, T)), "v": rng.standard_normal((P, T, D)), "rs": rs,
         "q": rng.uniform(0.1, 0.9, (P, T, R)), "valid": np.array([T, T - 5], np.int32)}
    dO = rng.standard_normal((P, T, D))
    written = np.zeros(P * S, bool)
    for p in range(P):
        for t in range(x["valid"][p]):
            written[p * S + ws[p, t]] = True
    y = dict(x)
    y["bank"] = x["bank"].copy()
    y["bank"][written] = rnd(x["bank"][written])
    ref = oracle.backward(*args(y), dO)
    got = oracle.backward_snapshot(*args(x), dO, chunk_size=C, snapshot=mode)
    for key in GRAD_KEYS + ("restored_bank",):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    # and the rounding changes the gradients (the snapshot is not silently exact)
    exact = oracle.backward(*args(x), dO)
    assert rel(got["grad_write_w"], exact["grad_write_w"]) > 1e-6


def test_backward_snapshot_fp8_restores_rounded_initial_rows():
    """An fp8 snapshot leaves every row some valid token writes at fp8(its initial value)
    (torch's float8_e4m3fn conversion, over normal and subnormal magnitudes), every other row
    untouched; values past the largest finite code saturate to +-448 (the reading for the
    format without infinity)."""
    _, x = rand_case(P=2, T=37, S=11, D=4, W=3, R=2, seed=46)
    rng = np.random.default_rng(47)
    x["bank"] = x["bank"] * np.exp(rng.uniform(-12, 5, x["bank"].shape))
    dO = rng.standard_normal((2, 37, 4))
    written = np.zeros(2 * 11, bool)
    for p in range(2):
        for t in range(x["valid"][p]):
            written[p * 11 + x["ws"][p, t]] = True
    big = np.flatnonzero(written)[:2]
    x["bank"][big[0], 0], x["bank"][big[1], 1] = 1000.0, -5000.0
    b = x["bank"][written]
    inside = np.abs(b) <= 448
    expect = x["bank"].copy()
    expect[written] = np.where(inside, fp8_of_f32(np.clip(b, -448, 448)), np.sign(b) * 448)
    got = oracle.backward_snapshot(*args(x), dO, chunk_size=8, snapshot="fp8")
    np.testing.assert_array_equal(got["restored_bank"], expect)
    assert got["restored_bank"][big[0], 0] == 448.0 and got["restored_bank"][big[1], 1] == -448.0


def test_per_token_gate_gradient_is_the_sum_over_writes():
    """One log-decay per token (the pages' g of width 1) is the per-write form with the gate
    repeated over the token's W writes; its gradient, by central differences of the token
    loop, is the sum of the W per-write gradients."""
    _, x = rand_case(P=2, T=9, S=6, D=3, W=3, R=2, seed=51, ragged=False)
    x["valid"] = np.array([9, 7], np.int32)
    gt = x["g"][..., 0].copy()                       # [P, T]
    x["g"] = np.repeat(gt[..., None], 3, axis=2)
    dO = np.random.default_rng(52).standard_normal((2, 9, 3))
    gr = oracle.backward(*args(x), dO)
    dgt = gr["grad_log_decay"].sum(axis=2)

    def loss(gate):
        y = dict(x)
        y["g"] = np.repeat(gate[..., None], 3, axis=2)
        return float((oracle.sequential(*args(y))[0] * dO).sum())

    h = 1e-6
    for p in range(2):
        for t in range(9):
            gp, gm = gt.copy(), gt.copy()
            gp[p, t] += h
            gm[p, t] -= h
            fd = (loss(gp) - loss(gm)) / (2 * h)
            assert abs(fd - dgt[p, t]) <= 1e-6 * max(1.0, abs(fd)), (p, t, fd, dgt[p, t])


# ---------------------------------------------------------------------------------------
# layer I/O (memory_ops.py "Layer I/O")
# ---------------------------------------------------------------------------------------

def test_head_split_is_the_pages_row_map_and_merge_inverts_it():
    """dst row (b*H + h)*T + t = src row (b*T + t)*H + h, by explicit loops over the rows of
    the flattened arrays; merge after split is the identity."""
    B, T, H, K = 2, 5, 3, 4
    x = np.arange(B * T * H * K, dtype=np.float64).reshape(B, T, H * K)
    y = oracle.head_split(x, H)
    src, dst = x.reshape(-1, K), y.reshape(-1, K)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                np.testing.assert_array_equal(dst[(b * H + h) * T + t], src[(b * T + t) * H + h])
    np.testing.assert_array_equal(oracle.head_merge(y, H), x)


def test_bank_sum_of_expand_is_b_times_the_bank():
    p = np.random.default_rng(91).standard_normal((7, 3))
    np.testing.assert_array_equal(oracle.bank_expand(p, 4)[2], p)
    np.testing.assert_allclose(oracle.bank_sum(oracle.bank_expand(p, 4)), 4 * p, rtol=1e-15)
