"""Seeded synthetic inputs for the chunked sparse-delta-memory (SDM) write/read.

This module is the only code that the CUDA path and the CPU oracle share. It draws the
inputs of a workload and rounds them to the stored dtypes; it holds none of the write/read
arithmetic itself.

Workloads (the five configurations the SDM pages' op is exercised on; the sizes are the
ones named beside each entry of ``WORKLOADS``):

  * bank rows N(0, 0.02), rounded to the bank dtype;
  * write/read slots distinct per token, either uniform over the S rows of a stream or
    Zipf(s) over them (rank r in 1..S with probability proportional to r**-s, slot id
    r - 1, drawn from an inverse-CDF table; a duplicate inside a token is redrawn until the
    token's slots are distinct), or the per-token mix "half Zipf(1.2), half uniform";
  * write/read weights: softmax of N(0, 1) draws over the token's slots, in the bank dtype;
  * log-decay g = -0.1 * softplus(N(0, 1)) per write entry, float32;
  * beta = sigmoid(N(0, 1)) per token, float32;
  * v ~ N(0, 1) in the bank dtype;
  * valid tokens per stream: all T, or uniform in [T/2, T] ("ragged");
  * the upstream gradient of the readings (backward workloads): N(0, 1) in the bank dtype.

Inputs of padding tokens (t >= valid[p]) are staged as zeros.

bfloat16 arrays are returned as their uint16 bit patterns (round to nearest even from the
float32 value).
"""

from __future__ import annotations

import dataclasses
import functools
from typing import Dict, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    P: int            # parallel streams
    T: int            # tokens per stream
    C: int            # chunk size
    S: int            # bank rows per stream
    D: int            # columns per row (head_dim)
    W: int            # write slots per token
    R: int            # read slots per token
    dtype: str        # bank dtype: "f32" or "bf16"
    slots: str        # "uniform", "zipf1.1", "mix" (half Zipf(1.2), half uniform, per token)
    ragged: bool      # valid tokens per stream uniform in [T/2, T]
    seed: int
    backward: bool = False

    @property
    def Nt(self) -> int:
        return -(-self.T // self.C)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five configurations (index = the seed, as the workload descriptions fix seed 0 for
# the first and leave the rest open).
WORKLOADS = {
    0: Workload("p1_t256_c16_s1024_d64_f32_w4", 1, 256, 16, 1024, 64, 4, 4, "f32", "uniform",
                False, 0),
    1: Workload("p8_t4096_c64_s65536_d128_bf16_w16_zipf1.1", 8, 4096, 64, 65536, 128, 16, 16,
                "bf16", "zipf1.1", False, 1),
    2: Workload("p32_t8192_c64_s262144_d128_bf16_w32_zipf1.1_ragged", 32, 8192, 64, 262144,
                128, 32, 32, "bf16", "zipf1.1", True, 2),
    3: Workload("p16_t4096_c128_s131072_d128_f32_w64_fwdbwd", 16, 4096, 128, 131072, 128, 64,
                64, "f32", "uniform", False, 3, backward=True),
    4: Workload("p4_t16384_c256_s1048576_d256_bf16_w256_mix", 4, 16384, 256, 1048576, 256, 256,
                256, "bf16", "mix", False, 4),
}


# ----------------------------------------------------------------------------------------
# dtype helpers
# ----------------------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of bfloat16(x), round to nearest even from float32."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def to_stored(x: np.ndarray, dtype: str) -> np.ndarray:
    """x (float64/float32) as the stored array of ``dtype`` (float32, or bf16 bits)."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


def stored_to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """The exact values of a stored array as float64."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f32(x).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# ----------------------------------------------------------------------------------------
# slot draws
# ----------------------------------------------------------------------------------------

@functools.lru_cache(maxsize=8)
def _zipf_cdf(S: int, s: float) -> np.ndarray:
    w = np.arange(1, S + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    return cdf / cdf[-1]


class _Zipf:
    """Inverse-CDF sampler of Zipf(s) ranks 1..S, returned as slot ids r - 1."""

    def __init__(self, S: int, s: float):
        self.cdf = _zipf_cdf(S, s)
        self.S = S

    def draw(self, rng: np.random.Generator, n) -> np.ndarray:
        u = rng.random(n)
        r = np.searchsorted(self.cdf, u, side="right")
        return np.minimum(r, self.S - 1).astype(np.int32)


def _distinct_rows(x: np.ndarray, redraw) -> np.ndarray:
    """Makes every row of x distinct: a value equal to an earlier one in its row (in column
    order) is redrawn with ``redraw(rng_mask)`` until none repeats."""
    rows = np.arange(x.shape[0])
    while True:
        sub = x[rows]
        order = np.argsort(sub, axis=1, kind="stable")
        srt = np.take_along_axis(sub, order, 1)
        dup_sorted = np.zeros(srt.shape, dtype=bool)
        dup_sorted[:, 1:] = srt[:, 1:] == srt[:, :-1]
        dup = np.zeros_like(dup_sorted)
        np.put_along_axis(dup, order, dup_sorted, 1)
        bad = dup.any(axis=1)
        if not bad.any():
            return x
        rows = rows[bad]
        dup = dup[bad]
        sub = sub[bad]
        sub[dup] = redraw(dup)
        x[rows] = sub


def draw_slots(rng: np.random.Generator, n_tok: int, width: int, S: int, kind: str) -> np.ndarray:
    """[n_tok, width] int32 slot ids in [0, S), distinct within each row."""
    if width > S:
        raise ValueError(f"{width} distinct slots per token need S >= {width}, got S={S}")
    if kind == "uniform":
        x = rng.integers(0, S, size=(n_tok, width), dtype=np.int64).astype(np.int32)
        return _distinct_rows(x, lambda m: rng.integers(0, S, size=int(m.sum())).astype(np.int32))
    if kind.startswith("zipf"):
        z = _Zipf(S, float(kind[4:]))
        x = z.draw(rng, (n_tok, width))
        return _distinct_rows(x, lambda m: z.draw(rng, int(m.sum())))
    if kind == "mix":
        # Per token: the first half Zipf(1.2)-distinct, the second half uniform and distinct
        # from all earlier slots of the token.
        z = _Zipf(S, 1.2)
        hz = width // 2
        x = np.empty((n_tok, width), dtype=np.int32)
        x[:, :hz] = z.draw(rng, (n_tok, hz))
        x[:, hz:] = rng.integers(0, S, size=(n_tok, width - hz), dtype=np.int64)
        col_is_zipf = np.arange(width) < hz

        def redraw(m):
            cols = np.nonzero(m)[1]
            out = np.empty(cols.shape[0], dtype=np.int32)
            zc = col_is_zipf[cols]
            out[zc] = z.draw(rng, int(zc.sum()))
            out[~zc] = rng.integers(0, S, size=int((~zc).sum()))
            return out
        return _distinct_rows(x, redraw)
    raise ValueError(f"unknown slot distribution {kind!r}")


def _softmax_rows(x: np.ndarray) -> np.ndarray:
    x = x - x.max(axis=-1, keepdims=True)
    e = np.exp(x)
    return e / e.sum(axis=-1, keepdims=True)


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


# ----------------------------------------------------------------------------------------
# workload inputs
# ----------------------------------------------------------------------------------------

_BANK_BLOCK = 1 << 24      # bank values per generator block
_TOKEN_BLOCK = 4096        # tokens per generator block


def _pool_map(fn, items):
    import os
    from concurrent.futures import ThreadPoolExecutor
    workers = max(1, min(len(items), os.cpu_count() or 1, 16))
    if workers == 1:
        return [fn(x) for x in items]
    with ThreadPoolExecutor(workers) as ex:
        return list(ex.map(fn, items))


def generate(wl: Workload, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """All inputs of ``wl`` as numpy arrays (stored dtypes; bf16 as uint16 bits).

    bank [P*S, D]; write_slots [P, T, W] int32; write_w [P, T, W]; log_decay [P, T, W] f32;
    beta [P, T] f32; v [P, T, D]; read_slots [P, T, R] int32; read_w [P, T, R];
    valid [P] int32; grad_readings [P, T, D] (backward workloads only).

    The draws are made in fixed blocks (bank values, then tokens), each from its own child
    of the seed, so the arrays do not depend on the number of threads used to fill them.
    """
    P, T, S, D, W, R = wl.P, wl.T, wl.S, wl.D, wl.W, wl.R
    root = np.random.SeedSequence(wl.seed if seed is None else seed)
    top, bank_seq, tok_seq = root.spawn(3)
    out: Dict[str, np.ndarray] = {}

    bank = np.empty((P * S, D), dtype=np.uint16 if wl.dtype == "bf16" else np.float32)
    flat = bank.reshape(-1)
    nb = -(-flat.size // _BANK_BLOCK)

    def bank_block(args):
        i, ss = args
        r = np.random.default_rng(ss)
        lo = i * _BANK_BLOCK
        n = min(_BANK_BLOCK, flat.size - lo)
        flat[lo:lo + n] = to_stored(r.standard_normal(n, dtype=np.float32) * np.float32(0.02),
                                    wl.dtype)
    _pool_map(bank_block, list(enumerate(bank_seq.spawn(nb))))
    out["bank"] = bank

    rng = np.random.default_rng(top)
    if wl.ragged:
        valid = rng.integers(T // 2, T + 1, size=P).astype(np.int32)
    else:
        valid = np.full(P, T, dtype=np.int32)
    out["valid"] = valid

    n = P * T
    bdt = np.uint16 if wl.dtype == "bf16" else np.float32
    ws = np.empty((n, W), np.int32)
    rs = np.empty((n, R), np.int32)
    kw = np.empty((n, W), bdt)
    qw = np.empty((n, R), bdt)
    g = np.empty((n, W), np.float32)
    beta = np.empty(n, np.float32)
    v = np.empty((n, D), bdt)
    gr = np.empty((n, D), bdt) if wl.backward else None
    tok = np.arange(n)
    pad_all = (tok % T) >= valid[tok // T]
    ntb = -(-n // _TOKEN_BLOCK)

    def token_block(args):
        i, ss = args
        r = np.random.default_rng(ss)
        lo = i * _TOKEN_BLOCK
        hi = min(n, lo + _TOKEN_BLOCK)
        m = hi - lo
        pad = pad_all[lo:hi]
        a_ws = draw_slots(r, m, W, S, wl.slots)
        a_rs = draw_slots(r, m, R, S, wl.slots)
        a_kw = _softmax_rows(r.standard_normal((m, W)))
        a_qw = _softmax_rows(r.standard_normal((m, R)))
        a_g = -0.1 * _softplus(r.standard_normal((m, W)))
        a_beta = _sigmoid(r.standard_normal(m))
        a_v = r.standard_normal((m, D))
        a_gr = r.standard_normal((m, D)) if gr is not None else None
        for a in (a_ws, a_rs, a_kw, a_qw, a_g, a_beta, a_v) + ((a_gr,) if a_gr is not None else ()):
            a[pad] = 0
        ws[lo:hi] = a_ws
        rs[lo:hi] = a_rs
        kw[lo:hi] = to_stored(a_kw, wl.dtype)
        qw[lo:hi] = to_stored(a_qw, wl.dtype)
        g[lo:hi] = a_g
        beta[lo:hi] = a_beta
        v[lo:hi] = to_stored(a_v, wl.dtype)
        if gr is not None:
            gr[lo:hi] = to_stored(a_gr, wl.dtype)
    _pool_map(token_block, list(enumerate(tok_seq.spawn(ntb))))

    out["write_slots"] = ws.reshape(P, T, W)
    out["read_slots"] = rs.reshape(P, T, R)
    out["write_w"] = kw.reshape(P, T, W)
    out["read_w"] = qw.reshape(P, T, R)
    out["log_decay"] = g.reshape(P, T, W)
    out["beta"] = beta.reshape(P, T)
    out["v"] = v.reshape(P, T, D)
    if gr is not None:
        out["grad_readings"] = gr.reshape(P, T, D)
    return out


def small(base: Workload, **kw) -> Workload:
    """A reduced copy of a workload (same distributions and dtype), for quick tests."""
    return base.replace(**kw)
