"""CPU oracle of the sparse-delta-memory write/read (fp64, plain C, loaded with ctypes).

TEST INFRASTRUCTURE ONLY: the checker of the CUDA path. Only the test-suite, the smoke
check and the benchmark's CPU-baseline leg may import this package; the product path never
does, and the two share no code (the seeded input generator ``sdm_inputs`` excepted).

Functions (every one cites the definition it follows in ``sdm_oracle.c``):
  sequential  the reference token loop (memory_ops.py, SDMWriteRead docstring)
  chunked     the Phase 1 / solve / Phase 2 form from the module docstrings, with the
              intermediates of one chunk exposed
  plan        the sorted kind row, groups, owners and single-entry flags of one chunk
              (phase2_kernels.py module docstring)
  backward    reverse mode of the token loop, with the bank restored
  backward_snapshot
              the reverse mode as the chunked backward runs it from a stored (optionally
              bfloat16) snapshot of the rows each chunk writes (memory_ops.py snapshot_quant)
  head_split, head_merge, bank_expand, bank_sum
              the layer I/O around the op (memory_ops.py "Layer I/O"), as array rearranges
  product_key (module)
              the exact top-k over product-key slots, the pages' staged selection rule
              (product_key_topk.py), with its backward

Pins (tests/test_oracle.py): dense brute force, closed forms (scalar delta rule, pure
decay), chunk-size invariance, the solve identity, brute-force grouping and central
finite differences.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles the oracle with gcc (OpenMP over streams, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
_dbl_or_null = ctypes.c_void_p


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            I = ctypes.c_int
            lib.sdm_oracle_sequential.argtypes = [I, I, I, I, I, I, _f64p, _i32p, _f64p, _f64p,
                                                  _f64p, _f64p, _i32p, _f64p, _i32p, _f64p, I]
            lib.sdm_oracle_sequential.restype = I
            lib.sdm_oracle_chunked.argtypes = ([I] * 7 + [_f64p, _i32p, _f64p, _f64p, _f64p, _f64p,
                                                          _i32p, _f64p, _i32p, _f64p, I, I]
                                               + [_dbl_or_null] * 12)
            lib.sdm_oracle_chunked.restype = I
            lib.sdm_oracle_plan.argtypes = [I, I, _i32p, _i32p, _u8p, _u8p, _u8p]
            lib.sdm_oracle_plan.restype = I
            lib.sdm_oracle_backward.argtypes = [I, I, I, I, I, I, _f64p, _i32p, _f64p, _f64p,
                                                _f64p, _f64p, _i32p, _f64p, _i32p, _f64p,
                                                _dbl_or_null, _f64p, _f64p, _f64p, _f64p,
                                                _f64p, _f64p, I]
            lib.sdm_oracle_backward.restype = I
            lib.sdm_oracle_backward_snapshot.argtypes = [I, I, I, I, I, I, I, I, _f64p, _i32p,
                                                         _f64p, _f64p, _f64p, _f64p, _i32p,
                                                         _f64p, _i32p, _f64p, _dbl_or_null,
                                                         _f64p, _f64p, _f64p, _f64p, _f64p,
                                                         _f64p, I]
            lib.sdm_oracle_backward_snapshot.restype = I
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.int32)


def _check(rc: int, what: str) -> None:
    if rc == -1:
        raise ValueError(f"oracle {what}: invalid input (slot out of range, repeated write "
                         "slot in a token, or bad sizes)")
    if rc == -2:
        raise MemoryError(f"oracle {what}: out of host memory")
    if rc < 0:
        raise RuntimeError(f"oracle {what}: error {rc}")


def _dims(bank, ws, rs, v):
    P, T, W = ws.shape
    R = rs.shape[2]
    D = v.shape[2]
    S = bank.shape[0] // P
    if bank.shape != (P * S, D):
        raise ValueError(f"bank {bank.shape} does not match P={P}, D={D}")
    return P, T, S, D, W, R


def sequential(bank, ws, k, g, beta, v, rs, q, valid=None, nthreads: int = 1
               ) -> Tuple[np.ndarray, np.ndarray]:
    """The token loop in fp64. Arrays: bank [P*S, D]; ws, k, g [P, T, W]; beta [P, T];
    v [P, T, D]; rs, q [P, T, R]; valid [P] (default: all T). Returns (readings [P, T, D],
    final bank [P*S, D]); the inputs are not modified."""
    B = _f64(bank).copy()
    ws, rs = _i32(ws), _i32(rs)
    P, T, S, D, W, R = _dims(B, ws, rs, v)
    valid = _i32(np.full(P, T) if valid is None else valid)
    out = np.zeros((P, T, D), np.float64)
    rc = _load().sdm_oracle_sequential(P, T, S, D, W, R, B, ws, _f64(k), _f64(g), _f64(beta),
                                       _f64(v), rs, _f64(q), valid, out, int(nthreads))
    _check(rc, "sequential")
    return out, B


_DBG_FIELDS = ("lw", "lr", "gw", "qw", "dw", "A", "QK", "X", "QX", "retrieved", "inter",
               "delta_v")


def chunked(C: int, bank, ws, k, g, beta, v, rs, q, valid=None,
            debug: Optional[Tuple[int, int]] = None):
    """The chunked form in fp64 with chunks of C tokens. Returns (readings, final bank,
    intermediates of chunk ``debug`` = (stream, chunk) as a dict, or None)."""
    B = _f64(bank).copy()
    ws, rs = _i32(ws), _i32(rs)
    P, T, S, D, W, R = _dims(B, ws, rs, v)
    valid = _i32(np.full(P, T) if valid is None else valid)
    out = np.zeros((P, T, D), np.float64)
    dbg = None
    ptrs = [None] * 12
    if debug is not None:
        shapes = {"lw": (C, W), "lr": (C, R), "gw": (C, W), "qw": (C, R), "dw": (C, W),
                  "A": (C, C), "QK": (C, C), "X": (C, C), "QX": (C, C),
                  "retrieved": (C, D), "inter": (C, D), "delta_v": (C, D)}
        dbg = {f: np.zeros(shapes[f], np.float64) for f in _DBG_FIELDS}
        ptrs = [dbg[f].ctypes.data for f in _DBG_FIELDS]
    dp, dc = debug if debug is not None else (-1, -1)
    rc = _load().sdm_oracle_chunked(P, T, C, S, D, W, R, B, ws, _f64(k), _f64(g), _f64(beta),
                                    _f64(v), rs, _f64(q), valid, out, dp, dc, *ptrs)
    _check(rc, "chunked")
    return out, B, dbg


def plan(slots) -> Dict[str, np.ndarray]:
    """Dedup plan of one kind of one chunk: ``slots`` [n, width] of the chunk's valid tokens.
    Returns perm (entry e = t*width + j at each sorted position), group_start, owner, only
    (uint8 flags per sorted position) and the group count."""
    s = _i32(slots)
    n, width = s.shape
    m = n * width
    perm = np.zeros(m, np.int32)
    gs, ow, on = (np.zeros(m, np.uint8) for _ in range(3))
    groups = _load().sdm_oracle_plan(n, width, s.reshape(-1), perm, gs, ow, on)
    _check(min(groups, 0), "plan")
    return {"perm": perm, "group_start": gs, "owner": ow, "only": on, "groups": int(groups)}


def backward(bank, ws, k, g, beta, v, rs, q, valid, grad_readings, nthreads: int = 1,
             grad_final_bank=None):
    """Reverse mode of the token loop. ``grad_final_bank`` (optional, [P*S, D]) is the loss
    gradient with respect to the final bank. Returns a dict with grad_bank [P*S, D] (with
    respect to the initial bank), grad_v, grad_beta, grad_write_w, grad_log_decay,
    grad_read_w and restored_bank (the bank after forward + backward, which equals the
    initial bank)."""
    B = _f64(bank).copy()
    ws, rs = _i32(ws), _i32(rs)
    P, T, S, D, W, R = _dims(B, ws, rs, v)
    valid = _i32(np.full(P, T) if valid is None else valid)
    dB = np.zeros((P * S, D), np.float64)
    dv = np.zeros((P, T, D), np.float64)
    db = np.zeros((P, T), np.float64)
    dk = np.zeros((P, T, W), np.float64)
    dg = np.zeros((P, T, W), np.float64)
    dq = np.zeros((P, T, R), np.float64)
    gfb = None
    if grad_final_bank is not None:
        gfb = _f64(grad_final_bank)
        if gfb.shape != (P * S, D):
            raise ValueError(f"grad_final_bank must be {(P * S, D)}, got {gfb.shape}")
    rc = _load().sdm_oracle_backward(P, T, S, D, W, R, B, ws, _f64(k), _f64(g), _f64(beta),
                                     _f64(v), rs, _f64(q), valid, _f64(grad_readings),
                                     None if gfb is None else gfb.ctypes.data, dB, dv, db, dk,
                                     dg, dq, int(nthreads))
    _check(rc, "backward")
    return {"grad_bank": dB, "grad_v": dv, "grad_beta": db, "grad_write_w": dk,
            "grad_log_decay": dg, "grad_read_w": dq, "restored_bank": B}


SNAPSHOT_MODES = {"none": 0, "bf16": 1, "fp8": 2}


def backward_snapshot(bank, ws, k, g, beta, v, rs, q, valid, grad_readings, *, chunk_size: int,
                      snapshot: str = "bf16", nthreads: int = 1, grad_final_bank=None):
    """Reverse mode as the chunked backward runs it from a stored snapshot: chunks in reverse,
    each restoring its written rows to Q(their value at the chunk start) ("none": Q is the
    identity; "bf16": float32 then bfloat16 rounding, to nearest even; "fp8": float32 then
    float8_e4m3fn rounding, to nearest even, saturating at 448), re-running the chunk and
    taking its reverse pass. Same outputs as ``backward``; ``restored_bank`` holds Q(initial
    value) on every row a valid token writes."""
    B = _f64(bank).copy()
    ws, rs = _i32(ws), _i32(rs)
    P, T, S, D, W, R = _dims(B, ws, rs, v)
    valid = _i32(np.full(P, T) if valid is None else valid)
    dB = np.zeros((P * S, D), np.float64)
    dv = np.zeros((P, T, D), np.float64)
    db = np.zeros((P, T), np.float64)
    dk = np.zeros((P, T, W), np.float64)
    dg = np.zeros((P, T, W), np.float64)
    dq = np.zeros((P, T, R), np.float64)
    gfb = None
    if grad_final_bank is not None:
        gfb = _f64(grad_final_bank)
        if gfb.shape != (P * S, D):
            raise ValueError(f"grad_final_bank must be {(P * S, D)}, got {gfb.shape}")
    rc = _load().sdm_oracle_backward_snapshot(
        P, T, int(chunk_size), S, D, W, R, SNAPSHOT_MODES[snapshot], B, ws, _f64(k), _f64(g),
        _f64(beta), _f64(v), rs, _f64(q), valid, _f64(grad_readings),
        None if gfb is None else gfb.ctypes.data, dB, dv, db, dk, dg, dq, int(nthreads))
    _check(rc, "backward_snapshot")
    return {"grad_bank": dB, "grad_v": dv, "grad_beta": db, "grad_write_w": dk,
            "grad_log_decay": dg, "grad_read_w": dq, "restored_bank": B}


# ---------------------------------------------------------------------------------------
# layer I/O (memory_ops.py "Layer I/O"): the definitions as array rearranges
# ---------------------------------------------------------------------------------------

def head_split(x: np.ndarray, H: int) -> np.ndarray:
    """rearrange 'b t (h k) -> (b h) t k': [B, T, H*K] -> [B*H, T, K]."""
    B, T, HK = x.shape
    return x.reshape(B, T, H, HK // H).transpose(0, 2, 1, 3).reshape(B * H, T, HK // H)


def head_merge(x: np.ndarray, H: int) -> np.ndarray:
    """rearrange '(b h) t d -> b t (h d)': [B*H, T, D] -> [B, T, H*D]."""
    BH, T, D = x.shape
    return x.reshape(BH // H, H, T, D).transpose(0, 2, 1, 3).reshape(BH // H, T, H * D)


def bank_expand(param: np.ndarray, B: int) -> np.ndarray:
    """[S, D] -> [B, S, D], every batch copy the parameter bank."""
    return np.broadcast_to(param, (B,) + param.shape).copy()


def bank_sum(x: np.ndarray) -> np.ndarray:
    """[B, S, D] -> [S, D], the sum over the batch in float64."""
    return np.asarray(x, np.float64).sum(axis=0)


def from_stored(inputs: Dict[str, np.ndarray], dtype: str) -> Dict[str, np.ndarray]:
    """The fp64 values of a generated input set (see ``sdm_inputs.generate``)."""
    import sdm_inputs
    f = lambda name: sdm_inputs.stored_to_f64(inputs[name], dtype)  # noqa: E731
    out = {"bank": f("bank"), "ws": inputs["write_slots"], "k": f("write_w"),
           "g": inputs["log_decay"].astype(np.float64), "beta": inputs["beta"].astype(np.float64),
           "v": f("v"), "rs": inputs["read_slots"], "q": f("read_w"), "valid": inputs["valid"]}
    if "grad_readings" in inputs:
        out["grad_readings"] = f("grad_readings")
    return out
