"""Shared helpers of the GPU parity tests: device copies of generated inputs, one call of the
CUDA path through the C ABI, the oracle on the same inputs, and the error metric.

Error metric (one number per output tensor): max |gpu - oracle| / max |oracle|, bounded by
1e-4 for float32 banks and 2e-2 for bfloat16 banks, for the readings and the final bank.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import sdm_inputs as si
import sparse_addressed_delta_gb300 as sdm

TOL = {"f32": 1e-4, "bf16": 2e-2}


def torch_dtype(wl) -> torch.dtype:
    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def stored_tensor(a: np.ndarray, dtype: str, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.to(device)


def to_device(inputs, wl, device="cuda"):
    f = lambda k: stored_tensor(inputs[k], wl.dtype, device)  # noqa: E731
    i = lambda k: torch.from_numpy(np.ascontiguousarray(inputs[k])).to(device)  # noqa: E731
    return {"bank": f("bank"), "write_slots": i("write_slots"), "write_w": f("write_w"),
            "log_decay": i("log_decay"), "beta": i("beta"), "v": f("v"),
            "read_slots": i("read_slots"), "read_w": f("read_w"), "valid": i("valid")}


def run_gpu(wl, dev_inputs, slab_steps: int = 0, bank=None, workspace=None, flags: int = 0):
    """One sdm_write_read call; returns (readings, final bank, workspace); the bank in
    ``dev_inputs`` is not modified (a copy is advanced) unless ``bank`` is given."""
    b = dev_inputs["bank"].clone() if bank is None else bank
    shape = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R, b.dtype, slab_steps, flags)
    ws = sdm.alloc_workspace(shape, b.device) if workspace is None else workspace
    r = sdm.sdm_write_read(b, dev_inputs["write_slots"], dev_inputs["write_w"],
                           dev_inputs["log_decay"], dev_inputs["beta"], dev_inputs["v"],
                           dev_inputs["read_slots"], dev_inputs["read_w"], dev_inputs["valid"],
                           chunk_size=wl.C, slab_steps=slab_steps, workspace=ws, flags=flags)
    torch.cuda.synchronize()
    return r, b, ws


def f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def oracle_args(x, streams=None, S=None):
    if streams is None:
        return (x["bank"], x["ws"], x["k"], x["g"], x["beta"], x["v"], x["rs"], x["q"],
                x["valid"])
    lo, hi = streams
    return (x["bank"][lo * S:hi * S], x["ws"][lo:hi], x["k"][lo:hi], x["g"][lo:hi],
            x["beta"][lo:hi], x["v"][lo:hi], x["rs"][lo:hi], x["q"][lo:hi], x["valid"][lo:hi])


class Err:
    """Running max |gpu - ref| and max |ref| over pieces of one tensor."""

    def __init__(self):
        self.num = 0.0
        self.den = 0.0

    def add(self, gpu: np.ndarray, ref: np.ndarray):
        if ref.size:
            if not np.all(np.isfinite(gpu)):
                self.num = float("inf")          # a NaN or inf result is never within tolerance
            else:
                self.num = max(self.num, float(np.abs(gpu - ref).max()))
            self.den = max(self.den, float(np.abs(ref).max()))

    @property
    def value(self) -> float:
        return self.num / self.den if self.den > 0 else self.num


def _slice_inputs(inputs, wl, lo, hi):
    out = {k: inputs[k][lo:hi] for k in ("write_slots", "write_w", "log_decay", "beta", "v",
                                         "read_slots", "read_w", "valid")}
    out["bank"] = inputs["bank"][lo * wl.S:hi * wl.S]
    return out


def compare_with_oracle(wl, inputs, readings: torch.Tensor, bank: torch.Tensor,
                        streams_per_call: int = 4, nthreads: int = 4):
    """Errors (readings, bank) of a GPU result against the sequential oracle, computed a
    group of streams at a time (inputs converted per group) to bound host memory."""
    er, eb = Err(), Err()
    for lo in range(0, wl.P, streams_per_call):
        hi = min(wl.P, lo + streams_per_call)
        x = oracle.from_stored(_slice_inputs(inputs, wl, lo, hi), wl.dtype)
        o, B = oracle.sequential(*oracle_args(x), nthreads=nthreads)
        del x
        er.add(f64(readings[lo:hi]), o)
        del o
        eb.add(f64(bank[lo * wl.S:hi * wl.S]), B)
        del B
    return er.value, eb.value


def small_workload(P=3, T=100, C=16, S=64, D=64, W=4, R=3, dtype="f32", slots="zipf1.1",
                   ragged=True, seed=0) -> si.Workload:
    return si.Workload(f"small_p{P}_t{T}_c{C}_s{S}_d{D}_w{W}_r{R}_{dtype}_{slots}", P, T, C, S,
                       D, W, R, dtype, slots, ragged, seed)
