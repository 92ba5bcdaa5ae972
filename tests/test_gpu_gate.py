"""One log-decay per token (SDM_FLAG_TOKEN_GATE; the pages' g of width 1) on the GPU.

A per-token gate is the per-write form with the gate repeated over the token's W writes: the
gated call must give bitwise the results of the per-write call on the repeated gates (Phase 1
reads the same values), for every entry point; its log-decay gradient is the sum of the
per-write gradients, held to the oracle's.
"""

import numpy as np
import pytest
import torch

import oracle
import sdm_inputs as si
import sparse_addressed_delta_gb300 as sdm
from sdm_case import TOL, Err, compare_with_oracle, f64, small_workload, stored_tensor, to_device

pytestmark = pytest.mark.gpu

NAMES = ("write_slots", "write_w", "log_decay", "beta", "v", "read_slots", "read_w", "valid")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    sdm.library()


def gated_inputs(wl):
    """(inputs with a [P, T] gate, the same inputs with it repeated to [P, T, W])."""
    inputs = si.generate(wl)
    gate = np.ascontiguousarray(inputs["log_decay"][..., 0])
    per_write = dict(inputs)
    per_write["log_decay"] = np.ascontiguousarray(np.repeat(gate[..., None], wl.W, axis=2))
    gated = dict(inputs)
    gated["log_decay"] = gate
    return gated, per_write


def call(wl, dev, flags=0):
    bank = dev["bank"].clone()
    r = sdm.sdm_write_read(bank, *(dev[k] for k in NAMES), chunk_size=wl.C, flags=flags,
                           slab_steps=2)
    torch.cuda.synchronize()
    return r, bank


@pytest.mark.parametrize("flags", [0, sdm.FLAG_PER_STEP_KERNELS])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gate_forward_is_the_repeated_gate(flags, dtype):
    wl = small_workload(P=3, T=90, C=16, S=60, D=64, W=5, R=4, dtype=dtype, seed=71)
    gated, per_write = gated_inputs(wl)
    r_g, b_g = call(wl, to_device(gated, wl), flags)
    r_w, b_w = call(wl, to_device(per_write, wl), flags)
    assert torch.equal(r_g, r_w) and torch.equal(b_g, b_w)
    er, eb = compare_with_oracle(wl, per_write, r_g, b_g)
    assert er <= TOL[dtype] and eb <= TOL[dtype], (er, eb)


def test_gate_host_and_noalloc_calls():
    wl = small_workload(P=2, T=70, C=16, S=50, D=64, W=4, R=4, dtype="bf16", seed=72)
    gated, _ = gated_inputs(wl)
    dev = to_device(gated, wl)
    r_d, b_d = call(wl, dev)
    host = {k: (stored_tensor(gated[k], wl.dtype, "cpu") if k in ("write_w", "v", "read_w")
                else torch.from_numpy(np.ascontiguousarray(gated[k]))).pin_memory()
            for k in NAMES}
    b_h = dev["bank"].clone()
    r_h = sdm.sdm_write_read_host(b_h, *(host[k] for k in NAMES), chunk_size=wl.C, slab_steps=2)
    b_n = dev["bank"].clone()
    r_n = torch.empty_like(r_d)
    sdm.sdm_write_read_noalloc(b_n, *(dev[k] for k in NAMES), chunk_size=wl.C, readings=r_n)
    torch.cuda.synchronize()
    assert torch.equal(r_h.cuda(), r_d) and torch.equal(b_h, b_d)
    assert torch.equal(r_n, r_d) and torch.equal(b_n, b_d)


@pytest.mark.parametrize("flags", [0, sdm.FLAG_PER_STEP_KERNELS])
def test_gate_backward(flags):
    """Every gradient but the log-decay one bitwise as with the repeated gate; the gate's
    gradient [P, T] within 1e-4 of the oracle's per-write gradients summed over the writes;
    the bank restored bitwise."""
    wl = small_workload(P=2, T=75, C=16, S=40, D=32, W=4, R=3, dtype="f32", seed=73)
    gated, per_write = gated_inputs(wl)
    rng = np.random.default_rng(74)
    gr = rng.standard_normal((wl.P, wl.T, wl.D))
    gr[np.arange(wl.T)[None, :] >= gated["valid"][:, None]] = 0.0
    gr = si.to_stored(gr, wl.dtype)
    outs = {}
    for name, inp in (("gated", gated), ("per_write", per_write)):
        dev = to_device(inp, wl)
        bank = dev["bank"].clone()
        args = tuple(dev[k] for k in NAMES)
        _, saved = sdm.sdm_write_read_save(bank, *args, chunk_size=wl.C, flags=flags)
        out = sdm.sdm_write_read_backward(bank, *args, saved, stored_tensor(gr, wl.dtype, "cuda"),
                                          chunk_size=wl.C)
        torch.cuda.synchronize()
        assert torch.equal(bank, dev["bank"]), name
        outs[name] = out
    assert tuple(outs["gated"]["grad_log_decay"].shape) == (wl.P, wl.T)
    for k in ("grad_bank", "grad_v", "grad_beta", "grad_write_w", "grad_read_w"):
        assert torch.equal(outs["gated"][k], outs["per_write"][k]), k
    x = oracle.from_stored(per_write, wl.dtype)
    ref = oracle.backward(x["bank"], x["ws"], x["k"], x["g"], x["beta"], x["v"], x["rs"], x["q"],
                          x["valid"], si.stored_to_f64(gr, wl.dtype))
    e = Err()
    e.add(f64(outs["gated"]["grad_log_decay"]), ref["grad_log_decay"].sum(axis=2))
    assert e.value <= 1e-4, e.value
