"""The host-buffer forward (sdm_write_read_host): inputs in host memory, readings written into
pinned host memory by the kernels, the bank on the device. It runs the same kernels as
sdm_write_read, so its results are bitwise those of the device call; one case is also held to
the oracle."""

import numpy as np
import pytest
import torch

import sdm_inputs as si
import sparse_addressed_delta_gb300 as sdm
from sdm_case import TOL, compare_with_oracle, small_workload, stored_tensor, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    sdm.library()


NAMES = ("write_slots", "write_w", "log_decay", "beta", "v", "read_slots", "read_w", "valid")


def host_inputs(inputs, wl):
    """Pinned host copies of the inputs (bank dtype for the weights and v)."""
    out = {}
    for k in NAMES:
        t = stored_tensor(inputs[k], wl.dtype, "cpu") if k in ("write_w", "v", "read_w") else \
            torch.from_numpy(np.ascontiguousarray(inputs[k]))
        out[k] = t.pin_memory()
    return out


def both_calls(wl, inputs, flags=0, slab_steps=0):
    dev = to_device(inputs, wl)
    host = host_inputs(inputs, wl)
    bank_d = dev["bank"].clone()
    r_d = sdm.sdm_write_read(bank_d, *(dev[k] for k in NAMES), chunk_size=wl.C,
                             slab_steps=slab_steps, flags=flags)
    bank_h = dev["bank"].clone()
    r_h = sdm.sdm_write_read_host(bank_h, *(host[k] for k in NAMES), chunk_size=wl.C,
                                  slab_steps=slab_steps, flags=flags)
    torch.cuda.synchronize()
    return r_d.cpu(), bank_d, r_h, bank_h


@pytest.mark.parametrize("flags", [0, sdm.FLAG_PER_STEP_KERNELS])
@pytest.mark.parametrize("dtype,C,W,ragged", [("bf16", 64, 16, True), ("f32", 16, 4, False),
                                              ("bf16", 48, 8, True)])
def test_host_call_matches_device_call(flags, dtype, C, W, ragged):
    wl = small_workload(P=3, T=5 * C + 7, C=C, S=700, D=128, W=W, R=W, dtype=dtype,
                        seed=C + W, ragged=ragged)
    r_d, b_d, r_h, b_h = both_calls(wl, si.generate(wl), flags=flags, slab_steps=2)
    assert torch.equal(r_d, r_h) and torch.equal(b_d, b_h)


def test_host_call_against_oracle():
    wl = small_workload(P=2, T=200, C=32, S=500, D=64, W=8, R=8, dtype="bf16", seed=11,
                        ragged=True)
    inputs = si.generate(wl)
    _, _, r_h, b_h = both_calls(wl, inputs)
    er, eb = compare_with_oracle(wl, inputs, r_h, b_h)
    assert er <= TOL[wl.dtype] and eb <= TOL[wl.dtype], (er, eb)


def test_host_call_bench_size_bitwise():
    """The bench workload (P=8, T=4096, C=64, bf16, W=R=16 Zipf) through both entry points."""
    wl = si.WORKLOADS[1]
    r_d, b_d, r_h, b_h = both_calls(wl, si.generate(wl))
    assert torch.equal(r_d, r_h) and torch.equal(b_d, b_h)


def test_host_call_in_cuda_graph():
    """Captured once (copies, the side-stream v copy and the kernels), replayed twice."""
    wl = small_workload(P=2, T=300, C=64, S=900, D=128, W=16, R=16, dtype="bf16", seed=5)
    inputs = si.generate(wl)
    dev = to_device(inputs, wl)
    host = host_inputs(inputs, wl)
    bank0 = dev["bank"]
    ref = dev["bank"].clone()
    r_ref = sdm.sdm_write_read(ref, *(dev[k] for k in NAMES), chunk_size=wl.C).cpu()
    bank = bank0.clone()
    shape = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R, bank.dtype)
    ws = torch.empty(sdm.host_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    readings = torch.empty((wl.P, wl.T, wl.D), dtype=bank.dtype, pin_memory=True)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):       # warm call outside the capture
        sdm.sdm_write_read_host(bank, *(host[k] for k in NAMES), chunk_size=wl.C,
                                readings=readings, workspace=ws, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sdm.sdm_write_read_host(bank, *(host[k] for k in NAMES), chunk_size=wl.C,
                                readings=readings, workspace=ws, stream=stream)
    for _ in range(2):
        bank.copy_(bank0)
        readings.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(readings, r_ref) and torch.equal(bank, ref)


def test_host_call_refuses_unmapped_readings():
    wl = small_workload(P=1, T=64, C=16, S=64, D=64, W=4, R=4, dtype="f32", seed=1)
    inputs = si.generate(wl)
    dev = to_device(inputs, wl)
    host = host_inputs(inputs, wl)
    bank = dev["bank"].clone()
    pageable = torch.empty((wl.P, wl.T, wl.D), dtype=torch.float32)
    with pytest.raises(sdm.SdmError):
        sdm.sdm_write_read_host(bank, *(host[k] for k in NAMES), chunk_size=wl.C,
                                readings=pageable)
    torch.cuda.synchronize()
    assert torch.equal(bank, dev["bank"])      # refused before any work


def test_host_call_pageable_inputs():
    """Inputs in ordinary (pageable) host memory take the per-array transfer path."""
    wl = small_workload(P=2, T=260, C=64, S=800, D=128, W=16, R=16, dtype="bf16", seed=8,
                        ragged=True)
    inputs = si.generate(wl)
    dev = to_device(inputs, wl)
    pinned = host_inputs(inputs, wl)
    pageable = {k: t.clone() for k, t in pinned.items()}
    assert not pageable["v"].is_pinned()
    ref = dev["bank"].clone()
    r_ref = sdm.sdm_write_read(ref, *(dev[k] for k in NAMES), chunk_size=wl.C).cpu()
    bank = dev["bank"].clone()
    r = sdm.sdm_write_read_host(bank, *(pageable[k] for k in NAMES), chunk_size=wl.C)
    torch.cuda.synchronize()
    assert torch.equal(r, r_ref) and torch.equal(bank, ref)
