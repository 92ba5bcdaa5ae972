"""The allocation-free entry point, sdm_write_read_noalloc, against sdm_write_read.

It exists for callers that own all device memory themselves (an engine or plugin host with
its own pool, a fixed-footprint service) and so cannot call cudaMalloc: its scratch is a
static 16 MiB device array inside the library instead of a caller workspace. This file runs
last (pytest collects it after the other test files) and also passes on its own.
"""

import ctypes

import pytest
import torch

import sdm_inputs as si
import sparse_addressed_delta_gb300 as sdm
from sdm_case import TOL, run_gpu, small_workload, to_device

pytestmark = pytest.mark.gpu


def _rel(a: torch.Tensor, b: torch.Tensor) -> float:
    a, b = a.double(), b.double()
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-300))


@pytest.mark.parametrize("wl", [
    small_workload(P=4, T=700, C=64, S=4096, D=128, W=16, R=16, dtype="bf16", slots="zipf1.1",
                   ragged=True, seed=41),
    small_workload(P=2, T=300, C=32, S=512, D=64, W=8, R=4, dtype="f32", slots="uniform",
                   ragged=False, seed=42),
], ids=["bf16", "f32"])
def test_noalloc_matches_workspace_entry_point(wl):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    dev = to_device(si.generate(wl), wl)
    bank_ref = dev["bank"].clone()
    bank_new = dev["bank"].clone()
    readings = torch.empty((wl.P, wl.T, wl.D), dtype=bank_new.dtype, device="cuda")
    args = (dev["write_slots"], dev["write_w"], dev["log_decay"], dev["beta"], dev["v"],
            dev["read_slots"], dev["read_w"], dev["valid"])
    tol = TOL[wl.dtype]
    for call in range(2):          # two calls in a row, each advancing its bank
        r_ref, _, _ = run_gpu(wl, dev, bank=bank_ref)
        if call == 1:
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
        sdm.sdm_write_read_noalloc(bank_new, *args, chunk_size=wl.C, readings=readings)
        torch.cuda.synchronize()
        if call == 1:   # no device memory was reserved by the second call
            assert torch.cuda.mem_get_info()[0] == free_before
        assert _rel(readings, r_ref) <= tol, call
        assert _rel(bank_new, bank_ref) <= tol, call


def test_noalloc_refuses_shapes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib = sdm.library()
    # chunks of P=4, C=256, W=R=256, D=256 need about 26 MB of scratch even one step at a time
    s = sdm.make_shape(4, 16384, 256, 1 << 20, 256, 256, 256, sdm.SDM_BF16)
    fake = ctypes.c_void_p(256)
    rc = lib.sdm_write_read_noalloc(ctypes.byref(s), fake, fake, fake, fake, fake, fake, fake,
                                    fake, None, fake, None)
    assert rc == -5
    assert "static scratch" in lib.sdm_last_error().decode()
