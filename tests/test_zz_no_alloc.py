"""The allocation-free entry point, sdm_write_read_noalloc, against sdm_write_read.

It exists for callers that own all device memory themselves (an engine or plugin host with
its own pool, a fixed-footprint service) and so cannot call cudaMalloc: its scratch is a
static 16 MiB device array inside the library instead of a caller workspace. This file runs
last (pytest collects it after the other test files) and also passes on its own.

The results do not depend on how many steps a slab holds, so the no-alloc call must give the
workspace call's readings and final bank bit for bit, also when it has to cut the call into
more slabs than the workspace call does.
"""

import ctypes

import pytest
import torch

import sdm_inputs as si
import sparse_addressed_delta_gb300 as sdm
from sdm_case import run_gpu, small_workload, to_device

pytestmark = pytest.mark.gpu

SCRATCH = 16 << 20          # SDM_NOALLOC_SCRATCH_BYTES

CASES = [
    small_workload(P=4, T=700, C=64, S=4096, D=128, W=16, R=16, dtype="bf16", slots="zipf1.1",
                   ragged=True, seed=41),
    small_workload(P=2, T=300, C=32, S=512, D=64, W=8, R=4, dtype="f32", slots="uniform",
                   ragged=False, seed=42),
    # all 8 steps need about 34 MiB of workspace, one step about 5 MiB: the no-alloc call
    # runs 3 steps per slab where the workspace call runs all 8 in one
    small_workload(P=4, T=1024, C=128, S=8192, D=128, W=64, R=64, dtype="bf16",
                   slots="zipf1.1", ragged=True, seed=43),
]


def _shape(wl, slab_steps=0):
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    return sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R, dt, slab_steps)


def _args(dev):
    return (dev["write_slots"], dev["write_w"], dev["log_decay"], dev["beta"], dev["v"],
            dev["read_slots"], dev["read_w"], dev["valid"])


@pytest.mark.parametrize("wl", CASES, ids=["bf16", "f32", "bf16_three_slabs"])
def test_noalloc_matches_workspace_entry_point(wl):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    if wl.C == 128:   # the case must need more than one slab inside the static scratch
        assert sdm.workspace_bytes(_shape(wl)) > SCRATCH >= sdm.workspace_bytes(_shape(wl, 1))
    dev = to_device(si.generate(wl), wl)
    bank_ref = dev["bank"].clone()
    bank_new = dev["bank"].clone()
    readings = torch.empty((wl.P, wl.T, wl.D), dtype=bank_new.dtype, device="cuda")
    for call in range(2):          # two calls in a row, each advancing its bank
        r_ref, _, _ = run_gpu(wl, dev, bank=bank_ref)
        if call == 1:
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
        sdm.sdm_write_read_noalloc(bank_new, *_args(dev), chunk_size=wl.C, readings=readings)
        torch.cuda.synchronize()
        if call == 1:   # no device memory was reserved by the second call
            assert torch.cuda.mem_get_info()[0] == free_before
        assert torch.equal(readings, r_ref), call
        assert torch.equal(bank_new, bank_ref), call
        st = sdm.noalloc_device_status()
        assert st["code"] == 0 and st["bad_slots"] == 0, st


def test_noalloc_explicit_slab_steps():
    """An explicit slab size that fits the scratch runs (and matches); one that does not is
    refused before any work."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    wl = CASES[2]
    fits = max(n for n in range(1, wl.Nt + 1) if sdm.workspace_bytes(_shape(wl, n)) <= SCRATCH)
    assert fits < wl.Nt
    dev = to_device(si.generate(wl), wl)
    r_ref, b_ref, _ = run_gpu(wl, dev)
    bank = dev["bank"].clone()
    readings = torch.empty((wl.P, wl.T, wl.D), dtype=bank.dtype, device="cuda")
    sdm.sdm_write_read_noalloc(bank, *_args(dev), chunk_size=wl.C, readings=readings,
                               slab_steps=fits)
    torch.cuda.synchronize()
    assert torch.equal(readings, r_ref) and torch.equal(bank, b_ref)
    before = bank.clone()
    with pytest.raises(sdm.SdmError) as ei:
        sdm.sdm_write_read_noalloc(bank, *_args(dev), chunk_size=wl.C, readings=readings,
                                   slab_steps=fits + 1)
    assert ei.value.code == -5 and "static scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.equal(bank, before)          # nothing was queued


def test_noalloc_device_status_reports_bad_slots():
    """A slot outside [0, S) is dropped and reported in the static scratch's status block."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    wl = small_workload(P=2, T=40, C=16, S=64, D=64, W=4, R=4, ragged=False, seed=44)
    inputs = si.generate(wl)
    inputs["write_slots"][1, 5, 2] = 1 << 30
    dev = to_device(inputs, wl)
    bank = dev["bank"].clone()
    readings = torch.empty((wl.P, wl.T, wl.D), dtype=bank.dtype, device="cuda")
    sdm.sdm_write_read_noalloc(bank, *_args(dev), chunk_size=wl.C, readings=readings)
    st = sdm.noalloc_device_status()
    assert st["code"] == -6 and st["bad_slots"] == 1 and st["first_bad_token"] == wl.T + 5, st
    _, _, ws = run_gpu(wl, dev)
    assert sdm.device_status(ws) == st        # the workspace call reports the same


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
