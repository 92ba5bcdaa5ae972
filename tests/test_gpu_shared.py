"""One bank shared by all streams (SDM_FLAG_SHARED_BANK; the pages' num_memory_slots 0 with
shared_bank=True) on the GPU.

Stream p of a per-stream layout owns rows [p*S, (p+1)*S); here the same problem is laid out
in one [P*S, D] bank with stream p's slot s at row s*P + p (interleaved, disjoint slot sets).
That is a relabelling of the rows that keeps every chunk's sort order, so the shared-bank
call must give bitwise the per-stream results, rows permuted, on every entry point.
"""

import numpy as np
import pytest
import torch

import sdm_inputs as si
import sparse_addressed_delta_gb300 as sdm
from sdm_case import TOL, compare_with_oracle, small_workload, stored_tensor, to_device

pytestmark = pytest.mark.gpu

NAMES = ("write_slots", "write_w", "log_decay", "beta", "v", "read_slots", "read_w", "valid")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    sdm.library()


def shared_layout(wl, inputs):
    """The shared-bank inputs and the row map: shared row s*P + p = per-stream row p*S + s."""
    P, S = wl.P, wl.S
    p_idx = np.arange(P, dtype=np.int64)[:, None, None]
    out = dict(inputs)
    out["write_slots"] = (inputs["write_slots"].astype(np.int64) * P + p_idx).astype(np.int32)
    out["read_slots"] = (inputs["read_slots"].astype(np.int64) * P + p_idx).astype(np.int32)
    rows = (np.arange(S)[None, :] * P + np.arange(P)[:, None]).reshape(-1)   # [p*S + s] -> s*P + p
    bank = np.empty_like(inputs["bank"])
    bank[rows] = inputs["bank"]
    out["bank"] = bank
    return out, torch.from_numpy(rows).cuda()


def call(wl, dev, shared, flags=0):
    bank = dev["bank"].clone()
    r = sdm.sdm_write_read(bank, *(dev[k] for k in NAMES), chunk_size=wl.C, flags=flags,
                           slab_steps=2, shared_bank=shared)
    torch.cuda.synchronize()
    return r, bank


@pytest.mark.parametrize("flags", [0, sdm.FLAG_PER_STEP_KERNELS])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_shared_bank_forward_is_the_relabelled_per_stream_call(flags, dtype):
    wl = small_workload(P=3, T=85, C=16, S=40, D=64, W=5, R=4, dtype=dtype, seed=81)
    inputs = si.generate(wl)
    shared, rows = shared_layout(wl, inputs)
    r_p, b_p = call(wl, to_device(inputs, wl), False, flags)
    r_s, b_s = call(wl, to_device(shared, wl), True, flags)
    assert torch.equal(r_s, r_p)
    assert torch.equal(b_s[rows], b_p)
    er, eb = compare_with_oracle(wl, inputs, r_p, b_p)
    assert er <= TOL[dtype] and eb <= TOL[dtype], (er, eb)


def test_shared_bank_host_and_noalloc_calls():
    wl = small_workload(P=2, T=70, C=16, S=50, D=64, W=4, R=4, dtype="bf16", seed=82)
    shared, _ = shared_layout(wl, si.generate(wl))
    dev = to_device(shared, wl)
    r_d, b_d = call(wl, dev, True)
    host = {k: (stored_tensor(shared[k], wl.dtype, "cpu") if k in ("write_w", "v", "read_w")
                else torch.from_numpy(np.ascontiguousarray(shared[k]))).pin_memory()
            for k in NAMES}
    b_h = dev["bank"].clone()
    r_h = sdm.sdm_write_read_host(b_h, *(host[k] for k in NAMES), chunk_size=wl.C, slab_steps=2,
                                  shared_bank=True)
    b_n = dev["bank"].clone()
    r_n = torch.empty_like(r_d)
    sdm.sdm_write_read_noalloc(b_n, *(dev[k] for k in NAMES), chunk_size=wl.C, readings=r_n,
                               shared_bank=True)
    torch.cuda.synchronize()
    assert torch.equal(r_h.cuda(), r_d) and torch.equal(b_h, b_d)
    assert torch.equal(r_n, r_d) and torch.equal(b_n, b_d)


@pytest.mark.parametrize("flags", [0, sdm.FLAG_PER_STEP_KERNELS])
def test_shared_bank_backward(flags):
    """Every gradient bitwise as in the per-stream layout (the bank gradient's rows permuted),
    and the shared bank restored bitwise."""
    wl = small_workload(P=2, T=75, C=16, S=30, D=32, W=4, R=3, dtype="f32", seed=83)
    inputs = si.generate(wl)
    shared, rows = shared_layout(wl, inputs)
    rng = np.random.default_rng(84)
    gr = rng.standard_normal((wl.P, wl.T, wl.D))
    gr[np.arange(wl.T)[None, :] >= inputs["valid"][:, None]] = 0.0
    gr = stored_tensor(si.to_stored(gr, wl.dtype), wl.dtype, "cuda")
    outs = {}
    for name, inp, sh in (("per_stream", inputs, False), ("shared", shared, True)):
        dev = to_device(inp, wl)
        bank = dev["bank"].clone()
        args = tuple(dev[k] for k in NAMES)
        _, saved = sdm.sdm_write_read_save(bank, *args, chunk_size=wl.C, flags=flags,
                                           shared_bank=sh)
        out = sdm.sdm_write_read_backward(bank, *args, saved, gr, chunk_size=wl.C,
                                          shared_bank=sh)
        torch.cuda.synchronize()
        assert torch.equal(bank, dev["bank"]), name
        outs[name] = out
    assert torch.equal(outs["shared"]["grad_bank"][rows], outs["per_stream"]["grad_bank"])
    for k in ("grad_v", "grad_beta", "grad_write_w", "grad_log_decay", "grad_read_w"):
        assert torch.equal(outs["shared"][k], outs["per_stream"][k]), k
