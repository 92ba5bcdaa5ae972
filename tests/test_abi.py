"""The C ABI library without a GPU: it loads, exports every function include/sdm.h declares,
and sizes/refuses shapes on the host (no compute call needs a device here)."""

import ctypes
import os
import re

import pytest

import sparse_addressed_delta_gb300 as sdm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "sdm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sdm_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = sdm.library()
    names = declared_functions()
    assert "sdm_write_read" in names and len(names) >= 6
    for name in names:
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_string():
    assert "sm_103a" in sdm.version()


def test_workspace_bytes_host_only():
    s = sdm.make_shape(8, 4096, 64, 65536, 128, 16, 16, sdm.SDM_BF16)
    n = sdm.workspace_bytes(s)
    assert n > 0 and n % 256 == 0
    # the slab is bounded: more tokens do not grow the workspace past the slab budget
    big = sdm.make_shape(4, 1 << 17, 256, 1 << 20, 256, 256, 256, sdm.SDM_BF16)
    huge = sdm.make_shape(4, 1 << 19, 256, 1 << 20, 256, 256, 256, sdm.SDM_BF16)
    assert sdm.workspace_bytes(huge) == sdm.workspace_bytes(big)
    # explicit slabs: fewer steps held, less workspace
    s1 = sdm.make_shape(8, 4096, 64, 65536, 128, 16, 16, sdm.SDM_BF16, slab_steps=4)
    assert sdm.workspace_bytes(s1) < n


def test_launch_count():
    s = sdm.make_shape(8, 4096, 64, 65536, 128, 16, 16, sdm.SDM_BF16)
    assert sdm.launch_count(s) == 3                      # Phase 1, solve, fused Phase 2
    s = sdm.make_shape(8, 4096, 64, 65536, 128, 16, 16, sdm.SDM_BF16,
                       flags=sdm.FLAG_PER_STEP_KERNELS)
    assert sdm.launch_count(s) == 2 + 3 * 64
    nt, slabs = 7, 3
    s = sdm.make_shape(1, 100, 16, 64, 64, 4, 4, sdm.SDM_F32, slab_steps=3)
    assert sdm.launch_count(s) == 3 * slabs
    s = sdm.make_shape(1, 100, 16, 64, 64, 4, 4, sdm.SDM_F32, slab_steps=3,
                       flags=sdm.FLAG_PER_STEP_KERNELS)
    assert sdm.launch_count(s) == 2 * slabs + 3 * nt
    # chunks whose metadata does not fit on chip twice take the per-step kernels; chunks whose
    # Phase-1 scratch does not fit on chip add Phase 1's row and dense-Gram kernels
    s = sdm.make_shape(16, 4096, 128, 131072, 128, 64, 64, sdm.SDM_F32, slab_steps=32)
    assert sdm.launch_count(s) == 4 + 3 * 32


@pytest.mark.parametrize("kw,code", [
    (dict(C=8), -1), (dict(C=300), -1), (dict(W=0), -1), (dict(R=257), -1), (dict(P=0), -1),
    (dict(T=0), -1), (dict(S=0), -1), (dict(D=96), -2), (dict(dtype=7), -1), (dict(flags=32), -1),
    (dict(P=1 << 16, T=1 << 16), -1)])
def test_refusals(kw, code):
    base = dict(P=2, T=64, C=16, S=128, D=64, W=4, R=4, dtype=sdm.SDM_F32, flags=0)
    base.update(kw)
    s = sdm.Shape(base["P"], base["T"], base["C"], base["S"], base["D"], base["W"], base["R"],
                  base["dtype"], 0, base["flags"])
    assert sdm.library().sdm_workspace_bytes(ctypes.byref(s)) == 0
    msg = sdm.library().sdm_last_error().decode()
    assert msg
    with pytest.raises(sdm.SdmError) as e:
        sdm.workspace_bytes(s)


def test_write_read_refuses_before_any_work():
    """A null pointer or a short workspace is refused on the host, before any launch."""
    lib = sdm.library()
    s = sdm.make_shape(1, 32, 16, 64, 64, 4, 4, sdm.SDM_F32)
    rc = lib.sdm_write_read(ctypes.byref(s), None, None, None, None, None, None, None, None,
                            None, None, None, 0, None)
    assert rc == -1
    fake = ctypes.c_void_p(1 << 40)
    rc = lib.sdm_write_read(ctypes.byref(s), fake, fake, fake, fake, fake, fake, fake, fake,
                            None, fake, fake, 16, None)
    assert rc == -5 and "workspace" in lib.sdm_last_error().decode()


def test_host_workspace_holds_the_inputs():
    s = sdm.make_shape(8, 4096, 64, 65536, 128, 16, 16, sdm.SDM_BF16)
    per_token = 16 * 4 + 16 * 2 + 16 * 4 + 4 + 128 * 2 + 16 * 4 + 16 * 2
    assert sdm.host_workspace_bytes(s) >= sdm.workspace_bytes(s) + 8 * 4096 * per_token
    bad = sdm.make_shape(8, 4096, 64, 65536, 100, 16, 16, sdm.SDM_BF16)
    with pytest.raises(sdm.SdmError):
        sdm.host_workspace_bytes(bad)


def test_bf16_snapshot_halves_saved_bytes():
    """SDM_FLAG_SNAPSHOT_BF16 stores a float32 bank's snapshot in bfloat16: half the bytes;
    a bfloat16 bank's snapshot is bfloat16 already. Unknown flag bits are refused."""
    for dt, ratio in ((sdm.SDM_F32, 2), (sdm.SDM_BF16, 1)):
        plain = sdm.saved_bytes(sdm.make_shape(3, 100, 16, 50, 64, 3, 4, dt))
        half = sdm.saved_bytes(sdm.make_shape(3, 100, 16, 50, 64, 3, 4, dt,
                                              flags=sdm.FLAG_SNAPSHOT_BF16))
        assert plain == 7 * 3 * 16 * 3 * 64 * (4 if dt == sdm.SDM_F32 else 2)
        assert plain == ratio * half
    with pytest.raises(sdm.SdmError):
        sdm.saved_bytes(sdm.make_shape(3, 100, 16, 50, 64, 3, 4, sdm.SDM_F32, flags=32))


def test_token_gate_flag():
    """SDM_FLAG_TOKEN_GATE (one log-decay per token) is accepted everywhere; the host-buffer
    call stages P*T gates instead of P*T*W."""
    plain = sdm.make_shape(4, 512, 64, 1000, 128, 16, 16, sdm.SDM_BF16)
    gated = sdm.make_shape(4, 512, 64, 1000, 128, 16, 16, sdm.SDM_BF16, flags=sdm.FLAG_TOKEN_GATE)
    assert sdm.workspace_bytes(gated) == sdm.workspace_bytes(plain)
    diff = sdm.host_workspace_bytes(plain) - sdm.host_workspace_bytes(gated)
    assert 4 * 4 * 512 * 15 - 256 <= diff <= 4 * 4 * 512 * 15 + 256


def test_binding_infers_flags_from_shapes():
    """Host logic of the binding (no GPU): the per-token gate from log_decay's shape, the
    rows of a per-stream or shared bank, the snapshot flag."""
    import torch

    P, T, W = 3, 10, 4
    assert sdm._gate(torch.zeros(P, T, W), P, T, W) == (0, (P, T, W))
    assert sdm._gate(torch.zeros(P, T), P, T, W) == (sdm.FLAG_TOKEN_GATE, (P, T))
    assert sdm._gate(torch.zeros(P, T, 1), P, T, W) == (sdm.FLAG_TOKEN_GATE, (P, T, 1))
    assert sdm._gate(torch.zeros(P, T, 1), P, T, 1) == (0, (P, T, 1))   # W = 1: per write
    bank = torch.zeros(P * 7, 8)
    assert sdm._bank_rows(bank, P, False) == (7, P * 7, 0)
    assert sdm._bank_rows(bank, P, True) == (P * 7, P * 7, sdm.FLAG_SHARED_BANK)
    with pytest.raises(ValueError):
        sdm._bank_rows(torch.zeros(P * 7 + 1, 8), P, False)
    assert sdm._snapshot_flag("none") == 0
    assert sdm._snapshot_flag("bf16") == sdm.FLAG_SNAPSHOT_BF16
    assert sdm._snapshot_flag("fp8") == sdm.FLAG_SNAPSHOT_FP8
    with pytest.raises(ValueError):
        sdm._snapshot_flag("int4")                # not built: the pages give no scale scheme
    flags = {sdm.FLAG_PER_STEP_KERNELS, sdm.FLAG_SNAPSHOT_BF16, sdm.FLAG_TOKEN_GATE,
             sdm.FLAG_SHARED_BANK, sdm.FLAG_SNAPSHOT_FP8}
    assert len(flags) == 5 and all(f & (f - 1) == 0 for f in flags)     # distinct bits


def test_binding_flags_match_the_header():
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "sdm.h")).read()
    defs = dict((k, int(v)) for k, v in re.findall(r"#define (SDM_FLAG_\w+) (\d+)", hdr))
    assert defs == {"SDM_FLAG_PER_STEP_KERNELS": sdm.FLAG_PER_STEP_KERNELS,
                    "SDM_FLAG_SNAPSHOT_BF16": sdm.FLAG_SNAPSHOT_BF16,
                    "SDM_FLAG_TOKEN_GATE": sdm.FLAG_TOKEN_GATE,
                    "SDM_FLAG_SHARED_BANK": sdm.FLAG_SHARED_BANK,
                    "SDM_FLAG_SNAPSHOT_FP8": sdm.FLAG_SNAPSHOT_FP8}


def test_wait_limit_setter_round_trips():
    """sdm_set_wait_limit returns the previous limit; polls < 1 restores the default."""
    lib = sdm.library()
    default = lib.sdm_set_wait_limit(0)
    assert default == 1 << 22
    assert lib.sdm_set_wait_limit(5) == default
    assert lib.sdm_set_wait_limit(-3) == 5
    assert lib.sdm_set_wait_limit(0) == default


def test_product_key_refusals_and_empty_call():
    """Bad widths or k are refused before any work; zero rows queue nothing."""
    lib = sdm.library()
    f = (ctypes.c_int * 2)(4, 5000)
    assert lib.sdm_product_key_topk(None, 1, f, 2, 8, 0, None, None, None) == -2
    f = (ctypes.c_int * 1)(4)
    assert lib.sdm_product_key_topk(None, 1, f, 1, 300, 0, None, None, None) == -1
    f5 = (ctypes.c_int * 5)(2, 2, 2, 2, 2)
    assert lib.sdm_product_key_topk(None, 1, f5, 5, 8, 0, None, None, None) == -1
    assert lib.sdm_product_key_topk(None, 0, f, 1, 8, 0, None, None, None) == 0


def test_fp8_snapshot_sizes_and_refusals():
    """An fp8 snapshot holds one byte an element (a quarter of a float32 bank's snapshot, half
    of a bfloat16 bank's); the two reduced snapshots exclude each other."""
    import torch
    for dt, ratio in ((torch.float32, 4), (torch.bfloat16, 2)):
        full = sdm.make_shape(2, 64, 16, 100, 64, 4, 3, dt)
        fp8 = sdm.make_shape(2, 64, 16, 100, 64, 4, 3, dt, flags=sdm.FLAG_SNAPSHOT_FP8)
        assert sdm.saved_bytes(full) == ratio * sdm.saved_bytes(fp8)
    both = sdm.make_shape(2, 64, 16, 100, 64, 4, 3, torch.float32,
                          flags=sdm.FLAG_SNAPSHOT_FP8 | sdm.FLAG_SNAPSHOT_BF16)
    assert sdm.library().sdm_workspace_bytes(ctypes.byref(both)) == 0


def test_phase1_launches_by_chunk_class():
    """Phase 1 per slab: one kernel with the chunk's scratch on chip; the sort and row kernels
    over global scratch; and the dense-Gram kernel besides from C = 128 on (shapes chosen so
    that one slab holds every step, per-step Phase 2: 3 launches per step)."""
    for (C, W, p1) in ((16, 4, 1), (64, 32, 2), (128, 64, 3), (256, 32, 3)):
        T = 2 * C
        s = sdm.make_shape(1, T, C, 4096, 64, W, W, sdm.SDM_F32, flags=sdm.FLAG_PER_STEP_KERNELS)
        assert sdm.launch_count(s) == p1 + 1 + 3 * 2, (C, W)


def test_dense_gram_workspace_is_bounded():
    """The dense Gram factors add three C x C float arrays per chunk for C >= 128, and the
    workspace still does not grow with T."""
    a = sdm.make_shape(2, 1 << 16, 128, 1 << 16, 64, 64, 64, sdm.SDM_BF16)
    b = sdm.make_shape(2, 1 << 18, 128, 1 << 16, 64, 64, 64, sdm.SDM_BF16)
    assert sdm.workspace_bytes(a) == sdm.workspace_bytes(b)
