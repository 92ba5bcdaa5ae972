"""GB300 (sm_103a) chunked sparse-delta-memory write/read.

A thin ctypes binding of ``libsdm.so`` (the C ABI in ``include/sdm.h``): it checks tensor
shapes, dtypes and devices, allocates the outputs and the workspace with PyTorch, and passes
raw device pointers and the current CUDA stream. Every step of the computation runs in the
library's CUDA kernels; there is no other implementation to fall back on, and a missing
library is an error.

Main entry point: :func:`sdm_write_read` (sparse-delta-memory 2.0.0, memory_ops.py
``sdm_write_read``, no-grad call) -> readings, with the bank advanced in place.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Dict, Optional

import torch

__all__ = ["FLAG_SNAPSHOT_BF16", "FLAG_SNAPSHOT_FP8", "FLAG_TOKEN_GATE", "FLAG_SHARED_BANK", "head_split",
           "head_merge", "bank_expand", "bank_sum", "sdm_write_read", "sdm_write_read_save", "sdm_write_read_backward",
           "sdm_write_read_noalloc", "noalloc_device_status", "profile_write_read", "workspace_bytes",
           "backward_workspace_bytes", "launch_count",
           "phase1_debug", "KERNEL_KINDS", "set_wait_limit", "product_key_topk",
           "product_key_topk_backward",
           "device_status", "SdmError", "Shape", "library", "library_path", "version"]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libsdm.so")

SDM_F32, SDM_BF16 = 0, 1
KERNEL_KINDS = ("phase1", "solve", "gather", "dualmm", "dw", "phase2")
FLAG_PER_STEP_KERNELS = 1
FLAG_SNAPSHOT_BF16 = 2
FLAG_TOKEN_GATE = 4
FLAG_SHARED_BANK = 8
FLAG_SNAPSHOT_FP8 = 16
SNAPSHOT_QUANT = {"none": 0, "bf16": FLAG_SNAPSHOT_BF16, "fp8": FLAG_SNAPSHOT_FP8}
_STATUS = {0: "SDM_OK", -1: "SDM_ERR_INVALID", -2: "SDM_ERR_UNSUPPORTED", -3: "SDM_ERR_CUDA",
           -4: "SDM_ERR_TIMEOUT", -5: "SDM_ERR_WORKSPACE", -6: "SDM_ERR_DEVICE"}


class SdmError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{_STATUS.get(code, code)}: {message}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int32), ("T", ctypes.c_int32), ("C", ctypes.c_int32),
                ("S", ctypes.c_int32), ("D", ctypes.c_int32), ("W", ctypes.c_int32),
                ("R", ctypes.c_int32), ("bank_dtype", ctypes.c_int32),
                ("slab_steps", ctypes.c_int32), ("flags", ctypes.c_int32)]


class _DeviceStatus(ctypes.Structure):
    _fields_ = [("code", ctypes.c_int32), ("first_bad_token", ctypes.c_int32),
                ("bad_slots", ctypes.c_int64), ("repeated_write_slots", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library() -> ctypes.CDLL:
    """The loaded libsdm.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise ImportError(
                    f"libsdm.so is not built ({library_path} is missing); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            lib = ctypes.CDLL(library_path)
            vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64
            sp = ctypes.POINTER(Shape)
            lib.sdm_workspace_bytes.argtypes = [sp]
            lib.sdm_workspace_bytes.restype = sz
            lib.sdm_launch_count.argtypes = [sp]
            lib.sdm_launch_count.restype = i64
            lib.sdm_write_read.argtypes = [sp] + [vp] * 10 + [vp, sz, vp]
            lib.sdm_write_read.restype = i32
            lib.sdm_saved_bytes.argtypes = [sp]
            lib.sdm_saved_bytes.restype = sz
            lib.sdm_backward_workspace_bytes.argtypes = [sp]
            lib.sdm_backward_workspace_bytes.restype = sz
            lib.sdm_write_read_save.argtypes = [sp] + [vp] * 10 + [vp, sz, vp, sz, vp]
            lib.sdm_write_read_save.restype = i32
            lib.sdm_write_read_backward.argtypes = ([sp] + [vp] * 9 + [vp, sz] + [vp] * 7
                                                    + [vp, sz, vp])
            lib.sdm_write_read_backward.restype = i32
            lib.sdm_host_workspace_bytes.argtypes = [sp]
            lib.sdm_host_workspace_bytes.restype = sz
            lib.sdm_write_read_host.argtypes = [sp] + [vp] * 10 + [vp, sz, vp]
            lib.sdm_write_read_host.restype = i32
            lib.sdm_write_read_noalloc.argtypes = [sp] + [vp] * 10 + [vp]
            lib.sdm_write_read_noalloc.restype = i32
            lib.sdm_noalloc_get_device_status.argtypes = [ctypes.POINTER(_DeviceStatus), vp]
            lib.sdm_noalloc_get_device_status.restype = i32
            lib.sdm_profile_write_read.argtypes = ([sp] + [vp] * 10 + [vp, sz]
                                                   + [ctypes.POINTER(ctypes.c_float),
                                                      ctypes.POINTER(ctypes.c_int32), vp])
            lib.sdm_profile_write_read.restype = i32
            lib.sdm_phase1_debug.argtypes = [sp] + [vp] * 7 + [vp] * 14 + [vp, sz, vp]
            lib.sdm_phase1_debug.restype = i32
            lib.sdm_get_device_status.argtypes = [vp, ctypes.POINTER(_DeviceStatus), vp]
            lib.sdm_get_device_status.restype = i32
            for name in ("sdm_head_split", "sdm_head_merge"):
                getattr(lib, name).argtypes = [vp, vp, i32, i32, i32, i32, i32, vp]
                getattr(lib, name).restype = i32
            for name in ("sdm_bank_expand", "sdm_bank_sum"):
                getattr(lib, name).argtypes = [vp, vp, i32, ctypes.c_longlong, i32, i32, vp]
                getattr(lib, name).restype = i32
            ll = ctypes.c_longlong
            lib.sdm_product_key_topk.argtypes = [vp, ll, ctypes.POINTER(ctypes.c_int), i32, i32,
                                                 i32, vp, vp, vp]
            lib.sdm_product_key_topk.restype = i32
            lib.sdm_product_key_topk_backward.argtypes = [vp, vp, ll, ctypes.POINTER(ctypes.c_int),
                                                          i32, i32, i32, vp, vp]
            lib.sdm_product_key_topk_backward.restype = i32
            lib.sdm_set_wait_limit.argtypes = [ctypes.c_longlong]
            lib.sdm_set_wait_limit.restype = ctypes.c_longlong
            lib.sdm_last_error.argtypes = []
            lib.sdm_last_error.restype = ctypes.c_char_p
            lib.sdm_version.argtypes = []
            lib.sdm_version.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def version() -> str:
    return library().sdm_version().decode()


def set_wait_limit(polls: int) -> int:
    """Testing aid: the number of polls after which a kernel's bounded wait for its own copies
    gives up, for calls queued from now on (process-wide; polls < 1 restores the default).
    Returns the previous limit."""
    return int(library().sdm_set_wait_limit(int(polls)))


def _check(rc: int) -> None:
    if rc != 0:
        raise SdmError(rc, library().sdm_last_error().decode())


def _dtype_code(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return SDM_F32
    if dtype == torch.bfloat16:
        return SDM_BF16
    raise TypeError(f"bank dtype must be float32 or bfloat16, got {dtype}")


def make_shape(P, T, C, S, D, W, R, dtype, slab_steps: int = 0, flags: int = 0) -> Shape:
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return Shape(P, T, C, S, D, W, R, code, slab_steps, flags)


def workspace_bytes(shape: Shape) -> int:
    n = library().sdm_workspace_bytes(ctypes.byref(shape))
    if n == 0:
        raise SdmError(-1, library().sdm_last_error().decode())
    return int(n)


def backward_workspace_bytes(shape: Shape) -> int:
    """Bytes of device workspace sdm_write_read_backward needs for ``shape``."""
    n = library().sdm_backward_workspace_bytes(ctypes.byref(shape))
    if n == 0:
        raise SdmError(-1, library().sdm_last_error().decode())
    return int(n)


def launch_count(shape: Shape) -> int:
    return int(library().sdm_launch_count(ctypes.byref(shape)))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _gate(log_decay: torch.Tensor, P: int, T: int, W: int):
    """(flag, shape) of the log-decays: one per write entry, [P, T, W]; or one per token,
    [P, T] (or [P, T, 1] with W > 1), which sets FLAG_TOKEN_GATE."""
    shp = tuple(log_decay.shape)
    if shp == (P, T) or (W > 1 and shp == (P, T, 1)):
        return FLAG_TOKEN_GATE, shp
    return 0, (P, T, W)


def _bank_rows(bank: torch.Tensor, P: int, shared_bank: bool):
    """(S, bank rows, flag): stream p owns rows [p*S, (p+1)*S) of a [P*S, D] bank, or with
    ``shared_bank`` all streams use the one [S, D] bank (their slot sets must be disjoint)."""
    if bank.dim() != 2 or (not shared_bank and bank.shape[0] % P):
        raise ValueError(f"bank must be [P*S, D] with P={P} (or [S, D] with shared_bank), "
                         f"got {tuple(bank.shape)}")
    if shared_bank:
        return bank.shape[0], bank.shape[0], FLAG_SHARED_BANK
    return bank.shape[0] // P, bank.shape[0], 0


def _need(t: torch.Tensor, name: str, shape, dtype, device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the bank on {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def alloc_workspace(shape: Shape, device) -> torch.Tensor:
    """A workspace tensor (uint8, 256-byte aligned by the caching allocator)."""
    return torch.empty(workspace_bytes(shape), dtype=torch.uint8, device=device)


def _stream_ptr(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def sdm_write_read(bank: torch.Tensor, write_slots: torch.Tensor, write_w: torch.Tensor,
                   log_decay: torch.Tensor, beta: torch.Tensor, v: torch.Tensor,
                   read_slots: torch.Tensor, read_w: torch.Tensor,
                   valid_tokens: Optional[torch.Tensor] = None, *, chunk_size: int,
                   slab_steps: int = 0, workspace: Optional[torch.Tensor] = None,
                   readings: Optional[torch.Tensor] = None, stream=None,
                   flags: int = 0, shared_bank: bool = False) -> torch.Tensor:
    """Chunked SDM write/read over P streams; returns readings [P, T, D] and advances
    ``bank`` ([P*S, D], float32 or bfloat16, stream p owning rows [p*S, (p+1)*S)) in place.

    write_slots [P, T, W] int32; write_w [P, T, W] bank dtype; log_decay [P, T, W] float32;
    beta [P, T] float32; v [P, T, D] bank dtype; read_slots [P, T, R] int32; read_w
    [P, T, R] bank dtype; valid_tokens [P] int32 (None: all T valid).
    """
    if write_slots.dim() != 3:
        raise ValueError("write_slots must be [P, T, W]")
    P, T, W = write_slots.shape
    R = read_slots.shape[-1]
    S, rows, sflag = _bank_rows(bank, P, shared_bank)
    flags |= sflag
    D = bank.shape[1]
    dev, dt = bank.device, bank.dtype
    if dev.type != "cuda":
        raise ValueError("the bank must be a CUDA tensor")
    _need(bank, "bank", (rows, D), dt, dev)
    _need(write_slots, "write_slots", (P, T, W), torch.int32, dev)
    _need(write_w, "write_w", (P, T, W), dt, dev)
    gflag, gshape = _gate(log_decay, P, T, W)
    flags |= gflag
    _need(log_decay, "log_decay", gshape, torch.float32, dev)
    _need(beta, "beta", (P, T), torch.float32, dev)
    _need(v, "v", (P, T, D), dt, dev)
    _need(read_slots, "read_slots", (P, T, R), torch.int32, dev)
    _need(read_w, "read_w", (P, T, R), dt, dev)
    if valid_tokens is not None:
        _need(valid_tokens, "valid_tokens", (P,), torch.int32, dev)
    shape = make_shape(P, T, chunk_size, S, D, W, R, dt, slab_steps, flags)
    if readings is None:
        readings = torch.empty((P, T, D), dtype=dt, device=dev)
    else:
        _need(readings, "readings", (P, T, D), dt, dev)
    if workspace is None:
        workspace = alloc_workspace(shape, dev)
    with torch.cuda.device(dev):
        rc = library().sdm_write_read(
            ctypes.byref(shape), _ptr(bank), _ptr(write_slots), _ptr(write_w), _ptr(log_decay),
            _ptr(beta), _ptr(v), _ptr(read_slots), _ptr(read_w), _ptr(valid_tokens),
            _ptr(readings), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return readings


def host_workspace_bytes(shape: Shape) -> int:
    n = library().sdm_host_workspace_bytes(ctypes.byref(shape))
    if n == 0:
        raise SdmError(-1, library().sdm_last_error().decode())
    return n


def sdm_write_read_host(bank: torch.Tensor, write_slots: torch.Tensor, write_w: torch.Tensor,
                        log_decay: torch.Tensor, beta: torch.Tensor, v: torch.Tensor,
                        read_slots: torch.Tensor, read_w: torch.Tensor,
                        valid_tokens: Optional[torch.Tensor] = None, *, chunk_size: int,
                        readings: Optional[torch.Tensor] = None, slab_steps: int = 0,
                        workspace: Optional[torch.Tensor] = None, stream=None,
                        flags: int = 0, shared_bank: bool = False) -> torch.Tensor:
    """sdm_write_read with the inputs in host memory and the readings written to pinned host
    memory ([P, T, D], bank dtype); the bank stays on its GPU. Same arguments and layouts as
    ``sdm_write_read``; pinned inputs make the copies asynchronous."""
    if write_slots.dim() != 3:
        raise ValueError("write_slots must be [P, T, W]")
    P, T, W = write_slots.shape
    R = read_slots.shape[-1]
    S, rows, sflag = _bank_rows(bank, P, shared_bank)
    flags |= sflag
    if bank.device.type != "cuda":
        raise ValueError("the bank must be a CUDA tensor")
    D = bank.shape[1]
    dev, dt, cpu = bank.device, bank.dtype, torch.device("cpu")
    _need(bank, "bank", (rows, D), dt, dev)
    _need(write_slots, "write_slots", (P, T, W), torch.int32, cpu)
    _need(write_w, "write_w", (P, T, W), dt, cpu)
    gflag, gshape = _gate(log_decay, P, T, W)
    flags |= gflag
    _need(log_decay, "log_decay", gshape, torch.float32, cpu)
    _need(beta, "beta", (P, T), torch.float32, cpu)
    _need(v, "v", (P, T, D), dt, cpu)
    _need(read_slots, "read_slots", (P, T, R), torch.int32, cpu)
    _need(read_w, "read_w", (P, T, R), dt, cpu)
    if valid_tokens is not None:
        _need(valid_tokens, "valid_tokens", (P,), torch.int32, cpu)
    shape = make_shape(P, T, chunk_size, S, D, W, R, dt, slab_steps, flags)
    if readings is None:
        readings = torch.empty((P, T, D), dtype=dt, pin_memory=True)
    else:
        _need(readings, "readings", (P, T, D), dt, cpu)
    if workspace is None:
        workspace = torch.empty(host_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = library().sdm_write_read_host(
            ctypes.byref(shape), _ptr(bank), _ptr(write_slots), _ptr(write_w), _ptr(log_decay),
            _ptr(beta), _ptr(v), _ptr(read_slots), _ptr(read_w), _ptr(valid_tokens),
            _ptr(readings), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return readings


def _shape_of(bank, write_slots, read_slots, chunk_size, slab_steps=0, flags=0,
              shared_bank=False):
    P, T, W = write_slots.shape
    R = read_slots.shape[-1]
    S, _, sflag = _bank_rows(bank, P, shared_bank)
    D = bank.shape[1]
    return (make_shape(P, T, chunk_size, S, D, W, R, bank.dtype, slab_steps, flags | sflag),
            (P, T, S, D, W, R))


def saved_bytes(shape: Shape) -> int:
    n = library().sdm_saved_bytes(ctypes.byref(shape))
    if n == 0:
        raise SdmError(-1, library().sdm_last_error().decode())
    return int(n)


def _snapshot_flag(snapshot_quant: str) -> int:
    if snapshot_quant not in SNAPSHOT_QUANT:
        raise ValueError(f"snapshot_quant must be one of {tuple(SNAPSHOT_QUANT)}, "
                         f"got {snapshot_quant!r}")
    return SNAPSHOT_QUANT[snapshot_quant]


def sdm_write_read_save(bank, write_slots, write_w, log_decay, beta, v, read_slots, read_w,
                        valid_tokens=None, *, chunk_size: int, slab_steps: int = 0,
                        workspace=None, readings=None, saved=None, stream=None, flags: int = 0,
                        snapshot_quant: str = "none", shared_bank: bool = False):
    """The saving forward: sdm_write_read plus the snapshot the backward needs.
    ``snapshot_quant`` "bf16" stores the snapshot of a float32 bank in bfloat16 (half the
    bytes), "fp8" in float8_e4m3fn (one byte an element, saturating at +-448); the backward
    then restores the written rows to their rounded values.
    Returns (readings, saved)."""
    flags |= _snapshot_flag(snapshot_quant)
    P, T, W = write_slots.shape
    gflag, gshape = _gate(log_decay, P, T, W)
    shape, (P, T, S, D, W, R) = _shape_of(bank, write_slots, read_slots, chunk_size,
                                          slab_steps, flags | gflag, shared_bank)
    dev, dt = bank.device, bank.dtype
    rows = S if shared_bank else P * S
    for t, name, shp, typ in ((bank, "bank", (rows, D), dt), (write_slots, "write_slots", (P, T, W), torch.int32),
                              (write_w, "write_w", (P, T, W), dt), (log_decay, "log_decay", gshape, torch.float32),
                              (beta, "beta", (P, T), torch.float32), (v, "v", (P, T, D), dt),
                              (read_slots, "read_slots", (P, T, R), torch.int32), (read_w, "read_w", (P, T, R), dt)):
        _need(t, name, shp, typ, dev)
    if readings is None:
        readings = torch.empty((P, T, D), dtype=dt, device=dev)
    if workspace is None:
        workspace = alloc_workspace(shape, dev)
    if saved is None:
        saved = torch.empty(saved_bytes(shape), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = library().sdm_write_read_save(
            ctypes.byref(shape), _ptr(bank), _ptr(write_slots), _ptr(write_w), _ptr(log_decay),
            _ptr(beta), _ptr(v), _ptr(read_slots), _ptr(read_w), _ptr(valid_tokens),
            _ptr(readings), _ptr(saved), saved.numel(), _ptr(workspace), workspace.numel(),
            _stream_ptr(stream))
    _check(rc)
    return readings, saved


def sdm_write_read_backward(bank, write_slots, write_w, log_decay, beta, v, read_slots, read_w,
                            valid_tokens, saved, grad_readings, *, chunk_size: int,
                            grad_bank=None, slab_steps: int = 0, workspace=None, stream=None,
                            snapshot_quant: str = "none", shared_bank: bool = False):
    """The backward after sdm_write_read_save (with the same ``snapshot_quant``): restores
    ``bank`` to its initial state (with "bf16", the rows the call wrote to their bfloat16
    rounding) and returns a dict of float32 gradients (grad_bank, grad_v, grad_beta,
    grad_write_w, grad_log_decay, grad_read_w). ``grad_bank`` (optional, [P*S, D] float32) is
    the loss gradient with respect to the final bank; it is updated in place to the gradient
    with respect to the initial bank."""
    P, T, W = write_slots.shape
    gflag, gshape = _gate(log_decay, P, T, W)
    shape, (P, T, S, D, W, R) = _shape_of(bank, write_slots, read_slots, chunk_size, slab_steps,
                                          _snapshot_flag(snapshot_quant) | gflag, shared_bank)
    dev, dt = bank.device, bank.dtype
    _need(grad_readings, "grad_readings", (P, T, D), dt, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    rows = S if shared_bank else P * S
    if grad_bank is None:
        grad_bank = torch.zeros((rows, D), **f32)
    _need(grad_bank, "grad_bank", (rows, D), torch.float32, dev)
    out = {"grad_bank": grad_bank, "grad_v": torch.empty((P, T, D), **f32),
           "grad_beta": torch.empty((P, T), **f32), "grad_write_w": torch.empty((P, T, W), **f32),
           "grad_log_decay": torch.empty(gshape, **f32),
           "grad_read_w": torch.empty((P, T, R), **f32)}
    if workspace is None:
        workspace = torch.empty(backward_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = library().sdm_write_read_backward(
            ctypes.byref(shape), _ptr(bank), _ptr(write_slots), _ptr(write_w), _ptr(log_decay),
            _ptr(beta), _ptr(v), _ptr(read_slots), _ptr(read_w), _ptr(valid_tokens),
            _ptr(saved), saved.numel(), _ptr(grad_readings), _ptr(out["grad_bank"]),
            _ptr(out["grad_v"]), _ptr(out["grad_beta"]), _ptr(out["grad_write_w"]),
            _ptr(out["grad_log_decay"]), _ptr(out["grad_read_w"]), _ptr(workspace),
            workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return out


def sdm_write_read_noalloc(bank: torch.Tensor, write_slots: torch.Tensor,
                           write_w: torch.Tensor, log_decay: torch.Tensor, beta: torch.Tensor,
                           v: torch.Tensor, read_slots: torch.Tensor, read_w: torch.Tensor,
                           valid_tokens: Optional[torch.Tensor] = None, *, chunk_size: int,
                           readings: torch.Tensor, slab_steps: int = 0, stream=None,
                           flags: int = 0, shared_bank: bool = False) -> torch.Tensor:
    """sdm_write_read for callers that cannot allocate device memory: the library's static
    device scratch (16 MiB per GPU) replaces the workspace, and the caller passes the
    readings buffer, so the call allocates nothing. Calls overlapping on the GPU race on the
    shared scratch; the first call on a device should come before any CUDA graph capture."""
    P, T, W = write_slots.shape
    R = read_slots.shape[-1]
    S, rows, sflag = _bank_rows(bank, P, shared_bank)
    flags |= sflag
    D = bank.shape[1]
    dev, dt = bank.device, bank.dtype
    gflag, gshape = _gate(log_decay, P, T, W)
    flags |= gflag
    for t, name, shp, typ in ((bank, "bank", (rows, D), dt), (write_slots, "write_slots", (P, T, W), torch.int32),
                              (write_w, "write_w", (P, T, W), dt), (log_decay, "log_decay", gshape, torch.float32),
                              (beta, "beta", (P, T), torch.float32), (v, "v", (P, T, D), dt),
                              (read_slots, "read_slots", (P, T, R), torch.int32), (read_w, "read_w", (P, T, R), dt),
                              (readings, "readings", (P, T, D), dt)):
        _need(t, name, shp, typ, dev)
    if valid_tokens is not None:
        _need(valid_tokens, "valid_tokens", (P,), torch.int32, dev)
    shape = make_shape(P, T, chunk_size, S, D, W, R, dt, slab_steps, flags)
    with torch.cuda.device(dev):
        rc = library().sdm_write_read_noalloc(
            ctypes.byref(shape), _ptr(bank), _ptr(write_slots), _ptr(write_w), _ptr(log_decay),
            _ptr(beta), _ptr(v), _ptr(read_slots), _ptr(read_w), _ptr(valid_tokens),
            _ptr(readings), _stream_ptr(stream))
    _check(rc)
    return readings


def profile_write_read(bank, write_slots, write_w, log_decay, beta, v, read_slots, read_w,
                       valid_tokens=None, *, chunk_size: int, slab_steps: int = 0,
                       workspace=None, readings=None, stream=None, flags: int = 0,
                       shared_bank: bool = False):
    """One sdm_write_read call with CUDA events around every kernel launch (synchronizes).
    Returns (readings, {family: (total_ms, launches)}) for the families in KERNEL_KINDS."""
    P, T, W = write_slots.shape
    R = read_slots.shape[-1]
    S, _, sflag = _bank_rows(bank, P, shared_bank)
    flags |= sflag
    D = bank.shape[1]
    dev, dt = bank.device, bank.dtype
    shape = make_shape(P, T, chunk_size, S, D, W, R, dt, slab_steps,
                       flags | _gate(log_decay, P, T, W)[0])
    if readings is None:
        readings = torch.empty((P, T, D), dtype=dt, device=dev)
    if workspace is None:
        workspace = alloc_workspace(shape, dev)
    for t, name in ((write_slots, "write_slots"), (read_slots, "read_slots")):
        _need(t, name, t.shape, torch.int32, dev)
    ms = (ctypes.c_float * len(KERNEL_KINDS))()
    cnt = (ctypes.c_int32 * len(KERNEL_KINDS))()
    with torch.cuda.device(dev):
        rc = library().sdm_profile_write_read(
            ctypes.byref(shape), _ptr(bank), _ptr(write_slots), _ptr(write_w), _ptr(log_decay),
            _ptr(beta), _ptr(v), _ptr(read_slots), _ptr(read_w), _ptr(valid_tokens),
            _ptr(readings), _ptr(workspace), workspace.numel(), ms, cnt, _stream_ptr(stream))
    _check(rc)
    return readings, {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(KERNEL_KINDS)}


def phase1_debug(write_slots, write_w, log_decay, beta, read_slots, read_w, valid_tokens=None,
                 *, S: int, D: int, chunk_size: int, slab_steps: int = 0,
                 stream=None) -> Dict[str, torch.Tensor]:
    """Phase 1 and the solve of every chunk (time-major chunk n = ti*P + p), as tensors:
    perm, group_start, owner [N, C*W]; ngroups [N]; lw, gw, dw [N, C*W]; lr, qw [N, C*R];
    A, QK, X, QX [N, C, C]; dense_groups [N] (the groups whose Gram pair sums were taken in
    the dense factor form)."""
    P, T, W = write_slots.shape
    R = read_slots.shape[-1]
    dev, dt = write_w.device, write_w.dtype
    C = chunk_size
    shape = make_shape(P, T, C, S, D, W, R, dt, slab_steps, _gate(log_decay, P, T, W)[0])
    N = P * (-(-T // C))
    f32 = dict(dtype=torch.float32, device=dev)
    out = {
        "perm": torch.empty((N, C * W), dtype=torch.int32, device=dev),
        "group_start": torch.empty((N, C * W), dtype=torch.uint8, device=dev),
        "owner": torch.empty((N, C * W), dtype=torch.uint8, device=dev),
        "ngroups": torch.empty((N,), dtype=torch.int32, device=dev),
        "lw": torch.empty((N, C * W), **f32), "gw": torch.empty((N, C * W), **f32),
        "dw": torch.empty((N, C * W), **f32), "lr": torch.empty((N, C * R), **f32),
        "qw": torch.empty((N, C * R), **f32), "A": torch.empty((N, C, C), **f32),
        "QK": torch.empty((N, C, C), **f32), "X": torch.empty((N, C, C), **f32),
        "QX": torch.empty((N, C, C), **f32),
        "dense_groups": torch.empty((N,), dtype=torch.int32, device=dev),
    }
    ws = alloc_workspace(shape, dev)
    order = ["perm", "group_start", "owner", "ngroups", "lw", "gw", "dw", "lr", "qw", "A", "QK",
             "X", "QX", "dense_groups"]
    with torch.cuda.device(dev):
        rc = library().sdm_phase1_debug(
            ctypes.byref(shape), _ptr(write_slots), _ptr(write_w), _ptr(log_decay), _ptr(beta),
            _ptr(read_slots), _ptr(read_w), _ptr(valid_tokens), *[_ptr(out[k]) for k in order],
            _ptr(ws), ws.numel(), _stream_ptr(stream))
    _check(rc)
    out["workspace"] = ws
    return out


def device_status(workspace: torch.Tensor, stream=None) -> Dict[str, int]:
    """The device status block of the last call that used ``workspace`` (synchronizes)."""
    st = _DeviceStatus()
    with torch.cuda.device(workspace.device):
        _check(library().sdm_get_device_status(_ptr(workspace), ctypes.byref(st),
                                               _stream_ptr(stream)))
    return {"code": st.code, "first_bad_token": st.first_bad_token, "bad_slots": st.bad_slots,
            "repeated_write_slots": st.repeated_write_slots}


def noalloc_device_status(device=None, stream=None) -> Dict[str, int]:
    """The device status block of the last ``sdm_write_read_noalloc`` call on ``device``
    (default: the current one); synchronizes."""
    st = _DeviceStatus()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        _check(library().sdm_noalloc_get_device_status(ctypes.byref(st), _stream_ptr(stream)))
    return {"code": st.code, "first_bad_token": st.first_bad_token, "bad_slots": st.bad_slots,
            "repeated_write_slots": st.repeated_write_slots}


# ------------------------------------------------------------------------------------------
# product-key exact top-k (product_key_topk.py)
# ------------------------------------------------------------------------------------------

def _factors_arg(factors):
    f = [int(x) for x in factors]
    return (ctypes.c_int * len(f))(*f), len(f)


def product_key_topk(raw: torch.Tensor, factors, k: int, stream=None):
    """Exact top-k over product-key slots: raw [..., sum(factors)] float32 or bfloat16 on a GPU
    -> (val [..., kk] in raw's dtype, lin [..., kk] int64), kk = min(k, prod(factors)), the kept
    slots sorted by lin. The selection rule is the pages' (include/sdm.h)."""
    if raw.device.type != "cuda" or not raw.is_contiguous():
        raise ValueError("raw must be a contiguous CUDA tensor")
    fa, F = _factors_arg(factors)
    if raw.shape[-1] != sum(int(x) for x in factors):
        raise ValueError("raw's last dimension must be sum(factors)")
    prod = 1
    for x in factors:
        prod *= int(x)
    kk = min(int(k), prod)
    rows = raw.numel() // raw.shape[-1]
    val = torch.empty(raw.shape[:-1] + (kk,), dtype=raw.dtype, device=raw.device)
    lin = torch.empty(raw.shape[:-1] + (kk,), dtype=torch.int64, device=raw.device)
    with torch.cuda.device(raw.device):
        _check(library().sdm_product_key_topk(_ptr(raw), rows, fa, F, int(k),
                                              _dtype_code(raw.dtype), _ptr(val), _ptr(lin),
                                              _stream_ptr(stream)))
    return val, lin


def product_key_topk_backward(lin: torch.Tensor, grad_val: torch.Tensor, factors, k: int,
                              stream=None) -> torch.Tensor:
    """d(loss)/d(raw) [..., sum(factors)] float32 from the forward's lin and grad_val."""
    fa, F = _factors_arg(factors)
    ld = sum(int(x) for x in factors)
    rows = lin.numel() // lin.shape[-1] if lin.dim() else 0
    grad_raw = torch.empty(lin.shape[:-1] + (ld,), dtype=torch.float32, device=lin.device)
    with torch.cuda.device(lin.device):
        _check(library().sdm_product_key_topk_backward(
            _ptr(lin), _ptr(grad_val.contiguous()), rows, fa, F, int(k),
            _dtype_code(grad_val.dtype), _ptr(grad_raw), _stream_ptr(stream)))
    return grad_raw


# ------------------------------------------------------------------------------------------
# layer I/O (memory_ops.py "Layer I/O: head split / merge and the per-batch bank expand")
# ------------------------------------------------------------------------------------------

def _io_tensor(x: torch.Tensor, name: str, ndim: int) -> None:
    if x.device.type != "cuda" or not x.is_contiguous() or x.dim() != ndim:
        raise ValueError(f"{name} must be a contiguous {ndim}-d CUDA tensor")
    _dtype_code(x.dtype)


def head_split(x: torch.Tensor, H: int, stream=None) -> torch.Tensor:
    """rearrange(x, 'b t (h k) -> (b h) t k', h=H) as a row copy: [B, T, H*CD] -> [B*H, T, CD]."""
    _io_tensor(x, "x", 3)
    B, T, HC = x.shape
    if HC % H:
        raise ValueError(f"the last dimension {HC} is not a multiple of H={H}")
    out = torch.empty((B * H, T, HC // H), dtype=x.dtype, device=x.device)
    with torch.cuda.device(x.device):
        _check(library().sdm_head_split(_ptr(x), _ptr(out), B, T, H, HC // H,
                                        _dtype_code(x.dtype), _stream_ptr(stream)))
    return out


def head_merge(x: torch.Tensor, H: int, stream=None) -> torch.Tensor:
    """rearrange(x, '(b h) t d -> b t (h d)', h=H): [B*H, T, CD] -> [B, T, H*CD]."""
    _io_tensor(x, "x", 3)
    BH, T, CD = x.shape
    if BH % H:
        raise ValueError(f"the first dimension {BH} is not a multiple of H={H}")
    out = torch.empty((BH // H, T, H * CD), dtype=x.dtype, device=x.device)
    with torch.cuda.device(x.device):
        _check(library().sdm_head_merge(_ptr(x), _ptr(out), BH // H, T, H, CD,
                                        _dtype_code(x.dtype), _stream_ptr(stream)))
    return out


def bank_expand(param: torch.Tensor, B: int, stream=None) -> torch.Tensor:
    """The per-batch bank: [S, D] -> [B, S, D], every copy the parameter bank."""
    _io_tensor(param, "param", 2)
    S, D = param.shape
    out = torch.empty((B, S, D), dtype=param.dtype, device=param.device)
    with torch.cuda.device(param.device):
        _check(library().sdm_bank_expand(_ptr(param), _ptr(out), B, S, D,
                                         _dtype_code(param.dtype), _stream_ptr(stream)))
    return out


def bank_sum(x: torch.Tensor, stream=None) -> torch.Tensor:
    """The expand's adjoint: [B, S, D] -> [S, D], summed over the batch in float32 in batch
    order and rounded once to the dtype."""
    _io_tensor(x, "x", 3)
    B, S, D = x.shape
    out = torch.empty((S, D), dtype=x.dtype, device=x.device)
    with torch.cuda.device(x.device):
        _check(library().sdm_bank_sum(_ptr(x), _ptr(out), B, S, D, _dtype_code(x.dtype),
                                      _stream_ptr(stream)))
    return out
