"""Parity of the CUDA backward (through the C ABI) with the oracle's reverse-mode token loop.

Per gradient tensor the error is max |gpu - oracle| / max |oracle|, bounded by 1e-4 for
float32 banks (the forward's float32 tolerance, applied to every gradient); the bank must be
restored to its initial state bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import sdm_inputs as si
import sparse_addressed_delta_gb300 as sdm
from sdm_case import Err, f64, small_workload, stored_tensor, to_device

pytestmark = pytest.mark.gpu

GRADS = ("grad_bank", "grad_v", "grad_beta", "grad_write_w", "grad_log_decay", "grad_read_w")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    sdm.library()


def gpu_backward(wl, inputs, grad_readings, grad_final=None, slab_steps=0, flags=0,
                 snapshot_quant="none"):
    dev = to_device(inputs, wl)
    bank = dev["bank"].clone()
    args = (dev["write_slots"], dev["write_w"], dev["log_decay"], dev["beta"], dev["v"],
            dev["read_slots"], dev["read_w"], dev["valid"])
    readings, saved = sdm.sdm_write_read_save(bank, *args, chunk_size=wl.C,
                                              slab_steps=slab_steps, flags=flags,
                                              snapshot_quant=snapshot_quant)
    gr = stored_tensor(grad_readings, wl.dtype, "cuda")
    gb = None if grad_final is None else torch.from_numpy(
        np.ascontiguousarray(grad_final, dtype=np.float32)).cuda()
    out = sdm.sdm_write_read_backward(bank, *args, saved, gr, chunk_size=wl.C, grad_bank=gb,
                                      slab_steps=slab_steps, snapshot_quant=snapshot_quant)
    torch.cuda.synchronize()
    return readings, bank, dev["bank"], out


def oracle_backward(wl, inputs, grad_readings, grad_final=None, streams_per_call=None,
                    nthreads=4):
    """Oracle gradients, a group of streams at a time; returns {name: fp64 array}."""
    P, S = wl.P, wl.S
    spc = streams_per_call or P
    res = {k: [] for k in GRADS}
    for lo in range(0, P, spc):
        hi = min(P, lo + spc)
        sub = {k: inputs[k][lo:hi] for k in ("write_slots", "write_w", "log_decay", "beta", "v",
                                             "read_slots", "read_w", "valid")}
        sub["bank"] = inputs["bank"][lo * S:hi * S]
        x = oracle.from_stored(sub, wl.dtype)
        g = si.stored_to_f64(grad_readings[lo:hi], wl.dtype)
        gf = None if grad_final is None else grad_final[lo * S:hi * S]
        r = oracle.backward(x["bank"], x["ws"], x["k"], x["g"], x["beta"], x["v"], x["rs"],
                            x["q"], x["valid"], g, nthreads=nthreads, grad_final_bank=gf)
        for k in GRADS:
            res[k].append(r[k])
    return {k: np.concatenate(v, axis=0) for k, v in res.items()}


def errors(out, ref):
    errs = {}
    for k in GRADS:
        e = Err()
        e.add(f64(out[k]), ref[k])
        errs[k] = e.value
    return errs


def make_case(wl, with_final=False, seed=100):
    inputs = si.generate(wl)
    rng = np.random.default_rng(seed)
    gr = rng.standard_normal((wl.P, wl.T, wl.D))
    pad = np.arange(wl.T)[None, :] >= inputs["valid"][:, None]
    gr[pad] = 0.0
    grad_readings = si.to_stored(gr, wl.dtype)
    grad_final = rng.standard_normal((wl.P * wl.S, wl.D)).astype(np.float32) if with_final else None
    return inputs, grad_readings, grad_final


def check(wl, with_final=False, tol=1e-4, slab_steps=0, flags=0):
    inputs, gr, gf = make_case(wl, with_final)
    _, bank, bank0, out = gpu_backward(wl, inputs, gr, gf, slab_steps, flags)
    assert torch.equal(bank, bank0), "bank not restored exactly"
    ref = oracle_backward(wl, inputs, gr, gf)
    errs = errors(out, ref)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, (wl.name, errs)
    return errs


@pytest.mark.parametrize("with_final", [False, True])
def test_backward_dense_collisions(with_final):
    check(small_workload(P=2, T=70, C=16, S=20, D=32, W=4, R=3, ragged=True, seed=31),
          with_final=with_final)


@pytest.mark.parametrize("C,D,W,R,S", [(16, 64, 1, 1, 8), (32, 64, 8, 5, 64), (64, 128, 16, 16, 500),
                                       (48, 32, 6, 7, 40), (128, 128, 64, 64, 4096)])
def test_backward_shapes(C, D, W, R, S):
    check(small_workload(P=3, T=2 * C + 9, C=C, S=S, D=D, W=W, R=R, ragged=True,
                         seed=C + W))


def test_backward_uniform_slots_fp32():
    check(small_workload(P=2, T=200, C=64, S=10000, D=128, W=32, R=32, slots="uniform",
                         ragged=False, seed=33))


@pytest.mark.parametrize("flags", [0, sdm.FLAG_PER_STEP_KERNELS])
def test_backward_slabs_and_paths(flags):
    """The snapshot written by either Phase-2 path, and slabs of one step."""
    check(small_workload(P=2, T=100, C=16, S=30, D=64, W=4, R=4, seed=34), slab_steps=2,
          flags=flags)


def test_backward_deterministic():
    wl = small_workload(P=2, T=130, C=32, S=50, D=64, W=8, R=8, seed=35)
    inputs, gr, gf = make_case(wl, True)
    _, _, _, o1 = gpu_backward(wl, inputs, gr, gf)
    _, _, _, o2 = gpu_backward(wl, inputs, gr, gf)
    for k in GRADS:
        assert torch.equal(o1[k], o2[k]), k


@pytest.mark.parametrize("seed", [36, 37])
def test_backward_bf16_bank(seed):
    """bfloat16 bank: every gradient within the bf16 forward tolerance (2e-2) of the oracle's
    unrounded reverse mode, the bank restored bit for bit."""
    errs = check(small_workload(P=2, T=100, C=32, S=60, D=64, W=8, R=8, dtype="bf16",
                                seed=seed), tol=2e-2)
    print(errs)


def test_backward_full_size_workload3():
    """P=16, T=4096, C=128, S=131072 x 128 fp32, W=R=64 uniform: every gradient within
    1e-4 of the oracle and the bank restored exactly."""
    wl = si.WORKLOADS[3]
    inputs = si.generate(wl)
    gr = inputs["grad_readings"]
    _, bank, bank0, out = gpu_backward(wl, inputs, gr)
    assert torch.equal(bank, bank0), "bank not restored exactly"
    ref = oracle_backward(wl, inputs, gr, streams_per_call=8, nthreads=8)
    errs = errors(out, ref)
    print(f"{wl.name}: " + ", ".join(f"{k} {v:.2e}" for k, v in errs.items()))
    assert all(v <= 1e-4 for v in errs.values()), errs


def test_backward_workspace_poison():
    """The backward reads no workspace byte it has not written: NaN-filled and zero-filled
    workspaces give the same gradients, bit for bit."""
    wl = small_workload(P=2, T=75, C=32, S=40, D=64, W=8, R=8, ragged=True, seed=37)
    inputs, gr, gf = make_case(wl, True)
    shape = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R, torch.float32)
    n = sdm.backward_workspace_bytes(shape)
    results = []
    for fill in (0x00, 0xFF):
        dev = to_device(inputs, wl)
        bank = dev["bank"].clone()
        args = (dev["write_slots"], dev["write_w"], dev["log_decay"], dev["beta"], dev["v"],
                dev["read_slots"], dev["read_w"], dev["valid"])
        _, saved = sdm.sdm_write_read_save(bank, *args, chunk_size=wl.C)
        ws = torch.full((n,), fill, dtype=torch.uint8, device="cuda")
        out = sdm.sdm_write_read_backward(
            bank, *args, saved, stored_tensor(gr, wl.dtype, "cuda"), chunk_size=wl.C,
            grad_bank=torch.from_numpy(gf).cuda(), workspace=ws)
        torch.cuda.synchronize()
        results.append(out)
    for k in GRADS:
        assert torch.isfinite(results[1][k]).all(), k
        assert torch.equal(results[0][k], results[1][k]), k


# ---------------------------------------------------------------------------------------
# bfloat16 snapshot of a float32 bank (SDM_FLAG_SNAPSHOT_BF16; memory_ops.py snapshot_quant)
# ---------------------------------------------------------------------------------------

def bf16_rows(x: np.ndarray) -> np.ndarray:
    """bfloat16 rounding (nearest even) of float32 rows, by torch's conversion."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).bfloat16().float().numpy()


def written_rows(inputs, S):
    P = inputs["write_slots"].shape[0]
    w = np.zeros(P * S, bool)
    for p in range(P):
        for t in range(int(inputs["valid"][p])):
            w[p * S + inputs["write_slots"][p, t]] = True
    return w


def separated_case(P, T, C, S, D, W, R, seed):
    """Float32 inputs in which chunk c writes only slots [cK, (c+1)K) and reads slots from its
    own range up: no chunk touches a row that an earlier chunk wrote, so every snapshot row is
    an initial bank row (the same float32 value on both sides) and the bfloat16 rounding of it
    is the same decision for the GPU and the oracle."""
    Nt = T // C
    K = S // (Nt + 1)
    rng = np.random.default_rng(seed)
    ws = np.zeros((P, T, W), np.int32)
    rs = np.zeros((P, T, R), np.int32)
    for p in range(P):
        for t in range(T):
            c = t // C
            ws[p, t] = c * K + rng.choice(K, W, replace=False)
            rs[p, t] = rng.integers(c * K, S, R)
    k = rng.standard_normal((P, T, W))
    q = rng.standard_normal((P, T, R))
    f = lambda a: np.ascontiguousarray(a, np.float32)  # noqa: E731
    inputs = {"bank": f(rng.standard_normal((P * S, D)) * 0.02), "write_slots": ws,
              "write_w": f(np.exp(k) / np.exp(k).sum(-1, keepdims=True)),
              "log_decay": f(-0.1 * np.log1p(np.exp(rng.standard_normal((P, T, W))))),
              "beta": f(1 / (1 + np.exp(-rng.standard_normal((P, T))))),
              "v": f(rng.standard_normal((P, T, D))), "read_slots": rs,
              "read_w": f(np.exp(q) / np.exp(q).sum(-1, keepdims=True)),
              "valid": np.array([T] + [T - 9] * (P - 1), np.int32)}
    wl = si.Workload(f"separated_p{P}_t{T}_c{C}_s{S}_d{D}_w{W}_r{R}", P, T, C, S, D, W, R,
                     "f32", "uniform", True, seed)
    gr = si.to_stored(rng.standard_normal((P, T, D)), "f32")
    gr[1:, T - 9:] = 0.0
    return wl, inputs, gr


def oracle_snapshot(wl, inputs, gr):
    x = oracle.from_stored(inputs, wl.dtype)
    return oracle.backward_snapshot(x["bank"], x["ws"], x["k"], x["g"], x["beta"], x["v"],
                                    x["rs"], x["q"], x["valid"],
                                    si.stored_to_f64(gr, wl.dtype), chunk_size=wl.C,
                                    snapshot="bf16")


@pytest.mark.parametrize("flags", [0, sdm.FLAG_PER_STEP_KERNELS])
def test_bf16_snapshot_matches_the_oracle(flags):
    """Gradients within 1e-4 of the oracle's reverse pass from a bfloat16 snapshot, the
    restored bank bit for bit: bf16(initial) on the written rows, initial elsewhere; and
    the gradients do move away from the exact ones (the rounding is applied)."""
    wl, inputs, gr = separated_case(P=3, T=64, C=16, S=100, D=64, W=4, R=3, seed=61)
    _, bank, bank0, out = gpu_backward(wl, inputs, gr, flags=flags, snapshot_quant="bf16")
    ref = oracle_snapshot(wl, inputs, gr)
    w = written_rows(inputs, wl.S)
    expect = inputs["bank"].copy()
    expect[w] = bf16_rows(inputs["bank"][w])
    assert np.array_equal(bank.cpu().numpy(), expect)
    assert np.array_equal(ref["restored_bank"].astype(np.float32), expect)
    errs = errors(out, ref)
    assert all(v <= 1e-4 for v in errs.values()), errs
    x = oracle.from_stored(inputs, wl.dtype)
    exact = oracle.backward(x["bank"], x["ws"], x["k"], x["g"], x["beta"], x["v"], x["rs"],
                            x["q"], x["valid"], si.stored_to_f64(gr, wl.dtype))
    assert errors(out, exact)["grad_write_w"] > 1e-6


@pytest.mark.parametrize("flags", [0, sdm.FLAG_PER_STEP_KERNELS])
def test_bf16_snapshot_general_slots(flags):
    """Zipf slots rewritten across chunks, ragged tokens, slabs: the restored bank is
    bf16(initial) on every written row, bit for bit. The gradients are held to the oracle's
    bfloat16-snapshot pass within 1e-2 only: an intermediate row that sits at a bfloat16
    rounding boundary can round one way from the GPU's float32 value and the other from the
    oracle's fp64 value."""
    wl = small_workload(P=2, T=90, C=16, S=30, D=64, W=4, R=3, dtype="f32", ragged=True,
                        seed=62)
    inputs, gr, _ = make_case(wl)
    _, bank, _, out = gpu_backward(wl, inputs, gr, slab_steps=2, flags=flags,
                                   snapshot_quant="bf16")
    w = written_rows(inputs, wl.S)
    expect = inputs["bank"].copy()
    expect[w] = bf16_rows(inputs["bank"][w])
    assert np.array_equal(bank.cpu().numpy(), expect)
    ref = oracle_snapshot(wl, inputs, gr)
    errs = errors(out, ref)
    assert all(v <= 1e-2 for v in errs.values()), errs


def test_bf16_snapshot_is_deterministic_and_halves_the_snapshot():
    wl, inputs, gr = separated_case(P=2, T=48, C=16, S=64, D=32, W=3, R=2, seed=63)
    res = [gpu_backward(wl, inputs, gr, snapshot_quant="bf16")[3] for _ in range(2)]
    for k in GRADS:
        assert torch.equal(res[0][k], res[1][k]), k
    shape = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R, torch.float32)
    half = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R, torch.float32,
                          flags=sdm.FLAG_SNAPSHOT_BF16)
    assert sdm.saved_bytes(shape) == 2 * sdm.saved_bytes(half)


# ---------------------------------------------------------------------------------------
# float8_e4m3fn snapshot (SDM_FLAG_SNAPSHOT_FP8; memory_ops.py snapshot_quant "fp8")
# ---------------------------------------------------------------------------------------

def fp8_rows(x: np.ndarray) -> np.ndarray:
    """float8_e4m3fn rounding (nearest even, saturating at +-448) of float32 rows, by torch's
    conversion of the clamped values."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).clamp(-448, 448)
    return t.to(torch.float8_e4m3fn).float().numpy()


def oracle_snapshot_mode(wl, inputs, gr, mode):
    x = oracle.from_stored(inputs, wl.dtype)
    return oracle.backward_snapshot(x["bank"], x["ws"], x["k"], x["g"], x["beta"], x["v"],
                                    x["rs"], x["q"], x["valid"],
                                    si.stored_to_f64(gr, wl.dtype), chunk_size=wl.C,
                                    snapshot=mode)


@pytest.mark.parametrize("flags", [0, sdm.FLAG_PER_STEP_KERNELS])
@pytest.mark.parametrize("bank_dtype", ["f32", "bf16"])
def test_fp8_snapshot_matches_the_oracle(flags, bank_dtype):
    """Gradients within the bank dtype's tolerance of the oracle's reverse pass from an fp8
    snapshot; the restored bank bit for bit: fp8(initial) on the written rows, initial
    elsewhere (no chunk touches a row an earlier chunk wrote, so both sides round the same
    initial values)."""
    wl, inputs, gr = separated_case(P=3, T=64, C=16, S=100, D=64, W=4, R=3, seed=71)
    if bank_dtype == "bf16":
        wl = wl.replace(dtype="bf16")
        for k in ("bank", "write_w", "v", "read_w"):
            inputs[k] = si.to_stored(inputs[k].astype(np.float64), "bf16")
        gr = si.to_stored(si.stored_to_f64(gr, "f32"), "bf16")
    _, bank, _, out = gpu_backward(wl, inputs, gr, flags=flags, snapshot_quant="fp8")
    ref = oracle_snapshot_mode(wl, inputs, gr, "fp8")
    w = written_rows(inputs, wl.S)
    b0 = si.stored_to_f64(inputs["bank"], wl.dtype).astype(np.float32)
    expect = b0.copy()
    expect[w] = fp8_rows(b0[w])
    assert np.array_equal(bank.float().cpu().numpy(), expect)
    assert np.array_equal(ref["restored_bank"].astype(np.float32), expect)
    errs = errors(out, ref)
    tol = 1e-4 if bank_dtype == "f32" else 2e-2
    assert all(v <= tol for v in errs.values()), errs


@pytest.mark.parametrize("flags", [0, sdm.FLAG_PER_STEP_KERNELS])
def test_fp8_snapshot_general_slots(flags):
    """Zipf slots rewritten across chunks, ragged tokens, slabs: the restored bank is
    fp8(initial) on every written row, bit for bit, and the run is deterministic. (Gradients
    are not compared here: an intermediate row at an fp8 rounding boundary can round one way
    from the GPU's float32 value and the other from the oracle's fp64 value, a step of up to
    one part in sixteen.)"""
    wl = small_workload(P=2, T=90, C=16, S=30, D=64, W=4, R=3, dtype="f32", ragged=True,
                        seed=72)
    inputs, gr, _ = make_case(wl)
    _, bank, _, out = gpu_backward(wl, inputs, gr, slab_steps=2, flags=flags,
                                   snapshot_quant="fp8")
    w = written_rows(inputs, wl.S)
    expect = inputs["bank"].copy()
    expect[w] = fp8_rows(inputs["bank"][w])
    assert np.array_equal(bank.cpu().numpy(), expect)
    _, _, _, out2 = gpu_backward(wl, inputs, gr, slab_steps=2, flags=flags,
                                 snapshot_quant="fp8")
    for k in GRADS:
        assert torch.equal(out[k], out2[k]), k
