"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on the GPU."""

import numpy as np
import pytest
import torch

import oracle
import sdm_inputs as si
import sparse_addressed_delta_gb300 as sdm
from sdm_case import (TOL, compare_with_oracle, f64, oracle_args, run_gpu, small_workload,
                      to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    sdm.library()


PATHS = [0, sdm.FLAG_PER_STEP_KERNELS]      # fused Phase 2 (default), per-step kernels


def check(wl, inputs=None, slab_steps=0, flags=(0, sdm.FLAG_PER_STEP_KERNELS)):
    """Both Phase-2 paths against the oracle (and each other, within the tolerance)."""
    inputs = si.generate(wl) if inputs is None else inputs
    dev = to_device(inputs, wl)
    tol = TOL[wl.dtype]
    errs = []
    for fl in flags:
        r, b, ws = run_gpu(wl, dev, slab_steps, flags=fl)
        st = sdm.device_status(ws)
        assert st["code"] == 0 and st["bad_slots"] == 0 and st["repeated_write_slots"] == 0, st
        er, eb = compare_with_oracle(wl, inputs, r, b)
        assert er <= tol and eb <= tol, (wl.name, fl, er, eb)
        errs.append((er, eb))
    return errs[0]


def test_workload0_full():
    er, eb = check(si.WORKLOADS[0])
    assert er <= 1e-4 and eb <= 1e-4


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("D", [32, 64, 128, 256, 512])
def test_head_dims(dtype, D):
    check(small_workload(P=2, T=77, C=16, S=50, D=D, W=3, R=5, dtype=dtype, seed=D))


@pytest.mark.parametrize("C", [16, 32, 48, 64, 100, 128, 256])
def test_chunk_sizes_ragged(C):
    """Several chunks per stream, a ragged last chunk and ragged valid tokens."""
    check(small_workload(P=3, T=3 * C + 7, C=C, S=97, D=64, W=5, R=4, seed=C))


@pytest.mark.parametrize("W,R", [(1, 1), (1, 7), (16, 16), (33, 9), (64, 64)])
def test_widths(W, R):
    check(small_workload(P=2, T=150, C=32, S=max(200, 3 * W), D=64, W=W, R=R,
                         slots="zipf1.1", seed=W * 100 + R))


@pytest.mark.parametrize("C,W,R,dtype", [(64, 20, 20, "bf16"), (32, 40, 40, "f32")])
def test_pipelined_more_entries_than_early_loads(C, W, R, dtype):
    """Pipelined Phase 2 with more than four entries per gather lane: the entries past the
    early-loaded ones (linked or not) are fetched in the step itself. Small banks make many
    entries link to the previous step's groups."""
    wl = small_workload(P=2, T=5 * C + 3, C=C, S=300, D=128, W=W, R=R, dtype=dtype,
                        slots="zipf1.1", seed=C + W)
    shape = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R,
                           torch.float32 if dtype == "f32" else torch.bfloat16)
    assert sdm.launch_count(shape) == 3          # the pipelined kernel runs
    check(wl)


def test_dense_collisions_tiny_bank():
    """A bank of W rows: every token writes every row (groups of the whole chunk)."""
    check(small_workload(P=2, T=130, C=64, S=8, D=32, W=8, R=8, slots="uniform", seed=5))


def test_mix_slots_bf16():
    check(small_workload(P=2, T=300, C=64, S=4096, D=128, W=32, R=32, dtype="bf16",
                         slots="mix", seed=9))


@pytest.mark.parametrize("flags", PATHS)
def test_empty_streams_and_full_padding(flags):
    wl = small_workload(P=4, T=64, C=16, S=40, D=64, W=3, R=3, ragged=False, seed=3)
    inputs = si.generate(wl)
    inputs["valid"] = np.array([0, 1, 17, 64], np.int32)
    for k in ("write_slots", "read_slots"):
        inputs[k][0] = 0
        inputs[k][1, 1:] = 0
        inputs[k][2, 17:] = 0
    dev = to_device(inputs, wl)
    r, b, _ = run_gpu(wl, dev, flags=flags)
    assert not f64(r[0]).any() and not f64(r[1, 1:]).any() and not f64(r[2, 17:]).any()
    assert torch.equal(b[:wl.S], dev["bank"][:wl.S])
    er, eb = compare_with_oracle(wl, inputs, r, b)
    assert er <= 1e-4 and eb <= 1e-4


@pytest.mark.parametrize("flags", PATHS)
def test_padding_inputs_never_read(flags):
    """NaN in every input of a padding token changes nothing, bit for bit."""
    wl = small_workload(P=3, T=90, C=32, S=64, D=64, W=4, R=4, ragged=True, seed=8)
    inputs = si.generate(wl)
    dev = to_device(inputs, wl)
    r1, b1, _ = run_gpu(wl, dev, flags=flags)
    pad = torch.arange(wl.T, device="cuda")[None, :] >= dev["valid"][:, None]
    for k in ("write_w", "log_decay", "v", "read_w"):
        dev[k][pad] = float("nan")
    dev["beta"][pad] = float("nan")
    dev["write_slots"][pad] = -5
    dev["read_slots"][pad] = 1 << 30
    r2, b2, ws = run_gpu(wl, dev, flags=flags)
    assert torch.equal(r1, r2) and torch.equal(b1, b2)
    assert sdm.device_status(ws)["code"] == 0


@pytest.mark.parametrize("flags", PATHS)
def test_deterministic_bitwise(flags):
    wl = small_workload(P=4, T=256, C=64, S=300, D=128, W=16, R=16, dtype="bf16", seed=11)
    dev = to_device(si.generate(wl), wl)
    r1, b1, _ = run_gpu(wl, dev, flags=flags)
    r2, b2, _ = run_gpu(wl, dev, flags=flags)
    assert torch.equal(r1, r2) and torch.equal(b1, b2)


@pytest.mark.parametrize("flags", PATHS)
def test_slab_invariance_bitwise(flags):
    wl = small_workload(P=3, T=200, C=16, S=100, D=64, W=4, R=4, seed=12)
    dev = to_device(si.generate(wl), wl)
    r0, b0, _ = run_gpu(wl, dev, slab_steps=0, flags=flags)
    for ns in (1, 2, 5):
        r, b, _ = run_gpu(wl, dev, slab_steps=ns, flags=flags)
        assert torch.equal(r, r0) and torch.equal(b, b0), ns


@pytest.mark.parametrize("flags", PATHS)
def test_bad_slot_is_reported_and_dropped(flags):
    """A slot outside [0, S) is reported and its entry dropped: the result equals the call
    in which that entry has weight 0 and log-decay 0 on an unused slot."""
    wl = small_workload(P=2, T=40, C=16, S=64, D=64, W=4, R=4, ragged=False, seed=13)
    inputs = si.generate(wl)
    ref_in = {k: v.copy() for k, v in inputs.items()}
    inputs["write_slots"][1, 5, 2] = 1 << 30
    inputs["read_slots"][0, 9, 1] = -3
    free = sorted(set(range(wl.S)) - set(ref_in["write_slots"][1, 5].tolist()))[0]
    ref_in["write_slots"][1, 5, 2] = free
    ref_in["write_w"][1, 5, 2] = 0
    ref_in["log_decay"][1, 5, 2] = 0
    ref_in["read_w"][0, 9, 1] = 0
    r, b, ws = run_gpu(wl, to_device(inputs, wl), flags=flags)
    st = sdm.device_status(ws)
    assert st["code"] == -6 and st["bad_slots"] == 2
    assert st["first_bad_token"] in (1 * wl.T + 5, 9)
    r2, b2, _ = run_gpu(wl, to_device(ref_in, wl), flags=flags)
    assert (r - r2).abs().max() <= 1e-5 * r2.abs().max()
    assert (b - b2).abs().max() <= 1e-5 * b2.abs().max()


def test_repeated_write_slot_is_counted():
    wl = small_workload(P=1, T=40, C=16, S=64, D=64, W=4, R=4, ragged=False, seed=14)
    inputs = si.generate(wl)
    inputs["write_slots"][0, 7, 3] = inputs["write_slots"][0, 7, 0]
    dev = to_device(inputs, wl)
    _, _, ws = run_gpu(wl, dev)
    assert sdm.device_status(ws)["repeated_write_slots"] == 1


def _phase1_launches(wl) -> int:
    """Phase-1 launches per slab for the shape of ``wl``: 1 with the chunk's scratch on chip,
    2 when Phase 1 splits into the sort kernel and the row kernel over global scratch, 3 with
    the dense-Gram kernel (C >= 128) (the per-step launch count of one slab is Phase 1 + solve
    + 3 per step)."""
    shape = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R,
                           torch.float32 if wl.dtype == "f32" else torch.bfloat16,
                           wl.Nt, sdm.FLAG_PER_STEP_KERNELS)
    return sdm.launch_count(shape) - 1 - 3 * wl.Nt


def _dense_groups(slots, lw, C):
    """Groups of one chunk that the split Phase-1 path should take in the dense Gram form
    (slots and lw of the chunk's valid write entries, token-major): none below C = 128; else
    the groups of at least thr members, thr the least of (C/8) * 2^L (L < 8) that leaves at
    most C of them, whose running log-decays lie within 64 of each other."""
    s, l = slots.ravel(), lw.ravel()
    if s.size == 0 or C < 128:
        return 0
    _, inv, cnt = np.unique(s, return_inverse=True, return_counts=True)
    thr0 = max(4, C // 8)
    for lev in range(8):
        thr = thr0 << lev
        if (cnt >= thr).sum() <= C:
            break
    else:
        return 0
    n = 0
    for gi in np.nonzero(cnt >= thr)[0]:
        ls = l[inv == gi]
        span = ls.max() - ls.min()
        assert abs(span - 64.0) > 1e-3, "a group's span is too close to the dense limit"
        n += int(span <= 64.0)
    return n


def _check_phase1(wl, values=True, inputs=None, dense=None):
    """Phase 1 and the solve against the oracle, chunk by chunk: the dedup plan (perm, group
    starts, owners, group count) bit for bit, and (``values``) lw, gw, dw, lr, qw, A, QK, X and
    QX within float32 rounding of the oracle's chunked form. ``dense`` (split path, with
    ``values``): check each chunk's dense Gram group count against the rule and require at
    least that many dense groups over the call (True: at least one)."""
    inputs = si.generate(wl) if inputs is None else inputs
    dev = to_device(inputs, wl)
    out = sdm.phase1_debug(dev["write_slots"], dev["write_w"], dev["log_decay"], dev["beta"],
                           dev["read_slots"], dev["read_w"], dev["valid"], S=wl.S, D=wl.D,
                           chunk_size=wl.C)
    torch.cuda.synchronize()
    assert sdm.device_status(out["workspace"])["code"] == 0
    x = oracle.from_stored(inputs, wl.dtype) if values else None
    C, W = wl.C, wl.W
    perm, gs, ow = (out[k].cpu().numpy() for k in ("perm", "group_start", "owner"))
    ng = out["ngroups"].cpu().numpy()
    ndense = out["dense_groups"].cpu().numpy()
    dense_total = 0
    for ti in range(wl.Nt):
        for p in range(wl.P):
            n = ti * wl.P + p
            nv = int(np.clip(inputs["valid"][p] - ti * C, 0, C))
            pl = oracle.plan(inputs["write_slots"][p, ti * C:ti * C + nv])
            m = nv * W
            assert np.array_equal(perm[n, :m], pl["perm"]), (ti, p)
            assert (perm[n, m:] == -1).all()
            assert np.array_equal(gs[n, :m], pl["group_start"]), (ti, p)
            assert np.array_equal(ow[n, :m], pl["owner"]), (ti, p)
            assert int(ng[n]) == pl["groups"]
            if not values:
                continue
            _, _, d = oracle.chunked(C, *oracle_args(x), debug=(p, ti))
            if dense is not None:
                want = _dense_groups(inputs["write_slots"][p, ti * C:ti * C + nv],
                                     d["lw"][:nv], C)
                assert int(ndense[n]) == want, (ti, p, int(ndense[n]), want)
                dense_total += want
            for key, ref in (("lw", d["lw"]), ("gw", d["gw"]), ("dw", d["dw"]), ("lr", d["lr"]),
                             ("qw", d["qw"]), ("A", d["A"]), ("QK", d["QK"]), ("X", d["X"]),
                             ("QX", d["QX"])):
                got = out[key][n].double().cpu().numpy().reshape(ref.shape)
                scale = max(np.abs(ref).max(), 1e-30)
                assert np.abs(got - ref).max() <= 2e-6 * scale + 1e-30, (key, ti, p)
    if dense is not None:
        assert dense_total >= (1 if dense is True else dense), dense_total


def test_phase1_plan_and_intermediates():
    """The on-chip Phase-1 path (the chunk's scratch in shared memory)."""
    wl = small_workload(P=2, T=70, C=16, S=20, D=32, W=4, R=3, ragged=True, seed=15)
    assert _phase1_launches(wl) == 1
    _check_phase1(wl)


def _steep_odd_slots(inputs, factor=40.0):
    """The log-decays of the writes to odd slots times ``factor``: large groups of odd slots
    then span far more than the dense form's limit and keep their pair sums."""
    g = inputs["log_decay"]
    odd = (inputs["write_slots"] % 2) == 1
    inputs["log_decay"] = np.where(odd, g * np.float32(factor), g).astype(np.float32)
    return inputs


@pytest.mark.parametrize("wl,values", [
    # the ragged workload's chunk shape (C=64, W=R=32, Zipf(1.1))
    (small_workload(P=2, T=3 * 64 + 9, C=64, S=4096, D=64, W=32, R=32, dtype="bf16",
                    slots="zipf1.1", ragged=True, seed=16), True),
    # the forward+backward workload's chunk shape (C=128, W=R=64 uniform), small bank
    (small_workload(P=2, T=2 * 128 + 50, C=128, S=2048, D=64, W=64, R=64, dtype="f32",
                    slots="uniform", ragged=True, seed=17), True),
    # C=256 with the half-Zipf(1.2) mix: hot groups of up to a whole chunk of members
    (small_workload(P=1, T=300, C=256, S=4096, D=64, W=32, R=32, dtype="bf16", slots="mix",
                    ragged=False, seed=18), True),
    # the widest workload's chunk shape (C=256, W=R=256 mix): the plan only (the oracle's
    # brute-force Gram sums would take minutes at this width)
    (small_workload(P=1, T=256 + 40, C=256, S=1 << 20, D=64, W=256, R=256, dtype="bf16",
                    slots="mix", ragged=False, seed=19), False),
], ids=["c64_w32_zipf", "c128_w64_uniform", "c256_w32_mix", "c256_w256_mix_plan"])
def test_phase1_split_path(wl, values):
    """The Phase-1 path over global scratch (sort kernel + row kernel + dense-Gram kernel),
    which the larger workloads take: its dedup plan bit for bit, and the values within float32
    rounding."""
    assert _phase1_launches(wl) == (3 if wl.C >= 128 else 2)
    _check_phase1(wl, values, dense=False if values else None)


@pytest.mark.parametrize("case", ["mix", "steep_odd", "crowded"])
def test_phase1_dense_gram_groups(case):
    """The large groups' Gram sums in the dense factor form, against the oracle's pair sums:
    - mix: the half-Zipf(1.2) mix at C=256, whose hot slots go dense;
    - steep_odd: the same with 40x the log-decay on odd slots, whose large groups then span
      past the dense limit and keep their pair sums beside the dense even ones;
    - crowded: 300 slots under 64 writes per token, so more than C groups reach the first
      size threshold and the threshold doubles."""
    if case == "crowded":
        wl = small_workload(P=1, T=256 + 60, C=256, S=300, D=64, W=64, R=48, dtype="f32",
                            slots="uniform", ragged=False, seed=21)
    else:
        wl = small_workload(P=1, T=300, C=256, S=4096, D=64, W=32, R=32, dtype="bf16",
                            slots="mix", ragged=False, seed=20)
    assert _phase1_launches(wl) == 3
    inputs = si.generate(wl)
    if case == "steep_odd":
        inputs = _steep_odd_slots(inputs)
    _check_phase1(wl, True, inputs=inputs, dense=True)
    if case == "steep_odd":
        # the large odd groups really were left to the pair sums
        x = oracle.from_stored(inputs, wl.dtype)
        _, _, d = oracle.chunked(wl.C, *oracle_args(x), debug=(0, 0))
        s = inputs["write_slots"][0, :wl.C].ravel()
        l = d["lw"].ravel()
        _, inv, cnt = np.unique(s, return_inverse=True, return_counts=True)
        odd_big = [gi for gi in np.nonzero(cnt >= 32)[0] if s[inv == gi][0] % 2 == 1]
        assert odd_big and all(np.ptp(l[inv == gi]) > 64.0 for gi in odd_big)
    # the dense form gives the same bits on a second call (fixed-order sums)
    dev = to_device(inputs, wl)
    outs = [sdm.phase1_debug(dev["write_slots"], dev["write_w"], dev["log_decay"], dev["beta"],
                             dev["read_slots"], dev["read_w"], dev["valid"], S=wl.S, D=wl.D,
                             chunk_size=wl.C) for _ in range(2)]
    for k in ("A", "QK", "X", "QX"):
        assert torch.equal(outs[0][k], outs[1][k]), k


def test_full_size_dense_gram_path():
    """The widest workload's chunk shape (C=256, W=R=256, the mix) reaches the dense form and
    stays within tolerance end to end (two streams, four chunks each)."""
    wl = small_workload(P=2, T=4 * 256, C=256, S=1 << 20, D=64, W=256, R=256, dtype="bf16",
                        slots="mix", ragged=False, seed=22)
    dev = to_device(si.generate(wl), wl)
    out = sdm.phase1_debug(dev["write_slots"], dev["write_w"], dev["log_decay"], dev["beta"],
                           dev["read_slots"], dev["read_w"], dev["valid"], S=wl.S, D=wl.D,
                           chunk_size=wl.C)
    assert (out["dense_groups"].cpu().numpy() > 16).all()
    check(wl)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_full_size_workloads(cfg):
    """The four larger workloads at full size (the launch configuration bench.py times),
    whole readings and final bank."""
    wl = si.WORKLOADS[cfg]
    inputs = si.generate(wl)
    dev = to_device(inputs, wl)
    r, b, ws = run_gpu(wl, dev)
    st = sdm.device_status(ws)
    assert st["code"] == 0 and st["repeated_write_slots"] == 0, st
    del dev
    group = max(1, min(8, (1 << 30) // (wl.S * wl.D * 8)))   # about 1 GiB of fp64 bank per group
    er, eb = compare_with_oracle(wl, inputs, r, b, streams_per_call=group, nthreads=group)
    tol = TOL[wl.dtype]
    print(f"{wl.name}: readings err {er:.3e}, bank err {eb:.3e} (tol {tol})")
    assert er <= tol and eb <= tol


@pytest.mark.parametrize("flags", PATHS)
@pytest.mark.parametrize("C,W", [(16, 4), (128, 64)])
def test_workspace_poison(flags, C, W):
    """Every workspace byte the call reads it has written first: a NaN-filled workspace gives
    the same bits as a zero-filled one."""
    wl = small_workload(P=3, T=3 * C + 5, C=C, S=300, D=64, W=W, R=W, dtype="bf16", seed=C)
    dev = to_device(si.generate(wl), wl)
    shape = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R, torch.bfloat16, 0, flags)
    n = sdm.workspace_bytes(shape)
    outs = []
    for fill in (0x00, 0xFF):
        ws = torch.full((n,), fill, dtype=torch.uint8, device="cuda")
        r, b, _ = run_gpu(wl, dev, workspace=ws, flags=flags)
        outs.append((r, b))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert torch.isfinite(outs[1][0].float()).all()
