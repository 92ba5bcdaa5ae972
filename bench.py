#!/usr/bin/env python
"""Benchmark of the chunked SDM write/read forward on GB300: forward tokens/s, and the
Phase-2 gather/DW achieved HBM bandwidth against the measured peak.

A step is one full sdm_write_read call (Phase 1, solve, and all Nt Phase-2 steps) over the
widest workload: P=4 streams x T=16384 tokens, C=256, S=1048576 x D=256 bf16 bank, W=R=256
slots per token (half Zipf(1.2), half uniform), slabbed Phase-1 state (seeded synthetic inputs,
``sdm_inputs``). The call is captured once in a CUDA graph and replayed; before every step the
bank is reset from a pristine copy and a 512 MiB buffer is written to flush L2 (both outside
the per-step CUDA events).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Other measurements (one JSON line each, same timing rules):
    --workload I                 another of the five workloads (sdm_inputs.WORKLOADS[I])
    --per-step-kernels           Phase 2 as three kernels per step
    --backward [--snapshot-quant none|bf16|fp8]
                                 the saving forward + backward (one step = both calls)
    --layer-io                   the head split/merge and bank expand/sum kernels, in GB/s

The ``roofline`` object describes the kernel family with the most device time in a call,
against its own bound: HBM bytes for the gather, DW and fused Phase 2 (one read of every
distinct row a chunk touches, one write of every distinct row it writes); tensor-core FLOPs for
the dual matmul (two C x C by C x D products per chunk, against the TF32 rate); FP32 FMA FLOPs
for the solve (C^3/3 multiply-adds per chunk); and Gram pair terms for Phase 1 (one exp per
pair of entries of a slot, against the exp unit's rate).

With N > 1 (torchrun, one rank per GPU) every rank runs its own copy of the workload
(different seed): weak scaling, no collective on the data path; value = all ranks' tokens /
the slowest rank's time. ``--impl reference`` times the CPU oracle (fp64 token loop, plain C)
on the host cores instead, rank 0 only, on a bounded sample of the workload (the first tokens
of every stream).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import sdm_inputs as si  # noqa: E402

METRIC = "SDM forward tokens/s on 1 GB300; Phase-2 achieved HBM GB/s vs peak"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4, help="index into sdm_inputs.WORKLOADS")
    ap.add_argument("--profile-steps", type=int, default=3)
    ap.add_argument("--per-step-kernels", action="store_true",
                    help="run Phase 2 as three kernels per step instead of the fused kernel")
    ap.add_argument("--backward", action="store_true",
                    help="time the saving forward + backward (one step = both calls) instead")
    ap.add_argument("--layer-io", action="store_true",
                    help="time the layer I/O kernels (head split/merge, bank expand/sum) on the "
                         "batch 4 x 8 heads layout of the ragged workload instead")
    ap.add_argument("--product-key", action="store_true",
                    help="time the product-key exact top-k (forward and backward) instead")
    ap.add_argument("--snapshot-quant", choices=["none", "bf16", "fp8"], default="none",
                    help="with --backward: store the snapshot in bfloat16 (float32 banks) or "
                         "float8_e4m3fn")
    ap.add_argument("--ncu-run", type=int, default=0, metavar="K",
                    help="profiling target: run K plain (eager) calls on the workload and exit, "
                         "printing no benchmark line")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_totals(ms: float, tokens: int, world: int, device=None):
    """Whole-job figures of a weak-scaling run: (the slowest rank's time, all ranks' tokens).
    Every rank calls it with its own numbers; with world > 1 it reduces over the default
    process group (MAX of the times, SUM of the tokens: ranks draw different seeds, so their
    valid-token counts differ on ragged workloads). Works with the nccl and gloo backends."""
    if world <= 1:
        return float(ms), int(tokens)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    n = torch.tensor([int(tokens)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def workload_config(wl, inputs):
    return {"workload": wl.name, "P": wl.P, "T": wl.T, "C": wl.C, "S": wl.S, "D": wl.D,
            "W": wl.W, "R": wl.R, "bank_dtype": wl.dtype, "slots": wl.slots,
            "valid_tokens": int(inputs["valid"].sum()), "seed": wl.seed,
            "l2": "flushed before every step (512 MiB write); bank reset from a pristine copy"}


# ------------------------------------------------------------------------------------------
# algorithmic bytes
# ------------------------------------------------------------------------------------------

def algorithmic_bytes(wl, inputs):
    """Bank bytes the method must move, summed over all steps: per chunk, one read of every
    distinct row it touches (writes and reads) and one write of every distinct written row.
    Split as the gather's reads (|U_w u U_r| rows), the DW's read+write (2 |U_w|) and the
    Phase-2 minimum (|U_w u U_r| + |U_w|)."""
    es = 4 if wl.dtype == "f32" else 2
    row = wl.D * es
    g_rows = dw_rows = 0
    for p in range(wl.P):
        v = int(inputs["valid"][p])
        for ti in range(wl.Nt):
            lo, hi = ti * wl.C, min(v, ti * wl.C + wl.C)
            if hi <= lo:
                continue
            uw = np.unique(inputs["write_slots"][p, lo:hi])
            ur = np.unique(inputs["read_slots"][p, lo:hi])
            g_rows += np.union1d(uw, ur).size
            dw_rows += uw.size
    return {"gather": g_rows * row, "dw": 2 * dw_rows * row, "phase2": (g_rows + dw_rows) * row}


def gram_pairs(wl, inputs):
    """Gram pair terms of the whole call (Phase 1's algorithmic unit): per chunk, every pair of
    write entries of one slot at tokens u < t (a term of A) and every pair (read of slot s at
    token t, write of s at token u <= t) (a term of QK). Each term is one exp of a difference of
    running log-decays, two multiplies and an add."""
    total = 0
    C = wl.C
    for p in range(wl.P):
        v = int(inputs["valid"][p])
        for ti in range(wl.Nt):
            lo, hi = ti * C, min(v, ti * C + C)
            if hi <= lo:
                continue
            w = inputs["write_slots"][p, lo:hi].astype(np.int64)
            r = inputs["read_slots"][p, lo:hi].astype(np.int64)
            _, cnt = np.unique(w, return_counts=True)
            total += int((cnt * (cnt - 1) // 2).sum())
            tw = np.repeat(np.arange(hi - lo, dtype=np.int64), w.shape[1])
            key_w = np.sort(w.ravel() * 1024 + tw)
            tr = np.repeat(np.arange(hi - lo, dtype=np.int64), r.shape[1])
            rr = r.ravel()
            total += int((np.searchsorted(key_w, rr * 1024 + tr, side="right")
                          - np.searchsorted(key_w, rr * 1024, side="left")).sum())
    return total


def kernel_units(wl, inputs, kind, launches_per_call):
    """(algorithmic units per launch, unit name, bound) of a kernel family; see the module
    docstring."""
    es = 4 if wl.dtype == "f32" else 2
    if kind in ("gather", "dw", "phase2"):
        alg = algorithmic_bytes(wl, inputs)
        return alg[kind] / max(1, launches_per_call), "bytes", "hbm"
    chunks = wl.P * wl.Nt
    if kind == "dualmm":      # delta_v = X u_pre and readings = QX u_pre per chunk
        return 2 * 2.0 * wl.C * wl.C * wl.D * chunks / max(1, launches_per_call), "flop", "tensor"
    if kind == "solve":       # X = (I + L)^-1 (C^3/6 FMA) and QX = QK X (C^3/6 FMA)
        return 2.0 * (wl.C ** 3 / 3.0) * chunks / max(1, launches_per_call), "flop", "alu"
    if kind == "phase1":
        return gram_pairs(wl, inputs) / max(1, launches_per_call), "pair terms", "alu"
    raise ValueError(kind)


def kernel_peak(kind):
    """(peak, unit, source) for a kernel family's bound on this GPU."""
    try:
        mp = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        mp = {}
    sm_hz = float(mp.get("sm_max_mhz", 2070.0)) * 1e6
    if kind in ("gather", "dw", "phase2"):
        hbm, src = measured_peak()
        return hbm * 1e9, "GB/s", f"{src} (MEASURED_PEAKS.json hbm_gbs)"
    if kind == "dualmm":
        bf16 = float(mp.get("bf16_tflops", 1900.0))
        return (bf16 * 1e12 * 1.1 / 2.25, "TFLOP/s",
                f"{'measured' if mp else 'fallback'} bf16 dense {bf16:.0f} TFLOP/s x the nominal "
                "TF32/bf16 ratio 1.1/2.25")
    if kind == "solve":
        return (152 * 128 * 2 * sm_hz, "TFLOP/s",
                "FP32 FMA: 152 SMs x 128 lanes x 2 flop x max SM clock")
    if kind == "phase1":
        return (152 * 16 * sm_hz, "G pair terms/s",
                "exp unit: 152 SMs x 16 exp per clock x max SM clock, one exp per pair term")
    raise ValueError(kind)


# ------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (every 200 ms) of the SM clock and throttle reasons of one GPU."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.5)          # let the first sample land before the timed region

    def stop(self):
        time.sleep(0.3)
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch of ``kernel`` on ``workload`` from the committed ncu summary, if
    every source the record names is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        for rec in json.load(open(path))[kernel]:
            if rec["workload"] != workload:
                continue
            h = hashlib.sha256()
            for name in rec["sources"]:
                h.update(open(os.path.join(ROOT, "sparse_addressed_delta_gb300", "csrc", name),
                              "rb").read())
            if h.hexdigest()[:16] != rec["sources_sha256_16"]:
                return None
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None
    return None


# ------------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline field)
# ------------------------------------------------------------------------------------------

def oracle_sample(wl, inputs, target_s: float):
    """A bounded sample of the workload for the CPU oracle: the first Ts tokens of every stream
    (Ts a multiple of C, sized so that one oracle run takes about ``target_s`` seconds on this
    host; the token loop's cost per token does not depend on the token's position). The bank
    rows the sample touches are gathered into a compact bank and the sample's slot ids renumbered
    to match (the oracle copies its whole bank in fp64 on every call; the untouched rows would
    only add that copy). Returns (fp64 oracle inputs, valid tokens in the sample, Ts, threads)."""
    import oracle

    threads = max(1, min(wl.P, os.cpu_count() or 1))

    def cut(ts):
        ws, rs = inputs["write_slots"][:, :ts], inputs["read_slots"][:, :ts]
        rows = [np.unique(np.concatenate([ws[p].ravel(), rs[p].ravel()])) for p in range(wl.P)]
        S2 = max(1, max(r.size for r in rows))
        bank = np.zeros((wl.P * S2, wl.D), inputs["bank"].dtype)
        ws2, rs2 = np.empty_like(ws), np.empty_like(rs)
        for p, r in enumerate(rows):
            bank[p * S2:p * S2 + r.size] = inputs["bank"][p * wl.S + r]
            ws2[p] = np.searchsorted(r, ws[p])
            rs2[p] = np.searchsorted(r, rs[p])
        sub = {k: inputs[k][:, :ts] for k in ("write_w", "log_decay", "beta", "v", "read_w")}
        sub.update(write_slots=ws2, read_slots=rs2, bank=bank,
                   valid=np.minimum(inputs["valid"], ts).astype(np.int32))
        return oracle.from_stored(sub, wl.dtype), int(sub["valid"].sum())

    ts = min(wl.T, wl.C)
    x, n = cut(ts)
    t = max(run_oracle(x, threads), 1e-6)
    ts = int(min(wl.T, max(wl.C, ts * target_s / t // wl.C * wl.C)))
    x, n = cut(ts)
    return x, n, ts, threads


def run_oracle(x, threads):
    import oracle

    t0 = time.perf_counter()
    oracle.sequential(x["bank"], x["ws"], x["k"], x["g"], x["beta"], x["v"], x["rs"], x["q"],
                      x["valid"], nthreads=threads)
    return time.perf_counter() - t0


def time_oracle(wl, inputs, target_s: float = 3.0, reps: int = 3):
    x, n, ts, threads = oracle_sample(wl, inputs, target_s)
    times = [run_oracle(x, threads) for _ in range(reps)]
    t = statistics.median(times)
    return {"value": n / t, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"the first {ts} of {wl.T} tokens of every stream ({n} tokens; the rows "
                      "they touch gathered into a compact bank), fp64 token loop in C, OpenMP "
                      f"over streams, median of {reps} runs ({t:.3f} s each)"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    wl = si.WORKLOADS[args.workload]
    inputs = si.generate(wl)
    # one step = the oracle over a sample of about one second of host work
    x, n, ts, threads = oracle_sample(wl, inputs, 1.0)
    for _ in range(args.warmup):
        run_oracle(x, threads)
    times = [run_oracle(x, threads) for _ in range(args.steps)]
    t = statistics.mean(times)
    value = n / t
    sample = (f"the first {ts} of {wl.T} tokens of every stream ({n} tokens; the rows they "
              "touch gathered into a compact bank) per step, fp64 token loop in C, OpenMP over "
              "streams")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, inputs),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist

    import sparse_addressed_delta_gb300 as sdm

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://", world_size=world, rank=rank,
                                device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    base = si.WORKLOADS[args.workload]
    wl = base.replace(seed=base.seed + 1000 * rank) if world > 1 else base
    inputs = si.generate(wl)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16

    def tens(name):
        t = torch.from_numpy(np.ascontiguousarray(inputs[name]))
        if wl.dtype == "bf16" and inputs[name].dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t

    host = {k: tens(k).pin_memory() for k in ("write_slots", "write_w", "log_decay", "beta", "v",
                                              "read_slots", "read_w", "valid")}
    d_in = {k: v.to(dev) for k, v in host.items()}
    bank0 = tens("bank").to(dev)
    bank = bank0.clone()
    flags = sdm.FLAG_PER_STEP_KERNELS if args.per_step_kernels else 0
    shape = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R, dt, flags=flags)
    ws = sdm.alloc_workspace(shape, dev)
    readings = torch.empty((wl.P, wl.T, wl.D), dtype=dt, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    tokens = int(inputs["valid"].sum())
    launches_per_call = sdm.launch_count(shape)

    stream = torch.cuda.Stream(device=dev)

    def call():
        sdm.sdm_write_read(bank, d_in["write_slots"], d_in["write_w"], d_in["log_decay"],
                           d_in["beta"], d_in["v"], d_in["read_slots"], d_in["read_w"],
                           d_in["valid"], chunk_size=wl.C, workspace=ws, readings=readings,
                           stream=stream, flags=flags)

    with torch.cuda.stream(stream):
        call()                                   # eager run (sets kernel attributes)
    stream.synchronize()
    st = sdm.device_status(ws, stream)
    if st["code"] != 0:
        raise RuntimeError(f"device status {st}")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()

    def prepare():
        bank.copy_(bank0)
        flush.zero_()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            prepare()
            graph.replay()
    stream.synchronize()

    # ---- timed region: K graph replays, device-timed per step ----
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            prepare()
            ev[k][0].record(stream)
            graph.replay()
            ev[k][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall1 = time.perf_counter()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(step_ms)
    ms_max, tokens_all = rank_totals(ms, tokens, world, dev)
    value = tokens_all / (ms_max / 1e3)

    # ---- per-kernel device times (same protocol, events around every launch) ----
    fam_ms = {k: 0.0 for k in sdm.KERNEL_KINDS}
    fam_n = {k: 0 for k in sdm.KERNEL_KINDS}
    for _ in range(args.profile_steps):
        with torch.cuda.stream(stream):
            prepare()
        _, prof = sdm.profile_write_read(bank, d_in["write_slots"], d_in["write_w"],
                                         d_in["log_decay"], d_in["beta"], d_in["v"],
                                         d_in["read_slots"], d_in["read_w"], d_in["valid"],
                                         chunk_size=wl.C, workspace=ws, readings=readings,
                                         stream=stream, flags=flags)
        for k, (t, n) in prof.items():
            fam_ms[k] += t
            fam_n[k] += n
    kernels = {k: {"ms_per_call": fam_ms[k] / args.profile_steps,
                   "launches_per_call": fam_n[k] // args.profile_steps,
                   "us_per_launch": 1e3 * fam_ms[k] / max(1, fam_n[k]),
                   "share": fam_ms[k] / max(1e-12, sum(fam_ms.values()))}
               for k in sdm.KERNEL_KINDS}

    # ---- roofline of the dominant kernel and of the Phase-2 gather + DW pair ----
    alg = algorithmic_bytes(wl, inputs)
    peak, peak_src = measured_peak()
    dom = max(sdm.KERNEL_KINDS, key=lambda k: fam_ms[k])
    n_per_call = max(1, fam_n[dom] // args.profile_steps)
    units, unit_name, bound = kernel_units(wl, inputs, dom, n_per_call)
    secs = fam_ms[dom] / max(1, fam_n[dom]) / 1e3
    pk, pk_unit, pk_src = kernel_peak(dom)
    scale = {"GB/s": 1e9, "TFLOP/s": 1e12, "G pair terms/s": 1e9}[pk_unit]
    ach = units / secs
    roofline = {"kernel": dom, "bound": bound, "achieved": ach / scale, "peak": pk / scale,
                "unit": pk_unit, "frac": ach / pk, "peak_source": pk_src,
                "alg_units_per_launch": units, "alg_unit": unit_name,
                "launch_us": secs * 1e6,
                "traffic": traffic_record(dom, wl.name)}
    p2_ms = fam_ms["gather"] + fam_ms["dw"] + fam_ms["phase2"]
    p2_secs = p2_ms / args.profile_steps / 1e3
    p2_ach = alg["phase2"] / p2_secs / 1e9
    phase2 = {"kernels": "fused phase2" if fam_n["phase2"] else "gather + dw",
              "alg_bytes_per_call": alg["phase2"], "achieved": p2_ach, "peak": peak,
              "unit": "GB/s", "frac": p2_ach / peak}

    # ---- end to end through the public API: sdm_write_read_host with the inputs in pinned
    #      host memory and the readings written back into pinned host memory, one call per
    #      step (captured in a CUDA graph like the device call) ----
    h_read = torch.empty((wl.P, wl.T, wl.D), dtype=dt, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = h_read.numel() * h_read.element_size()
    ws_h = torch.empty(sdm.host_workspace_bytes(shape), dtype=torch.uint8, device=dev)

    def host_call():
        sdm.sdm_write_read_host(bank, host["write_slots"], host["write_w"], host["log_decay"],
                                host["beta"], host["v"], host["read_slots"], host["read_w"],
                                host["valid"], chunk_size=wl.C, readings=h_read,
                                workspace=ws_h, stream=stream, flags=flags)

    with torch.cuda.stream(stream):
        prepare()
        host_call()
    stream.synchronize()
    graph_h = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_h, stream=stream):
        host_call()
    e2e_ms = []
    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 3) + max(3, args.steps // 2)):
            prepare()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph_h.replay()
            b.record(stream)
            b.synchronize()
            if k >= max(args.warmup, 3):
                e2e_ms.append(a.elapsed_time(b))
    if not torch.equal(h_read, readings.cpu()):
        raise RuntimeError("the host-buffer call does not reproduce the device call's readings")
    e2e_max, _ = rank_totals(statistics.mean(e2e_ms), tokens, world, dev)
    e2e = {"value": tokens_all / (e2e_max / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "path": "sdm_write_read_host: pinned host inputs copied in by the call (v on a "
                   "second stream under Phase 1), readings stored into pinned host memory by "
                   "the kernels; graph-replayed, bank reset and L2 flushed outside the events"}

    cpu = None
    if rank == 0 and world == 1:
        cpu = time_oracle(wl, inputs)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "storage_dtype": wl.dtype, "data": "synthetic",
                "config": workload_config(wl, inputs), "roofline": roofline,
                "phase2_roofline": phase2, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_call * args.steps, "clocks": clk,
                "step_ms": {"min": min(step_ms), "median": statistics.median(step_ms),
                            "max": max(step_ms)},
                "wall_s_timed_region": wall1 - wall0, "gpu": torch.cuda.get_device_name(dev)}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_backward(args):
    """Saving forward + backward on one GPU: one step = sdm_write_read_save then
    sdm_write_read_backward (with a zero upstream gradient on the final bank), captured in one
    CUDA graph; the bank is reset and L2 flushed before each step outside the events."""
    import torch

    import sparse_addressed_delta_gb300 as sdm

    wl = si.WORKLOADS[args.workload]
    inputs = si.generate(wl)
    dev = torch.device("cuda", 0)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16

    def tens(name):
        t = torch.from_numpy(np.ascontiguousarray(inputs[name]))
        if wl.dtype == "bf16" and inputs[name].dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(dev)

    d = {k: tens(k) for k in inputs}
    if "grad_readings" not in d:
        d["grad_readings"] = torch.randn((wl.P, wl.T, wl.D), device=dev).to(dt)
    bank0 = d["bank"]
    bank = bank0.clone()
    sq = args.snapshot_quant
    shape = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R, dt,
                           flags=sdm.SNAPSHOT_QUANT[sq])
    ws = sdm.alloc_workspace(shape, dev)
    nb = sdm.backward_workspace_bytes(shape)
    wsb = torch.empty(nb, dtype=torch.uint8, device=dev)
    saved = torch.empty(sdm.saved_bytes(shape), dtype=torch.uint8, device=dev)
    readings = torch.empty((wl.P, wl.T, wl.D), dtype=dt, device=dev)
    gbank = torch.zeros((wl.P * wl.S, wl.D), dtype=torch.float32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    tokens = int(inputs["valid"].sum())
    args_in = (d["write_slots"], d["write_w"], d["log_decay"], d["beta"], d["v"],
               d["read_slots"], d["read_w"], d["valid"])
    # the bank the backward leaves: the initial one, or with a reduced snapshot its written rows
    # rounded (bfloat16 of a float32 bank; float8_e4m3fn, saturating, of either)
    restored = bank0
    if sq == "fp8" or (sq == "bf16" and dt == torch.float32):
        rows = np.unique(np.concatenate([p * wl.S + inputs["write_slots"][p, :int(v)].ravel()
                                         for p, v in enumerate(inputs["valid"])]))
        idx = torch.from_numpy(rows.astype(np.int64)).to(dev)
        restored = bank0.clone()
        if sq == "bf16":
            restored[idx] = bank0[idx].bfloat16().float()
        else:
            restored[idx] = bank0[idx].float().clamp(-448, 448).to(torch.float8_e4m3fn).to(dt)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        sdm.sdm_write_read_save(bank, *args_in, chunk_size=wl.C, workspace=ws, readings=readings,
                                saved=saved, stream=stream, snapshot_quant=sq)
        gbank.zero_()
        sdm.sdm_write_read_backward(bank, *args_in, saved, d["grad_readings"], chunk_size=wl.C,
                                    grad_bank=gbank, workspace=wsb, stream=stream,
                                    snapshot_quant=sq)
    stream.synchronize()
    if not torch.equal(bank, restored):
        raise RuntimeError("backward did not restore the bank")
    def fwd():
        sdm.sdm_write_read_save(bank, *args_in, chunk_size=wl.C, workspace=ws, readings=readings,
                                saved=saved, stream=stream, snapshot_quant=sq)

    def bwd():
        gbank.zero_()
        sdm.sdm_write_read_backward(bank, *args_in, saved, d["grad_readings"], chunk_size=wl.C,
                                    grad_bank=gbank, workspace=wsb, stream=stream,
                                    snapshot_quant=sq)

    gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(gf, stream=stream):
        fwd()
    with torch.cuda.graph(gb, stream=stream):
        bwd()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            bank.copy_(bank0)
            flush.zero_()
            gf.replay()
            gb.replay()
    stream.synchronize()
    clocks = ClockSampler(0)
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            bank.copy_(bank0)
            flush.zero_()
            ev[k][0].record(stream)
            gf.replay()
            ev[k][1].record(stream)
            gb.replay()
            ev[k][2].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if not torch.equal(bank, restored):
        raise RuntimeError("backward did not restore the bank")
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in ev)
    bwd_ms = statistics.mean(b.elapsed_time(c) for _, b, c in ev)
    ms = fwd_ms + bwd_ms
    line = {"metric": "SDM forward+backward tokens/s on 1 GB300", "value": tokens / (ms / 1e3),
            "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "storage_dtype": wl.dtype, "data": "synthetic",
            "config": workload_config(wl, inputs),
            "split_ms": {"saving_forward": fwd_ms, "backward": bwd_ms},
            "snapshot_quant": sq, "saved_bytes": saved.numel(),
            "backward_workspace_bytes": nb, "clocks": clk,
            "gpu": torch.cuda.get_device_name(dev)}
    print(json.dumps(line), flush=True)


def run_for_profiler(args):
    """K eager sdm_write_read calls on the workload, for an external profiler (ncu)."""
    import torch

    import sparse_addressed_delta_gb300 as sdm

    wl = si.WORKLOADS[args.workload]
    inputs = si.generate(wl)
    dev = torch.device("cuda", 0)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16

    def tens(name):
        t = torch.from_numpy(np.ascontiguousarray(inputs[name]))
        if wl.dtype == "bf16" and inputs[name].dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(dev)

    d = {k: tens(k) for k in inputs}
    flags = sdm.FLAG_PER_STEP_KERNELS if args.per_step_kernels else 0
    for _ in range(args.ncu_run):
        sdm.sdm_write_read(d["bank"], d["write_slots"], d["write_w"], d["log_decay"], d["beta"],
                           d["v"], d["read_slots"], d["read_w"], d["valid"], chunk_size=wl.C,
                           flags=flags)
    torch.cuda.synchronize()
    print(f"ncu target: {args.ncu_run} calls of {wl.name} done")


def run_layer_io(args):
    """The layer I/O kernels on the layout of the P=32 = batch 4 x 8 heads workload (T=8192,
    head_dim 128, S=262144 x 128 bf16 bank): head split [4, 8192, 1024] -> [32, 8192, 128] and
    back, bank expand [262144, 128] -> [4, 262144, 128] and the batch sum back. Each op is timed
    with CUDA events over K launches after W warm-ups, L2 flushed (512 MiB write) before each;
    GB/s counts the bytes read and written once."""
    import torch

    import sparse_addressed_delta_gb300 as sdm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B, H, T, CD, S, D = 4, 8, 8192, 128, 262144, 128
    g = torch.Generator(device=dev).manual_seed(5)
    x = torch.randn((B, T, H * CD), device=dev, generator=g).bfloat16()
    y = sdm.head_split(x, H)
    param = torch.randn((S, D), device=dev, generator=g).bfloat16()
    e = sdm.bank_expand(param, B)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    # outputs allocated once: the timed region holds the kernel only (C ABI, current stream)
    lib, bf, st = sdm.library(), sdm.SDM_BF16, sdm._stream_ptr(None)
    o_split, o_merge = torch.empty_like(y), torch.empty_like(x)
    o_exp, o_sum = torch.empty_like(e), torch.empty_like(param)
    P_ = sdm._ptr

    def run(rc):
        if rc != 0:
            raise RuntimeError(lib.sdm_last_error().decode())

    ops = {"head_split": (lambda: run(lib.sdm_head_split(P_(x), P_(o_split), B, T, H, CD, bf, st)),
                          2 * x.numel() * 2),
           "head_merge": (lambda: run(lib.sdm_head_merge(P_(y), P_(o_merge), B, T, H, CD, bf, st)),
                          2 * y.numel() * 2),
           "bank_expand": (lambda: run(lib.sdm_bank_expand(P_(param), P_(o_exp), B, S, D, bf, st)),
                           param.numel() * 2 * (1 + B)),
           "bank_sum": (lambda: run(lib.sdm_bank_sum(P_(e), P_(o_sum), B, S, D, bf, st)),
                        param.numel() * 2 * (B + 1))}
    peak, peak_src = measured_peak()
    res = {}
    clocks = ClockSampler(0)
    for name, (fn, nbytes) in ops.items():
        for _ in range(args.warmup):
            fn()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        res[name] = {"us": 1e3 * ms, "bytes": nbytes, "GB/s": nbytes / ms / 1e6,
                     "frac": nbytes / ms / 1e6 / peak}
    clk = clocks.stop()
    torch.cuda.synchronize()
    if not (torch.equal(o_split, y) and torch.equal(o_merge, x) and torch.equal(o_exp, e)):
        raise RuntimeError("layer I/O outputs differ from the binding's")
    line = {"metric": "SDM layer I/O achieved HBM GB/s (head split/merge, bank expand/sum)",
            "value": statistics.mean(r["GB/s"] for r in res.values()), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "batch 4 x 8 heads, T=8192, head_dim 128; bank 262144 x 128",
                       "l2": "flushed before every launch (512 MiB write)"},
            "peak": peak, "peak_source": peak_src, "ops": res, "clocks": clk,
            "gpu": torch.cuda.get_device_name(dev)}
    print(json.dumps(line), flush=True)


def run_product_key(args):
    """The product-key exact top-k on the GPU: 65536 rows of N(0, 1) scores in bfloat16 and
    float32, k = 256, two factors of 512 (2^18 slots) and four of 32 (2^20 slots). Forward and
    backward are each timed with CUDA events over K launches after W warm-ups, L2 flushed (512
    MiB write) before each; rows/s per case."""
    import torch

    import sparse_addressed_delta_gb300 as sdm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rows, k = 65536, 256
    g = torch.Generator(device=dev).manual_seed(7)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    res = {}
    clocks = ClockSampler(0)
    for dt in (torch.bfloat16, torch.float32):
        for factors in ((512, 512), (32, 32, 32, 32)):
            raw = torch.randn((rows, sum(factors)), device=dev, generator=g).to(dt)
            val, lin = sdm.product_key_topk(raw, factors, k)
            gv = torch.randn(val.shape, device=dev, generator=g).to(dt)

            def timed(fn):
                for _ in range(args.warmup):
                    fn()
                ts = []
                for _ in range(args.steps):
                    flush.zero_()
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record()
                    fn()
                    b.record()
                    b.synchronize()
                    ts.append(a.elapsed_time(b))
                return statistics.median(ts)
            fwd = timed(lambda: sdm.product_key_topk(raw, factors, k))
            bwd = timed(lambda: sdm.product_key_topk_backward(lin, gv, factors, k))
            name = f"{'bf16' if dt == torch.bfloat16 else 'f32'}_F{len(factors)}x{factors[0]}"
            res[name] = {"forward_ms": fwd, "forward_rows_per_s": rows / fwd * 1e3,
                         "backward_ms": bwd, "backward_rows_per_s": rows / bwd * 1e3}
    clk = clocks.stop()
    line = {"metric": "product-key exact top-k rows/s (forward)",
            "value": statistics.mean(r["forward_rows_per_s"] for r in res.values()),
            "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "dtype": "bf16+f32", "data": "synthetic",
            "config": {"workload": f"{rows} rows, k={k}, factors 2 x 512 and 4 x 32",
                       "l2": "flushed before every launch (512 MiB write)"},
            "cases": res, "clocks": clk, "gpu": torch.cuda.get_device_name(dev)}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.product_key:
        run_product_key(args)
        return
    if args.ncu_run:
        run_for_profiler(args)
        return
    if args.backward:
        run_backward(args)
        return
    if args.layer_io:
        run_layer_io(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
