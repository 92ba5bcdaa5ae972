"""The multi-rank arithmetic of bench.py on CPU: world_size-2 process groups over gloo.

With N ranks every rank runs its own copy of the workload (its own seed, so the valid-token
counts differ on the ragged workload); the job's throughput is all ranks' tokens over the
slowest rank's time. No kernel runs here: the ranks report made-up times and the token counts
of their own generated inputs.
"""

import multiprocessing as mp
import os
import socket

import pytest

import sdm_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, queue):
    import sys

    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", world_size=world, rank=rank)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        base = si.small(si.WORKLOADS[2], P=3, T=64, S=257)       # ragged valid tokens
        wl = base.replace(seed=base.seed + 1000 * rank)            # the per-rank seed of bench.py
        tokens = int(si.generate(wl)["valid"].sum())
        ms, total = bench.rank_totals(times[rank], tokens, world)
        queue.put((rank, tokens, ms, total))
    finally:
        dist.destroy_process_group()


def _run(world, times):
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, queue))
             for r in range(world)]
    for p in procs:
        p.start()
    out = [queue.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_two_ranks_slowest_time_and_all_tokens():
    out = _run(2, [3.5, 7.25])
    tokens = [t for _, t, _, _ in out]
    assert tokens[0] != tokens[1], "ranks should draw different ragged workloads"
    for rank, _, ms, total in out:
        assert ms == 7.25                       # every rank sees the slowest rank's time
        assert total == sum(tokens)             # and the whole job's tokens


def test_single_rank_passthrough():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.rank_totals(2.0, 123, 1) == (2.0, 123)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import sys

    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.run_reference(bench.parse_args()) is None
    assert capsys.readouterr().out == ""
