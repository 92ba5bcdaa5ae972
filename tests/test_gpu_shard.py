"""Sharding by streams: the path's unit of work is a stream (its own bank rows, its own chunk
steps), so P streams split over ranks, each rank calling sdm_write_read on its streams and
their bank rows, must give the single call's readings and final bank bit for bit. Two ranks in
two processes on one GPU (their kernels never wait on each other; the results are gathered on
the host over gloo)."""

import os
import socket

import pytest
import torch

pytestmark = pytest.mark.gpu

WL = dict(P=6, T=300, C=64, S=2048, D=128, W=16, R=16, dtype="bf16", slots="zipf1.1",
          ragged=True, seed=61)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out: str):
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    sys.path[:0] = [here, os.path.dirname(here)]
    import torch.distributed as dist

    import sdm_inputs as si
    from sdm_case import run_gpu, small_workload, to_device

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    torch.cuda.set_device(0)
    wl = small_workload(**WL)
    inputs = si.generate(wl)
    lo, hi = rank * wl.P // world, (rank + 1) * wl.P // world
    part = {k: v[lo:hi] for k, v in inputs.items() if k != "bank"}
    part["bank"] = inputs["bank"][lo * wl.S:hi * wl.S]
    sub = wl.replace(P=hi - lo)
    r, b, _ = run_gpu(sub, to_device(part, sub))
    rs = [None] * world
    bs = [None] * world
    dist.all_gather_object(rs, r.view(torch.int16).cpu())
    dist.all_gather_object(bs, b.view(torch.int16).cpu())
    if rank == 0:
        r_all, b_all, _ = run_gpu(wl, to_device(inputs, wl))
        same = (torch.equal(torch.cat(rs), r_all.view(torch.int16).cpu()) and
                torch.equal(torch.cat(bs), b_all.view(torch.int16).cpu()))
        with open(out, "w") as f:
            f.write("same" if same else "differ")
    dist.barrier()
    dist.destroy_process_group()


def test_streams_split_over_two_ranks_bitwise(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import torch.multiprocessing as mp

    out = str(tmp_path / "result.txt")
    mp.start_processes(_rank, args=(2, _free_port(), out), nprocs=2, join=True,
                       start_method="spawn")
    assert open(out).read() == "same"
