"""Multi-process host logic of bench.py on CPU: two gloo ranks, no GPU.

Each rank runs its own batch of requests (weak scaling, no collective on the data path); the
only collective is the MAX over ranks of the timed region, and the reported value is the steps
of all ranks divided by the slowest rank's time. The reference arm runs on rank 0 only.
"""
import contextlib
import io
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch.distributed as dist

    import bench
    from hierarchical_sparse_attention_index_gb300 import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_local = 1.0 + rank                       # rank 1 is the slower one
        tmax = bench.max_over_ranks(t_local, world, dist)
        value = bench.whole_job_value(10, world, tmax)
        seed = bench.rank_seed(1000, rank)
        lat = synth.latents_bf16(seed, 20, 0, 64)
        gathered = [None] * world
        dist.all_gather_object(gathered, (seed, lat.tobytes()))
        # the reference arm prints on rank 0 only; the other ranks return at once
        buf = io.StringIO()
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                bench.run_reference(None)
        q.put((rank, tmax, value, [g[0] for g in gathered], len({g[1] for g in gathered}), buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_bench_host_logic():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, tmax, value, seeds, distinct, out in res:
        assert tmax == 2.0                          # the slowest rank's time on every rank
        assert value == pytest.approx(10.0)         # 2 ranks x 10 steps / 2 s
        assert seeds[0] != seeds[1]                 # each rank has its own batch
        assert distinct == 2                        # ... and so its own inputs
        if rank == 1:
            assert out == ""


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.whole_job_value(200, 1, 0.5) == 400.0
