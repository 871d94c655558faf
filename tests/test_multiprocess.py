"""The multi-GPU path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Under torchrun every rank runs an independent replica of the workload (no data
exchange); the only collectives are the timing barrier and the max over ranks,
which these tests exercise with the gloo backend, plus the rule that only rank 0
runs and prints the reference (oracle) arm."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    from pathlib import Path

    sys.path.insert(0, str(Path(__file__).resolve().parent.parent))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        slowest = bench.max_over_ranks(10.0 * (rank + 1), world)
        # the reference arm: only rank 0 works; the others return at once
        args = type("A", (), {"steps": 1, "warmup": 0, "impl": "reference"})()
        ran = None
        if rank != 0:
            ran = bench.run_reference(args, world, rank)
        out.put((rank, slowest, ran))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {r: (m, ran) for r, m, ran in results}
    assert by_rank[0][0] == pytest.approx(20.0)
    assert by_rank[1][0] == pytest.approx(20.0)
    assert by_rank[1][1] is None


def test_single_rank_helpers_need_no_process_group():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
