"""bench.py's multi-rank logic on CPU (gloo, world size 2): the job's step time
is the slowest rank's, and the CPU-oracle reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = bench.max_over_ranks(10.0 + 5.0 * rank)
        dist.barrier()

        class A:
            workload = "prefill_8k"
            steps = 1
            warmup = 0
        ref = bench.run_reference(A, rank, world) if rank != 0 else "rank0-skipped"
        q.put((rank, mx, ref))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_reference_rank_gating():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {r: (mx, ref) for r, mx, ref in res}
    assert by_rank[0][0] == 15.0 and by_rank[1][0] == 15.0
    assert by_rank[1][1] is None          # non-zero ranks do no reference work


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
