"""The N>1 bench path on CPU: two gloo ranks run the rank bookkeeping that
`bench.py --gpus 2` uses under torchrun (replicas only: no collective on the
data path, barrier + max over ranks for timing, rank 0 alone reports)."""
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


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    import torch.distributed as dist

    import bench

    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # each rank's step time differs; every rank must see the slowest one
    t = bench.max_over_ranks(1.0 + 0.25 * rank, w)

    class Args:
        gpus, steps, warmup = world, 1, 0

    # the reference arm runs on rank 0 only: the other ranks return at once
    rc = bench.run_reference(Args, w, r) if r != 0 else 0
    bench.barrier(w)
    dist.destroy_process_group()
    out.put((rank, t, rc))


def test_two_gloo_ranks_time_by_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    if any(c is None for c in codes):
        for p in procs:
            p.kill()
        pytest.fail("gloo ranks did not finish")
    assert codes == [0, 0]
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert got == [(0, 1.25, 0), (1, 1.25, 0)]
