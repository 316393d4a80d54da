"""The multi-GPU path of bench.py is replicas only: N independent decoders,
one process per GPU, exchanging nothing but their timings and token counts.
This runs that exchange on the CPU with two gloo ranks: the process group
comes up from the launcher's environment, the barrier returns, the whole-job
throughput is every rank's tokens over the slowest rank's time, and only
rank 0 runs the reference arm."""
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
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    # rank r decoded 10 (r + 1) tokens in 100 + 50 r ms
    tokens_all, ms_max, value = bench.aggregate(w, 10 * (rank + 1), 100.0 + 50.0 * rank)
    # the reference arm: rank 0 alone does the work
    class Args:
        workload = "qwen7b"
        warmup = 0
        steps = 0
    ran = bench.run_reference(Args(), w, r) if r != 0 else "rank 0 not run here"
    bench.barrier(w)
    dist.destroy_process_group()
    out.put((rank, tokens_all, ms_max, value, ran))


@pytest.mark.parametrize("world", [2])
def test_two_gloo_replicas(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    tot_tokens = sum(10 * (r + 1) for r in range(world))
    ms_max = 100.0 + 50.0 * (world - 1)
    for rank, tokens_all, mx, value, ran in res:
        assert tokens_all == tot_tokens and mx == ms_max
        assert value == pytest.approx(tot_tokens / (ms_max / 1e3))
        if rank != 0:
            assert ran is None   # the other ranks return without work
