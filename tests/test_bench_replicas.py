"""The bench's multi-GPU path runs one replica per rank (weak scaling, no data-path
collective): each rank times its own batch, the slowest rank's time is taken, and the
whole-job throughput counts every rank's tokens.  Checked here with two gloo ranks on CPU."""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [40.0, 55.0][rank]                     # rank 1 is the slow one
    mx = bench._max_over_ranks(local_ms, world, "cpu")
    ms, value = bench._aggregate(32768, 10, mx, world)

    class Args:
        warmup, steps = 3, 1
    ref = bench.run_reference(Args, rank, world) if rank == 1 else "skipped"
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, mx, ms, value, ref))


def test_two_replicas_take_the_slowest_rank_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, ms, value, _ in out:
        assert mx == 55.0
        assert ms == pytest.approx(5.5)
        assert value == pytest.approx(2 * 32768 / 5.5e-3)
    assert out[1][4] is None          # the reference arm prints from rank 0 only
