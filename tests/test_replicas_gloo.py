"""The multi-GPU path is independent replicas (rows never exchange data); what crosses ranks
is only the timing: every rank times its own steps, the job takes the slowest rank's time,
and the whole-job throughput is all ranks' tokens over that time.  Two gloo ranks on the CPU
run bench.py's reduction and throughput functions, and the reference arm's rank rule (rank 0
alone works)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [0.25, 0.40][rank]  # each replica's own timed seconds
    slow = bench.slowest_over_ranks(mine, dist)
    value = bench.replicas_throughput(8, 128, world, slow)

    class Args:
        workload, layers, steps, reference_budget = "7b-bf16-b8", None, 1, 1.0
    ref = bench.reference_arm(Args, rank) if rank != 0 else "skipped"
    out.put((rank, slow, value, ref))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slow, value, ref in got:
        assert slow == pytest.approx(0.40)           # the max over ranks, on every rank
        assert value == pytest.approx(8 * 128 * 2 / 0.40)
    assert got[1][3] is None                         # the reference arm runs on rank 0 only


def test_single_process_is_the_plain_value():
    import bench
    assert bench.slowest_over_ranks(0.3) == pytest.approx(0.3)
    assert bench.replicas_throughput(4, 10, 1, 2.0) == pytest.approx(20.0)
