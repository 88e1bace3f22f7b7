"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks (127.0.0.1)
reduce their per-call times to the maximum, draw different batches, and only
rank 0 runs the reference arm."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        vals = bench.reduce_max_over_ranks([1.0 + rank, 10.0 * (world - rank)], device="cpu")
        out.put((rank, vals, bench.rank_seed("mtp_decode", rank)))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_max_and_draw_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    res = dict((r, (v, sd)) for r, v, sd in (q.get(timeout=120) for _ in procs))
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    assert res[0][0] == res[1][0] == [2.0, 20.0]
    assert res[0][1] != res[1][1]


def test_reduce_without_process_group_is_identity():
    import bench
    assert bench.reduce_max_over_ranks([3.0, 4.0], device="cpu") == [3.0, 4.0]


def test_reference_arm_is_silent_on_other_ranks(capsys):
    import bench

    class A:
        workload = "tiny_decode"
        steps = 1
        warmup = 0

    bench.run_reference(A(), world=2, rank=1)
    assert capsys.readouterr().out == ""
