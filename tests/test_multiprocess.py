"""Multi-rank host logic on the CPU (gloo, world size 2): the bench's max-over-ranks timing and weak-scaling
aggregation, and detection of a rank that fails between steps (the survivor's next collective ends with an
error after a short process-group timeout instead of waiting forever)."""
import datetime
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port, timeout_s=30):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=timeout_s))
    return dist


def _agg_worker(rank, world, port, q):
    import bench
    dist = _init(rank, world, port)
    ms = [1.5, 2.5][rank]                      # rank 1 is the slow one
    got = bench.max_over_ranks(ms, world, "cpu")
    tokens = 4096
    q.put((rank, got, world * tokens / (got * 1e-3)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_agg_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [2.5, 2.5]
    assert all(abs(o[2] - 2 * 4096 / 2.5e-3) < 1e-6 for o in out)


def _fail_worker(rank, world, port, q):
    import torch
    dist = _init(rank, world, port, timeout_s=5)
    dist.barrier()                             # step 1 completes on both ranks
    if rank == 1:
        q.put((rank, "left"))
        q.close()
        q.join_thread()                        # the message is out before the process dies
        os._exit(3)                            # dies between steps, with nothing in flight
    try:
        t = torch.ones(1)
        dist.all_reduce(t)                     # step 2: the peer is gone
        q.put((rank, "no error"))
    except Exception as e:                     # noqa: BLE001
        q.put((rank, "detected: " + type(e).__name__))


def test_failed_rank_is_detected_by_the_survivor():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_fail_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    assert out[1] == "left"
    assert out[0].startswith("detected"), out[0]
    assert procs[1].exitcode == 3
