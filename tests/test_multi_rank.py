"""Multi-rank host logic on CPU with the gloo backend (world size 2): the
ranks run independent shards, then agree on the job time as the max over
ranks, and the job throughput counts every rank's units."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as tmp  # noqa: E402

from structured_state_space_gb300 import multi  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = multi.dist_env()
        assert (r, lr, w) == (rank, rank, world)
        multi.barrier()
        ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
        ms_max = multi.max_over_ranks(ms)
        lo, hi = multi.channel_shard(256, rank, world)
        out.put((rank, ms_max, lo, hi, multi.job_throughput(1000, 4, world, ms_max)))
        multi.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_max_time_and_count_all_units():
    world, port = 2, _free_port()
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [15.0, 15.0]
    assert [(r[2], r[3]) for r in res] == [(0, 128), (128, 256)]
    assert res[0][4] == pytest.approx(1000 * 2 * 4 / 0.015)


def test_channel_shard_covers_everything_once():
    for H in [1, 7, 256, 1023]:
        for world in [1, 2, 3, 8]:
            spans = [multi.channel_shard(H, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == H
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(h - l for l, h in spans) - min(h - l for l, h in spans) <= 1


def test_single_process_passthrough():
    assert multi.max_over_ranks(3.5) == 3.5
    assert multi.job_throughput(10, 2, 1, 1000.0) == 20.0
