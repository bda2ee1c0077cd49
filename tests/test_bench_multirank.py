"""The multi-replica bench path on CPU: two gloo ranks on 127.0.0.1 each time
a different region; both must see the slowest one, and the whole-job
throughput counts every rank's tokens."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [40.0, 55.0][rank]
    got = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    q.put((rank, got, bench.job_tokens_per_s(8192, 20, world, got)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [55.0, 55.0]
    assert res[0][2] == 8192 * 20 * 2 / 0.055


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(12.5, None, None) == 12.5
    assert bench.job_tokens_per_s(8192, 10, 1, 100.0) == 8192 * 10 / 0.1
