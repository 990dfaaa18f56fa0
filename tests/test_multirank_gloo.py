"""The benchmark's multi-rank plumbing on CPU with two gloo ranks (no GPU needed).

The decode path shards by sequence: every rank runs its own replica and the only
cross-rank steps are the barrier around the timed region and the max / sum of
the per-rank numbers.  These run here as two processes on 127.0.0.1.
"""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    mx = bench.all_max(float(10 + rank), world)
    sm = bench.all_sum(float(1 + rank), world)
    # ranks hold different sequence shards: the per-rank algorithmic bytes add up
    from paged_kv_cache_207_gb300 import workloads as W
    wl = W.make_decode_workload("shard", context_lens=[20 + rank, 700], num_q_heads=8,
                                num_kv_heads=2, head_dim=64, dtype="bf16", seed=rank)
    total = bench.all_sum(float(bench.decode_bytes(wl)), world)
    q.put((rank, mx, sm, total, bench.decode_bytes(wl)))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_and_sum():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [11.0, 11.0]
    assert [r[2] for r in res] == [3.0, 3.0]
    assert res[0][3] == res[1][3] == res[0][4] + res[1][4]
