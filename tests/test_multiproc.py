"""The benchmark's multi-rank host logic on CPU: two gloo ranks, no GPU.

The decode path has no exchange step, so ranks run independent replicas; what
needs checking is the plumbing around them: process-group set-up from the
torchrun environment, the barrier, the max-over-ranks timing and the
whole-job aggregation, and that per-rank shards of a batch recombine into the
single-process result.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import oracle
    from paged_kv_cache_04_gb300 import workloads
    r, w, local = bench.dist_init(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # each rank "times" a different amount; everyone must see the slowest
    slowest = bench.max_over_ranks(10.0 + rank, w, torch.device("cpu"))
    # shard a batch by sequence, run the oracle on this rank's shard
    wl = workloads.tiny()
    mine = [s for s in range(wl.S) if s % w == r]
    out = oracle.decode(wl.q[mine], wl.k_cache, wl.v_cache, wl.block_tables[mine],
                        wl.context_lens[mine], wl.scale)
    import torch.distributed as dist
    gathered = [None] * w
    dist.all_gather_object(gathered, (mine, out))
    q.put((rank, slowest, gathered if rank == 0 else None))
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    assert [r[1] for r in results] == [11.0, 11.0]
    gathered = results[0][2]
    sys.path.insert(0, ROOT)
    import oracle
    from paged_kv_cache_04_gb300 import workloads
    wl = workloads.tiny()
    full = oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    combined = np.zeros_like(full)
    for seqs, out in gathered:
        combined[seqs] = out
    assert np.array_equal(combined, full)


def test_weak_scaling_aggregate():
    """value = ranks x bytes per rank / slowest rank's time."""
    world, per_rank_bytes, ms = 4, 2.4e9, 0.5
    value = world * per_rank_bytes / (ms * 1e-3) / 1e9
    assert value == pytest.approx(19200.0)
