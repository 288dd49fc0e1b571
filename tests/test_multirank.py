"""Host-side logic of the multi-GPU benchmark path on CPU ranks (gloo, world 2).

The layer shards by tokens with no collective on the data path; the only
cross-rank steps are the barrier and the max over ranks of the timed region.
Each rank must hold a different token shard, and the reduction must return
the slowest rank's time on every rank.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    from synth import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    seed = bench.shard_seed(r)
    h = W.make_h(W.WORKLOADS["tiny"], 8, seed=seed)
    bench.barrier()
    mx = bench.reduce_max(10.0 + 5.0 * r)
    dist.destroy_process_group()
    q.put((r, w, local, seed, int(h[0, 0]), mx))


def test_two_cpu_ranks_shard_tokens_and_take_the_max_time():
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
    (r0, w0, l0, s0, h0, m0), (r1, w1, l1, s1, h1, m1) = res
    assert (r0, r1, w0, w1, l0, l1) == (0, 1, 2, 2, 0, 1)
    assert s0 == 0 and s1 != s0            # rank 0 holds the reference batch
    assert h0 != h1                         # different token shards
    assert m0 == m1 == 15.0                 # max over ranks on every rank


def test_workload_config_names_the_layer():
    import bench
    from synth import workloads as W
    c = bench.workload_config(W.WORKLOADS["mix"], 4096, 2)
    assert c["global_batch"] == 8192 and "mixtral-like" in c["workload"]
    assert "no collective" in c["parallelism"]
    c = bench.workload_config(W.WORKLOADS["cap"], 8192, 2)
    assert "all-gather" in c["parallelism"]   # the capacity exchange


def _skewed_routes(T, N, k, seed):
    # k distinct experts per token, drawn with a skewed preference so that
    # some experts overflow their capacity
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, N + 1) ** 1.2
    p /= p.sum()
    return np.stack([rng.choice(N, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def _exchange_worker(rank, world, port, bounds, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    from invariant_expert_routing_gb300 import shard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    N, k = 8, 2
    idx = _skewed_routes(bounds[-1], N, k, seed=5)
    lo, hi = bounds[rank], bounds[rank + 1]
    load = torch.from_numpy(np.bincount(idx[lo:hi].reshape(-1), minlength=N).astype(np.int32))
    offset, global_tokens = shard.shard_exchange(load, hi - lo)
    dist.destroy_process_group()
    q.put((rank, offset.numpy().tolist(), global_tokens))


def test_shard_exchange_keeps_the_unsharded_capacity_decisions():
    # Three CPU ranks with uneven token shards of one capacity-limited batch:
    # with each rank's exchanged offsets, the keep rule of
    # moe_dispatch_align_shard (a route is kept iff its rank among the
    # shard's routes to its expert is below C - offset) reproduces the
    # oracle's decisions on the whole batch, route for route.
    import oracle
    bounds = [0, 170, 171, 300]   # a one-token shard in the middle
    world = len(bounds) - 1
    N, k, B, cf = 8, 2, 8, 0.6
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_exchange_worker, args=(r, world, port, bounds, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    T = bounds[-1]
    idx = _skewed_routes(T, N, k, seed=5)
    C = oracle.capacity(T, N, k, cf)
    ref = oracle.dispatch(idx, N, B, C)["route_kept"]
    assert 0 < int((ref == 0).sum()) < T * k          # some routes dropped, some kept
    for rank, offset, global_tokens in res:
        assert global_tokens == T
        lo, hi = bounds[rank], bounds[rank + 1]
        assert offset == np.bincount(idx[:lo].reshape(-1), minlength=N).tolist()
        seen = np.zeros(N, np.int64)
        for r, e in enumerate(idx[lo:hi].reshape(-1)):
            keep = seen[e] < max(0, C - offset[e])
            seen[e] += 1
            assert keep == bool(ref[lo * k + r]), (rank, r)
