"""The multi-GPU path of bench.py on CPU: world_size 2 over gloo. Each rank is
an independent replica; the only collective takes the max of the per-rank
timings, and the whole-job rate divides all replicas' work by the slowest."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 1 is the slow replica on the first timing, rank 0 on the second
        mine = [10.0 + rank, 5.0 - rank, 7.0]
        got = bench.max_over_ranks(mine, torch.device("cpu"))
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import socket

    import torch.multiprocessing as mp
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0] == out[1] == [11.0, 5.0, 7.0]


def test_replica_throughput():
    sys.path.insert(0, ROOT)
    import bench
    # two replicas of 1 TFLOP each, the slower taking 100 ms: 20 TFLOP/s
    assert bench.replica_throughput(1e12, 2, 100.0) == pytest.approx(2e13)
    assert bench.replica_throughput(1e12, 1, 100.0) == pytest.approx(1e13)


def _shard_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    from bitwise_reproducible_fp32_gb300 import inputs, shards
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        g = inputs.shard_grads(nshards=8, n=5003)
        k = 8 // world
        local = torch.from_numpy(np.ascontiguousarray(g[rank * k:(rank + 1) * k]))
        out = shards.ordered_shard_mean(
            local, sum_fn=lambda x, s: torch.from_numpy(oracle.shardsum(x.numpy(), scale=s)))
        q.put((rank, out.numpy().tobytes()))
    finally:
        dist.destroy_process_group()


def test_gathered_shard_sum_gloo_world2():
    # two ranks, four shards each: gathering unreduced in global shard order
    # and summing left to right gives, on every rank, the bits of one device's
    # sum of all eight shards
    import socket

    import numpy as np
    import torch.multiprocessing as mp
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from bitwise_reproducible_fp32_gb300 import inputs
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = oracle.shardsum(inputs.shard_grads(nshards=8, n=5003), scale=1.0 / 8).tobytes()
    assert out[0] == out[1] == want


def test_input_digests_name_the_exact_inputs():
    # the bench's per-workload SHA-256: stable, and changed by a value, the
    # order of the arrays, or their shape
    import hashlib

    import numpy as np

    import bench
    a = np.arange(12, dtype=np.float32).reshape(3, 4)
    b = np.ones(5, np.int32)
    d = bench.input_digests({"w": [a, b]})["w"]
    h = hashlib.sha256()
    h.update(b"<f4(3, 4)")
    h.update(a.tobytes())
    h.update(b"<i4(5,)")
    h.update(b.tobytes())
    assert d == h.hexdigest()
    assert bench.input_digests({"w": [b, a]})["w"] != d
    assert bench.input_digests({"w": [a.reshape(4, 3), b]})["w"] != d
    a2 = a.copy()
    a2[1, 2] = np.nextafter(a2[1, 2], np.float32(np.inf))
    assert bench.input_digests({"w": [a2, b]})["w"] != d
