"""The N > 1 host logic of bench.py on CPU: world size 2 over gloo. Each rank
is an independent replica (its own seeded problem); the timing line takes
the max over ranks and the byte total sums over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
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
    import bench
    from bit_quantized_kv_kvq_gb300 import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        mx = bench.reduce_max(1.5 + rank)
        sm = bench.reduce_sum(10.0 * (rank + 1))
        bench.barrier()
        seed = bench.replica_seed(W.LLAMA7B_16K, rank)
        q.put((r, w, lr, mx, sm, seed))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, mx0, sm0, s0), (r1, w1, l1, mx1, sm1, s1) = out
    assert (r0, r1) == (0, 1) and w0 == w1 == 2 and (l0, l1) == (0, 1)
    assert mx0 == mx1 == 2.5          # max over ranks
    assert sm0 == sm1 == 30.0         # bytes of all ranks
    assert s0 != s1                   # independent replicas


def test_single_process_reductions_are_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.reduce_max(3.0) == 3.0 and bench.reduce_sum(4.0) == 4.0
    assert bench.dist_env()[1] >= 1
