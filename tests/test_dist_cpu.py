"""The benchmark's multi-replica host logic on CPU: two gloo ranks, max time and summed bytes.

The path shards as independent replicas (each GPU owns its own sequences' states and a
full copy of the weights), so ranks exchange only the timing reduction.
"""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr = bench.dist_setup()
    t, b = bench.reduce_over_ranks(0.5 + rank, 1000 * (rank + 1), w)
    bench.barrier(w)
    q.put((rank, w, r, lr, t, b))
    dist.destroy_process_group()


def test_two_rank_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, w, r, lr, t, b in results:
        assert (w, r, lr) == (2, rank, rank)
        assert t == 1.5 and b == 3000.0


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_over_ranks(0.25, 42, 1) == (0.25, 42)


def test_byte_accounting():
    import bench
    b = bench.layer_bytes(64, 200)
    # expert weights dominate: (U + shared) x 3 matrices x 2048 x 7168 x 2 bytes
    assert b["experts"] > 201 * 3 * 2048 * 7168 * 2
    assert bench.kda_bytes(1, o_bytes=4) == 32 * 132868
    s = bench.spec_bytes(16, 4, [0] * 16)
    assert s["replay"] == 0 and s["verify"] > 16 * 32 * 4 * 128 * 128
