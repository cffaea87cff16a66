"""Multi-process host logic on CPU (gloo, world size 2): row sharding of a packed matrix reproduces the
single-process product after one all-gather, and the benchmark's max-over-ranks timing reduction."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_weight_quantized_qpack_gb300.shard import row_range


def test_row_range_balanced_and_covering():
    for N in (0, 1, 7, 4096, 11008):
        for world in (1, 2, 3, 8):
            ranges = [row_range(N, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == N
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        row_range(4, 2, 2)


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from bit_weight_quantized_qpack_gb300.shard import shard_packed
    N, K = 37, 512
    rng = np.random.default_rng(5)
    W = rng.laplace(0, 0.02, (N, K)).astype(np.float32)
    x = rng.standard_normal(K).astype(np.float16).view(np.uint16)
    packed, gs, _ = oracle.quantize_pack(oracle.Q5S, W)
    p, g, r0, r1 = shard_packed(packed, gs, N, world, rank)
    y_local = oracle.gemv(oracle.Q5S, r1 - r0, K, np.ascontiguousarray(p), g, x)
    # gather variable-size shards: pad to the largest shard
    size = torch.tensor([r1 - r0])
    sizes = [torch.zeros(1, dtype=torch.long) for _ in range(world)]
    dist.all_gather(sizes, size)
    mx = int(max(s.item() for s in sizes))
    buf = torch.zeros(mx, dtype=torch.float64)
    buf[: r1 - r0] = torch.from_numpy(y_local)
    parts = [torch.zeros(mx, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(parts, buf)
    y = torch.cat([parts[i][: int(sizes[i].item())] for i in range(world)]).numpy()
    # max-over-ranks timing, as bench.py does
    t = torch.tensor([0.5 + rank], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        full = oracle.gemv(oracle.Q5S, N, K, packed, gs, x)
        out.put((bool(np.array_equal(y, full)), float(t.item())))
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_gemv_matches_single_process():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok, tmax = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
    assert ok and tmax == 1.5
    assert all(p.exitcode == 0 for p in procs)
