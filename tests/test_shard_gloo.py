"""Host-side sharding across ranks, checked with world_size-2 gloo process groups.

Add, SAXPY, ReLU and copy split into independent contiguous slices, so the
only cross-rank traffic is host bookkeeping: the union of the slices and the
max-over-ranks step time that the benchmark reports.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from memory_bound_elementwise_gb300.shard import shard_range, weak_scaling_range


@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("n", [0, 1, 7, 8, 1000, (1 << 20) + 3])
@pytest.mark.parametrize("align", [1, 8, 16])
def test_shard_range_partitions(n, world, align):
    spans = [shard_range(n, r, world, align) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == n
    for (lo, hi), (lo2, _) in zip(spans, spans[1:]):
        assert hi == lo2
    for r, (lo, hi) in enumerate(spans):
        assert lo <= hi
        assert lo % align == 0
        if r < world - 1:
            assert hi % align == 0
    sizes = [hi - lo for lo, hi in spans]
    assert max(sizes) - min(sizes) <= 2 * align


def test_shard_range_rejects_bad_args():
    with pytest.raises(ValueError):
        shard_range(10, 2, 2)
    with pytest.raises(ValueError):
        shard_range(-1, 0, 1)
    with pytest.raises(ValueError):
        shard_range(10, 0, 1, align=0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, n, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lo, hi = shard_range(n, rank, world, align=8)
        # each rank computes its slice of c = a + b independently (CPU stand-in)
        a = torch.arange(n, dtype=torch.float32)
        b = torch.full((n,), 0.5)
        part = a[lo:hi] + b[lo:hi]
        counts = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(counts, torch.tensor([hi - lo]))
        # the benchmark's timing rule: every rank reports, the max is kept
        t = torch.tensor([1.0 + rank])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        wlo, whi = weak_scaling_range(n, rank)
        q.put((rank, lo, hi, float(part.sum()), [int(c) for c in counts], float(t), wlo, whi))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_slices_and_max_time():
    world, n = 2, 1001
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, lo0, hi0, s0, c0, t0, w0lo, w0hi), (r1, lo1, hi1, s1, c1, t1, w1lo, w1hi) = res
    assert (lo0, hi1) == (0, n) and hi0 == lo1
    assert c0 == c1 == [hi0 - lo0, hi1 - lo1]
    assert s0 + s1 == pytest.approx(float(torch.arange(n, dtype=torch.float64).sum() + 0.5 * n))
    assert t0 == t1 == 2.0
    assert (w0lo, w0hi, w1lo, w1hi) == (0, n, n, 2 * n)
