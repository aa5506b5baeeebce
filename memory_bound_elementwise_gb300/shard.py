"""Host-side partitioning of an elementwise problem across ranks.

Each output element depends only on the same index of the inputs
("逐元素操作算子" §一.1, data parallelism), so add, SAXPY, ReLU and copy split
into contiguous slices with no exchange between ranks.  Slice boundaries are
rounded to ``align`` elements so that every rank's slice starts on the same
vector alignment as the whole array.  The strided gather reads the whole input
for any output slice and is therefore not split here.
"""


def shard_range(n: int, rank: int, world: int, align: int = 1):
    """Return [lo, hi) of the slice of ``n`` elements owned by ``rank``.

    Slices are contiguous, disjoint, cover [0, n) and differ in size by at most
    ``align`` elements (the last rank takes the ragged remainder).
    """
    if world <= 0 or not (0 <= rank < world):
        raise ValueError("bad rank/world: %r/%r" % (rank, world))
    if n < 0 or align <= 0:
        raise ValueError("bad n/align: %r/%r" % (n, align))
    units = n // align              # whole aligned units
    base, extra = divmod(units, world)
    lo_u = rank * base + min(rank, extra)
    hi_u = lo_u + base + (1 if rank < extra else 0)
    lo = lo_u * align
    hi = hi_u * align if rank < world - 1 else n
    return lo, hi


def weak_scaling_range(n_per_rank: int, rank: int):
    """Weak scaling: rank r owns [r*n, (r+1)*n) of a problem of world*n."""
    return rank * n_per_rank, (rank + 1) * n_per_rank
