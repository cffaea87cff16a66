"""Row sharding of a packed weight matrix across ranks.

Output rows are independent units (DBHOO-CIM article, pwwt.cn/news/4452170, §4.3: split by output channel,
no write conflicts), so a product over N rows shards into contiguous row ranges with no exchange step; a
consumer that needs the whole output gathers the N * 4 output bytes once. Packed rows are contiguous, so a
shard is a contiguous byte range of the packed array (and of the INT4 scale array).
"""
from __future__ import annotations


def row_range(N: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous, balanced [r0, r1) row range of `rank` (sizes differ by at most one row)."""
    if world < 1 or not 0 <= rank < world or N < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(N, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def shard_packed(packed, group_scales, N: int, world: int, rank: int):
    """Views of this rank's rows of a packed matrix ([N, row_stride] bytes) and its scales (or None)."""
    r0, r1 = row_range(N, world, rank)
    return packed[r0:r1], (None if group_scales is None else group_scales[r0:r1]), r0, r1
