"""Expert-parallel partition of one MoE layer (host logic only).

Under expert parallelism every GPU holds a contiguous range of experts
(``expert_begin`` / ``expert_end`` of the layer config), receives the whole verify
block and the router, computes the contribution of its own experts to y, and one
all-reduce (sum) of y [T, H] combines the ranks (the deployment sections of
"MiMo x TileRT" and 万亿参数推理为什么特别难: experts spread over GPUs, a long tail
of cold experts).  The cost of a rank is the bytes its experts stream, not their
number, so the ranges below balance a per-expert cost (for example the expected
touched bytes: routing frequency x expert bytes).
"""
from __future__ import annotations

from typing import Sequence


def expert_ranges(num_experts: int, world_size: int, cost: Sequence[float] | None = None) -> list[tuple[int, int]]:
    """Contiguous ranges [begin, end) of experts, one per rank, covering 0..num_experts
    in order, that minimise the largest summed cost of a range (uniform cost when
    ``cost`` is None).  A rank may get an empty range when there are more ranks than
    experts.  Exact: a binary search over the bound, each bound checked by the greedy
    fill (the greedy fill is optimal for a fixed bound on contiguous ranges)."""
    if num_experts < 0 or world_size < 1:
        raise ValueError("num_experts >= 0 and world_size >= 1")
    c = [1.0] * num_experts if cost is None else [float(v) for v in cost]
    if len(c) != num_experts or any(v < 0 for v in c):
        raise ValueError("cost: one non-negative value per expert")

    def fill(bound: float) -> list[tuple[int, int]] | None:
        lim = bound + 1e-9 * max(1.0, bound)   # the sums below may round differently from the prefix sums
        out, b, acc = [], 0, 0.0
        for e, v in enumerate(c):
            if v > lim:
                return None
            if acc + v > lim:
                out.append((b, e))
                b, acc = e, 0.0
            acc += v
        out.append((b, num_experts))
        if len(out) > world_size:
            return None
        return out + [(num_experts, num_experts)] * (world_size - len(out))

    # candidate bounds are sums of contiguous runs; search over them exactly
    prefix = [0.0]
    for v in c:
        prefix.append(prefix[-1] + v)
    cands = sorted({prefix[j] - prefix[i] for i in range(num_experts + 1) for j in range(i, num_experts + 1)})
    lo, hi = 0, len(cands) - 1
    while lo < hi:
        mid = (lo + hi) // 2
        if fill(cands[mid]) is not None:
            hi = mid
        else:
            lo = mid + 1
    ranges = fill(cands[lo])
    assert ranges is not None
    return ranges
