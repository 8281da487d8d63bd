"""One workload split across ranks with no exchange (one process per GPU).

Every case of the path is independent per row or per parameter, and the
pages put the work in one global memory with no collective between its
parts (presk PSK-Realize, "Memory placement and collectives"), so a rank
takes a disjoint share and runs it alone:

* a group: a contiguous range of output rows; full-size inputs are read from
  the same rows, row vectors and scalars whole, column vectors [R, 1] from the
  same rows;
* a softmax or norm region: a contiguous range of rows;
* an AdamW tree: a contiguous range of the tree's parameters in leaf order,
  cut into pieces of leaves (AdamW is elementwise, so a piece of a leaf is a
  leaf of its own and updates to the same bits).

The shares of ranks 0..world-1 cover every row and parameter exactly once, in
order.  Pure host arithmetic on sizes; no device work, no torch types.
"""

from __future__ import annotations

# AdamW cut points fall on multiples of this many parameters, so that every
# piece of a leaf keeps the leaf's 16-byte alignment (and the kernel's vector
# path) when the leaf's storage starts on a 256-byte boundary.
PARAM_CUT_QUANTUM = 64


def _check(world: int, rank: int) -> None:
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")


def row_range(rows: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [lo, hi) of rank `rank`: lo = rank * rows // world (balanced to
    within one row, contiguous, in rank order)."""
    _check(world, rank)
    if rows < 0:
        raise ValueError(f"rows {rows}")
    return rows * rank // world, rows * (rank + 1) // world


def param_cut(total: int, world: int, k: int, quantum: int = PARAM_CUT_QUANTUM) -> int:
    """The k-th cut point (0 <= k <= world) of `total` parameters: k * total /
    world rounded down to a multiple of `quantum`; cut 0 is 0, cut `world`
    is total."""
    if k <= 0:
        return 0
    if k >= world:
        return total
    return (total * k // world) // quantum * quantum


def param_pieces(numels, world: int, rank: int, quantum: int = PARAM_CUT_QUANTUM):
    """The pieces of rank `rank`'s parameter range [cut(rank), cut(rank + 1))
    of a tree whose leaves hold `numels` parameters (leaf order): a list of
    (leaf index, lo, hi), element ranges within their leaves, in order; empty
    leaves carry no piece."""
    _check(world, rank)
    numels = [int(n) for n in numels]
    if any(n < 0 for n in numels):
        raise ValueError("negative leaf size")
    total = sum(numels)
    a, b = param_cut(total, world, rank, quantum), param_cut(total, world, rank + 1, quantum)
    out, base = [], 0
    for i, n in enumerate(numels):
        lo, hi = max(a, base), min(b, base + n)
        if hi > lo:
            out.append((i, lo - base, hi - base))
        base += n
    return out
