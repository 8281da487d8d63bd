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

The clipped AdamW step is the one case with an exchange: the global
||g||^2 (presk "The language", The optimizer) over a declared tree of
blocks of 1024 elements and groups of 64 blocks.  For it the tree is cut on
group boundaries (clip_pieces), so that each rank's group sums are the
one-process step's, and the ranks gather them (reduction_groups_gb300.sharded).
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


# The squared-norm tree of clipping: blocks of SQ_BLOCK elements, groups of
# SQ_GROUP blocks, within each leaf.
SQ_BLOCK = 1024
SQ_GROUP = 64
CLIP_QUANTUM = SQ_BLOCK * SQ_GROUP


def leaf_groups(n: int) -> int:
    """Groups of the squared-norm tree in a leaf (or piece) of n elements."""
    nb = -(-int(n) // SQ_BLOCK)
    return -(-nb // SQ_GROUP)


def groups_per_leaf(numels):
    """Groups of every leaf of the tree, in leaf order (0 for an empty leaf)."""
    return [leaf_groups(n) for n in numels]


def clip_cut(numels, world: int, k: int) -> int:
    """The k-th cut point of the tree's flattened parameters for the sharded
    clipped step: k * total / world moved down to the nearest group boundary
    of the leaf it falls in (a multiple of CLIP_QUANTUM elements from the
    leaf's start, or the leaf's start); cut 0 is 0, cut `world` is total."""
    numels = [int(n) for n in numels]
    total = sum(numels)
    if k <= 0:
        return 0
    if k >= world:
        return total
    t = total * k // world
    base = 0
    for n in numels:
        if t < base + n:
            return base + (t - base) // CLIP_QUANTUM * CLIP_QUANTUM
        base += n
    return total


def clip_pieces(numels, world: int, rank: int):
    """The pieces of rank `rank` for the sharded clipped step: (leaf index,
    lo, hi) element ranges within their leaves, in order, between clip cuts
    rank and rank + 1 -- every piece starts on a group boundary of its leaf
    (lo a multiple of CLIP_QUANTUM), so its group sums are the leaf's."""
    _check(world, rank)
    numels = [int(n) for n in numels]
    if any(n < 0 for n in numels):
        raise ValueError("negative leaf size")
    a, b = clip_cut(numels, world, rank), clip_cut(numels, world, rank + 1)
    out, base = [], 0
    for i, n in enumerate(numels):
        lo, hi = max(a, base), min(b, base + n)
        if hi > lo:
            out.append((i, lo - base, hi - base))
        base += n
    return out


def clip_piece_groups(numels, world: int, rank: int) -> int:
    """Group sums rank `rank` contributes: the groups of its clip pieces."""
    return sum(leaf_groups(hi - lo) for _, lo, hi in clip_pieces(numels, world, rank))
