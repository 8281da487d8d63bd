"""The clipped AdamW step over a parameter tree split across ranks (one
process per GPU).

Everything of the step is elementwise except the global norm of clipping
(presk "The language", The optimizer: g scaled by min(1, c / (||g||_2 +
1e-6))).  Its declared f32 tree -- blocks of 1024 elements, groups of 64
blocks, a leaf's groups, the leaves, each in order -- makes the group sums
the unit to exchange: with the tree cut on group boundaries
(shard.clip_pieces), each rank computes its pieces' group sums on its GPU,
the ranks all-gather them (the one collective), and every rank then forms
the same ||g||^2 and scale as the one-process step and updates its pieces:
the bits of a one-process clipped step, on every world size.
"""

from __future__ import annotations

from . import ops as O
from . import shard as S


def adamw_tree_clipped(pieces, numels, world: int, rank: int, hp, grad_clip: float, workspace, kind="constant",
                       warmup=0, total=1, group=None, stream=None):
    """One clipped step of this rank's share of a tree.

    pieces: this rank's leaves as (theta, m, v, grad) device tensors, the
    element ranges shard.clip_pieces(numels, world, rank) names, in order;
    numels: the whole tree's leaf sizes; workspace: a device tensor of at
    least psk_adamw_workspace(pieces, grad_clip=grad_clip) bytes; group: the
    torch.distributed process group of the ranks (None: the default one).
    Returns the clip scale (a one-element device tensor)."""
    import torch
    import torch.distributed as dist

    counts = [S.clip_piece_groups(numels, world, r) for r in range(world)]
    dev = workspace.device
    width = max(1, max(counts))
    local = torch.zeros(width, dtype=torch.float32, device=dev)
    if counts[rank]:
        O.psk_adamw_group_sqsums(pieces, local[:counts[rank]], workspace, stream)
    if world > 1:
        parts = [torch.empty_like(local) for _ in range(world)]
        dist.all_gather(parts, local, group=group)
    else:
        parts = [local]
    sums = torch.cat([p[:c] for p, c in zip(parts, counts)])
    scale = torch.empty(1, dtype=torch.float32, device=dev)
    O.psk_adamw_clip_scale(sums, S.groups_per_leaf(numels), grad_clip, scale, stream)
    O.psk_adamw_tree_scaled(pieces, hp, scale, kind, warmup, total, stream)
    return scale
