"""Splitting one workload across ranks (reduction_groups_gb300.shard): the
shares cover every row and parameter exactly once, and, over two gloo ranks
on CPU, the oracle run on each rank's share, gathered in rank order, gives
the one-rank result bit for bit (the cases are independent per row and per
parameter: nothing is exchanged).  The clipped AdamW step exchanges the
group sums of its squared-norm tree: the tree cut on group boundaries, the
sums gathered, the norm, scale and updates are the one-rank step's."""

import os
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from reduction_groups_gb300 import shard as S
from synth import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("rows", [0, 1, 7, 37, 8192, 32768, 32771])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_row_ranges_cover_every_row_once(rows, world):
    seen = np.zeros(rows, dtype=np.int64)
    prev = 0
    for r in range(world):
        lo, hi = S.row_range(rows, world, r)
        assert lo == prev and hi >= lo and hi - lo in (rows // world, rows // world + 1)
        seen[lo:hi] += 1
        prev = hi
    assert prev == rows and (seen == 1).all()


@pytest.mark.parametrize("tree", ["gpt", "llama", "ragged"])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_param_pieces_cover_every_parameter_once(tree, world):
    if tree == "gpt":
        numels = W.gpt_adamw_leaves().numels
    elif tree == "llama":
        numels = W.llama_adamw_leaves().numels
    else:
        numels = [5, 0, 130, 1, 64, 0, 1000, 3]
    total = sum(numels)
    starts = np.concatenate([[0], np.cumsum(numels)])
    count = {}
    shares = []
    for r in range(world):
        pieces = S.param_pieces(numels, world, r)
        share = 0
        for i, lo, hi in pieces:
            assert 0 <= lo < hi <= numels[i]
            count[i] = count.get(i, []) + [(lo, hi)]
            share += hi - lo
        # contiguous in the flat order, starting at the rank's cut point
        flat = [(starts[i] + lo, starts[i] + hi) for i, lo, hi in pieces]
        for (a0, a1), (b0, b1) in zip(flat, flat[1:]):
            assert a1 == b0
        if flat:
            assert flat[0][0] == S.param_cut(total, world, r)
            assert S.param_cut(total, world, r) % S.PARAM_CUT_QUANTUM == 0 or r == 0
        shares.append(share)
    assert sum(shares) == total
    for i, n in enumerate(numels):
        got = sorted(count.get(i, []))
        if n == 0:
            assert not got
            continue
        assert got[0][0] == 0 and got[-1][1] == n
        for (a0, a1), (b0, b1) in zip(got, got[1:]):
            assert a1 == b0
    if total >= 64 * world:
        assert max(shares) - min(shares) <= 2 * S.PARAM_CUT_QUANTUM


@pytest.mark.parametrize("tree", ["llama", "ragged", "long"])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_clip_pieces_start_on_group_boundaries_and_cover_once(tree, world):
    if tree == "llama":
        numels = W.llama_adamw_leaves().numels
    elif tree == "ragged":
        numels = [5, 0, 130, 1, 64, 0, 1000, 3]
    else:
        numels = [200_000, 5, 70_000, 131_072, 0, 65_536 * 3 + 7]
    hits = [np.zeros(n, dtype=np.int64) for n in numels]
    groups = 0
    prev_end = 0
    starts = np.concatenate([[0], np.cumsum(numels)])
    for r in range(world):
        pieces = S.clip_pieces(numels, world, r)
        for i, lo, hi in pieces:
            assert lo % S.CLIP_QUANTUM == 0 and 0 <= lo < hi <= numels[i]
            hits[i][lo:hi] += 1
            assert starts[i] + lo == prev_end          # contiguous, in rank order
            prev_end = starts[i] + hi
        groups += S.clip_piece_groups(numels, world, r)
    assert prev_end == sum(numels)
    assert all((h == 1).all() for h in hits)
    assert groups == sum(S.groups_per_leaf(numels))


def test_shares_refuse_a_bad_rank():
    with pytest.raises(ValueError):
        S.row_range(10, 2, 2)
    with pytest.raises(ValueError):
        S.param_pieces([4], 0, 0)


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle.adamw as OA
        import oracle.group as OG
        import oracle.softmax as OS

        # the 64-node group, rows split; the column vector read from the same rows
        R, C = 37, 200
        wl = W.cap_group(R, C)
        (x, _), (row, _), (col, _), (sc, _) = wl.host_inputs()
        lo, hi = S.row_range(R, world, rank)
        gy = OG.evaluate(wl.tokens, wl.imm, [(x[lo:hi], "bf16", (C, 1)), (row, "bf16", (0, 1)),
                                             (col.reshape(-1)[lo:hi], "bf16", (1, 0)), (sc.reshape(1), "bf16", (0, 0))],
                         (hi - lo, C), "bf16")
        # the softmax region, rows split, both orders
        sx = W.softmax_rows(29, 300).host_x()
        a, b = S.row_range(29, world, rank)
        sy = [OS.softmax_region(sx[a:b], "bf16", "bf16", o) for o in (("sequential",), ("interleaved", 8))]
        # the GPT AdamW tree, parameters split into pieces of leaves
        tree = W.gpt_adamw_leaves()
        hl = [tree.host_leaf(i) for i in range(len(tree.leaves))]
        pieces = S.param_pieces(tree.numels, world, rank)
        ay = OA.step_tree([tuple(t[p0:p1] for t in hl[i]) for i, p0, p1 in pieces], tree.grad_dtype, tree.hp)
        # the clipped step on a tree of leaves several groups long: the tree
        # cut on group boundaries, each rank's group sums of ||g||^2 gathered
        # (the one exchange), the scale formed from them, the pieces updated
        rng = np.random.default_rng(5)
        cn = [200_000, 5, 70_000, 131_072, 0, 65_536 * 3 + 7]
        ct = [tuple(rng.standard_normal(n).astype(np.float32) * s_ for s_ in (0.02, 1e-3, 1e-4, 1e-2)) for n in cn]
        ct = [(a, b, np.abs(c), d) for a, b, c, d in ct]
        cp = S.clip_pieces(cn, world, rank)
        cg = np.concatenate([OA.leaf_group_sqsums(ct[i][3][p0:p1], "f32") for i, p0, p1 in cp] or
                            [np.zeros(0, np.float32)])
        parts = [None] * world
        dist.all_gather_object(parts, cg)
        norm = OA.sq_norm_from_groups(np.concatenate(parts), S.groups_per_leaf(cn))
        cscale = OA.clip_scale(norm, 0.5)
        cy = OA.step_tree_scaled([tuple(t[p0:p1] for t in ct[i]) for i, p0, p1 in cp], "f32", tree.hp, cscale)
        mine = {"gy": gy, "sy": sy, "pieces": pieces, "ay": ay, "norm": norm, "cp": cp, "cy": cy}
        every = [None] * world
        dist.all_gather_object(every, mine)
        if rank == 0:
            ok = []
            want = OG.evaluate(wl.tokens, wl.imm, [(x, "bf16", (C, 1)), (row, "bf16", (0, 1)),
                                                   (col.reshape(-1), "bf16", (1, 0)), (sc.reshape(1), "bf16", (0, 0))],
                               (R, C), "bf16")
            ok.append(np.array_equal(np.concatenate([e["gy"] for e in every]), want))
            for k, o in enumerate((("sequential",), ("interleaved", 8))):
                ok.append(np.array_equal(np.concatenate([e["sy"][k] for e in every]),
                                         OS.softmax_region(sx, "bf16", "bf16", o)))
            whole = OA.step_tree(hl, tree.grad_dtype, tree.hp)
            got = [[np.zeros_like(t) for t in w] for w in whole]
            hits = [np.zeros(n, dtype=np.int64) for n in tree.numels]
            for e in every:
                for (i, p0, p1), res in zip(e["pieces"], e["ay"]):
                    hits[i][p0:p1] += 1
                    for j in range(3):
                        got[i][j][p0:p1] = res[j]
            ok.append(all((h == 1).all() for h in hits))
            ok.append(all(np.array_equal(g.view(np.uint32), w_.view(np.uint32))
                          for gl, wl_ in zip(got, whole) for g, w_ in zip(gl, wl_)))
            # the sharded clipped step: the same norm on every rank, equal to
            # the one-rank norm, and the pieces' updates the one-rank step's
            want_norm = OA.grad_sq_norm([t[3] for t in ct], "f32")
            ok.append(all(e["norm"].view(np.uint32) == want_norm.view(np.uint32) for e in every))
            cwhole, _ = OA.step_tree_scheduled(ct, "f32", tree.hp, grad_clip=0.5)
            cgot = [[np.zeros_like(t) for t in w] for w in cwhole]
            for e in every:
                for (i, p0, p1), res in zip(e["cp"], e["cy"]):
                    for j in range(3):
                        cgot[i][j][p0:p1] = res[j]
            ok.append(all(np.array_equal(g.view(np.uint32), w_.view(np.uint32))
                          for gl, wl_ in zip(cgot, cwhole) for g, w_ in zip(gl, wl_)))
            q.put(ok)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_sharded_oracle_equals_one_rank_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_worker, args=(r, 2, 29631, q)) for r in range(2)]
    for p in ps:
        p.start()
    ok = q.get(timeout=300)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ok == [True] * 7, ok
