"""Parity of the scheduled, clipped AdamW step (psk_adamw_tree_ex) with the
oracle, bit for bit: the squared-norm tree, the clip scale, the scheduled lr
and every updated parameter."""

import numpy as np
import pytest

import oracle.adamw as OA
from oracle.f32 import bf16_to_f32, f32_to_bf16
from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import reduction_groups_gb300 as R

    return R


def _to_dev(a, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _to_host(t):
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


def _workspace(dev, leaves, **sched):
    n = dev.psk_adamw_workspace(leaves, **sched)
    return torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")


def _check(leaves, want):
    for (th, m, v, g), (wt, wm, wv) in zip(leaves, want):
        assert np.array_equal(_to_host(th).view(np.uint32), wt.view(np.uint32))
        assert np.array_equal(_to_host(m).view(np.uint32), wm.view(np.uint32))
        assert np.array_equal(_to_host(v).view(np.uint32), wv.view(np.uint32))


@pytest.mark.parametrize("kind,w,total", [("cosine", 3, 40), ("linear", 0, 25), ("constant", 0, 1)])
@pytest.mark.parametrize("clip", [0.0, 1e-2, 1e3])
def test_gpt_tree_scheduled_and_clipped_bitwise(dev, kind, w, total, clip):
    """clip 1e-2 scales every gradient (scale < 1), 1e3 leaves them (scale 1)."""
    tree = W.gpt_adamw_leaves()
    host = [tree.host_leaf(i) for i in range(len(tree.leaves))]
    want, scale = OA.step_tree_scheduled(host, tree.grad_dtype, tree.hp, kind, w, total, grad_clip=clip)
    leaves = [tuple(_to_dev(a, tree.grad_dtype if k == 3 else "f32") for k, a in enumerate(h)) for h in host]
    ws = _workspace(dev, leaves, kind=kind, warmup=w, total=total, grad_clip=clip)
    dev.psk_adamw_tree_ex(leaves, tree.hp, kind, w, total, clip, ws)
    torch.cuda.synchronize()
    _check(leaves, want)
    if clip > 0:
        got = ws[:4].cpu().numpy().view(np.float32)[0]
        assert got.view(np.uint32) == np.float32(scale).view(np.uint32)
        assert (scale < 1) == (clip < 1)


def test_ragged_unaligned_bf16_leaves_clipped(dev):
    rng = np.random.default_rng(9)
    hp = W.AdamWHyper(lr=1e-3, t=5)
    sizes = [1, 3, 1023, 1025, 4097, 64 * 1024 + 3, 0, 10007]
    host, leaves, fulls = [], [], []
    for n in sizes:
        # one element before and 64 after each leaf: canaries the step must not touch
        th = (rng.standard_normal(n + 65) * 0.02).astype(np.float32)
        m = (rng.standard_normal(n + 65) * 1e-3).astype(np.float32)
        v = np.abs(rng.standard_normal(n + 65) * 1e-4).astype(np.float32)
        g = f32_to_bf16((rng.standard_normal(n + 65) * 0.3).astype(np.float32))
        host.append((th[1:n + 1], m[1:n + 1], v[1:n + 1], g[1:n + 1]))
        full = tuple(_to_dev(a, "bf16" if k == 3 else "f32") for k, a in enumerate((th, m, v, g)))
        fulls.append((full, (th, m, v)))
        leaves.append(tuple(t[1:n + 1] for t in full))
    want, scale = OA.step_tree_scheduled(host, "bf16", hp, "linear", 2, 9, grad_clip=0.5)
    assert scale < 1
    ws = _workspace(dev, leaves, kind="linear", warmup=2, total=9, grad_clip=0.5)
    dev.psk_adamw_tree_ex(leaves, hp, "linear", 2, 9, 0.5, ws)
    torch.cuda.synchronize()
    _check(leaves, want)
    for (full, orig), n in zip(fulls, sizes):
        for t, o in zip(full[:3], orig):
            h = _to_host(t)
            assert h[0] == o[0] and np.array_equal(h[n + 1:], o[n + 1:]), "a store landed outside a leaf"


def test_two_layer_llama_tree_clipped_sampled(dev):
    """A 2-layer Llama-style tree (~200M parameters, bf16 gradients): the scale
    against the oracle's squared-norm tree over every gradient, and sampled
    parameters against the oracle's step."""
    tree = W.llama_adamw_leaves(layers=2)
    leaves = [tree.device_leaf(i) for i in range(len(tree.leaves))]
    grads = [_to_host(g) for (_, _, _, g) in leaves]
    scale = OA.clip_scale(OA.grad_sq_norm(grads, "bf16"), 1.0)
    rng = np.random.default_rng(12)
    picks, before = [], []
    for (th, m, v, g) in leaves:
        n = th.numel()
        idx = np.unique(np.concatenate([np.arange(min(n, 4)), np.arange(max(0, n - 4), n),
                                        rng.integers(0, n, min(n, 8192))]))
        it = torch.from_numpy(idx).cuda()
        picks.append(it)
        before.append(tuple(_to_host(a[it]) for a in (th, m, v, g)))
    h = OA.hyper_f32(tree.hp.lr, tree.hp.beta1, tree.hp.beta2, tree.hp.eps, tree.hp.weight_decay, tree.hp.t)
    h["lr"] = OA.lr_scheduled(tree.hp.lr, "cosine", 100, 5000, tree.hp.t)
    ws = _workspace(dev, leaves, kind="cosine", warmup=100, total=5000, grad_clip=1.0)
    dev.psk_adamw_tree_ex(leaves, tree.hp, "cosine", 100, 5000, 1.0, ws)
    torch.cuda.synchronize()
    assert ws[:4].cpu().numpy().view(np.float32)[0].view(np.uint32) == scale.view(np.uint32)
    for (th, m, v, g), it, (bt, bm, bv, bg) in zip(leaves, picks, before):
        gs = (bf16_to_f32(bg) * scale).astype(np.float32)
        wt, wm, wv = OA.step_leaf(bt, bm, bv, gs, "f32", h)
        assert np.array_equal(_to_host(th[it]).view(np.uint32), wt.view(np.uint32))
        assert np.array_equal(_to_host(m[it]).view(np.uint32), wm.view(np.uint32))
        assert np.array_equal(_to_host(v[it]).view(np.uint32), wv.view(np.uint32))


def test_clip_needs_a_workspace(dev):
    leaves = [tuple(torch.zeros(100, device="cuda") for _ in range(4))]
    hp = W.AdamWHyper(t=1)
    with pytest.raises(dev.PskError) as e:
        dev.psk_adamw_tree_ex(leaves, hp, grad_clip=1.0)
    assert e.value.name == "PSK_E_NULL"
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(dev.PskError) as e:
        dev.psk_adamw_tree_ex(leaves, hp, grad_clip=1.0, workspace=small)
    assert e.value.name == "PSK_E_ARG"


def test_mixed_bf16_and_f32_leaves_at_rest(dev):
    """Leaves stored in bf16 at rest next to f32 ones, clipped and scheduled,
    aligned and not: every output against the oracle, bit for bit."""
    rng = np.random.default_rng(61)
    hp = W.AdamWHyper(lr=1e-3, t=9)
    specs = [(4096, "bf16", "bf16"), (10007, "bf16", "f32"), (4096, "f32", "bf16"), (3, "bf16", "bf16"),
             (70000, "bf16", "bf16"), (513, "f32", "f32")]
    host, leaves, pdts = [], [], []
    for n, pdt, gdt in specs:
        th = (rng.standard_normal(n + 1) * 0.02).astype(np.float32)
        m = (rng.standard_normal(n + 1) * 1e-3).astype(np.float32)
        v = np.abs(rng.standard_normal(n + 1) * 1e-4).astype(np.float32)
        g = (rng.standard_normal(n + 1) * 0.1).astype(np.float32)
        arrs = [f32_to_bf16(a) if pdt == "bf16" else a for a in (th, m, v)] + [f32_to_bf16(g) if gdt == "bf16" else g]
        off = 1 if n % 2 else 0                        # odd sizes: unaligned views
        host.append(tuple(a[off:off + n] for a in arrs))
        leaves.append(tuple(_to_dev(a, pdt if k < 3 else gdt)[off:off + n] for k, a in enumerate(arrs)))
        pdts.append((pdt, gdt))
    h = OA.hyper_f32(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.t)
    h["lr"] = OA.lr_scheduled(hp.lr, "linear", 2, 30, hp.t)
    widened = [OA.widen(np.asarray(g), gdt) for (_, _, _, g), (_, gdt) in zip(host, pdts)]
    scale = OA.clip_scale(OA.grad_sq_norm(widened, "f32"), 0.5)
    ws = torch.empty(max(16, dev.psk_adamw_workspace(leaves, "linear", 2, 30, 0.5)), dtype=torch.uint8, device="cuda")
    dev.psk_adamw_tree_ex(leaves, hp, "linear", 2, 30, 0.5, ws)
    torch.cuda.synchronize()
    for (th, m, v, g), (pdt, gdt), (bt, bm, bv, bg), gw in zip(leaves, pdts, host, widened):
        want = OA.step_leaf(bt, bm, bv, (gw * scale).astype(np.float32), "f32", h, param_dtype=pdt)
        for got_t, w in zip((th, m, v), want):
            got = _to_host(got_t)
            assert np.array_equal(got.view(np.uint16 if pdt == "bf16" else np.uint32),
                                  w.view(np.uint16 if pdt == "bf16" else np.uint32))


def test_clip_norm_over_mixed_gradient_types_in_one_warp(dev):
    """Leaves of whole 1024-element blocks whose gradients alternate f32 and
    bf16, so the squared-norm pass's warp-cooperative loads mix both types and
    several leaves in one warp, plus a ragged leaf (the per-lane path): the
    clip scale and every updated parameter bit for bit."""
    rng = np.random.default_rng(21)
    hp = W.AdamWHyper(lr=2e-3, t=7)
    sizes = [1024, 3072, 2048, 1024, 32 * 1024, 5 * 1024, 1024 * 40, 777, 4096]
    host, leaves, gf32 = [], [], []
    for i, n in enumerate(sizes):
        gdt = "bf16" if i % 2 else "f32"
        th = (rng.standard_normal(n) * 0.02).astype(np.float32)
        m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        v = np.abs(rng.standard_normal(n) * 1e-4).astype(np.float32)
        g32 = (rng.standard_normal(n) * (0.1 + i)).astype(np.float32)
        g = f32_to_bf16(g32) if gdt == "bf16" else g32
        host.append((th, m, v, g, gdt))
        gf32.append(bf16_to_f32(g) if gdt == "bf16" else g)
        leaves.append((_to_dev(th, "f32"), _to_dev(m, "f32"), _to_dev(v, "f32"), _to_dev(g, gdt)))
    scale = OA.clip_scale(OA.grad_sq_norm(gf32, "f32"), 0.25)
    assert scale < 1
    ws = _workspace(dev, leaves, kind="linear", warmup=2, total=20, grad_clip=0.25)
    dev.psk_adamw_tree_ex(leaves, hp, "linear", 2, 20, 0.25, ws)
    torch.cuda.synchronize()
    assert ws[:4].cpu().numpy().view(np.float32)[0].view(np.uint32) == scale.view(np.uint32)
    h = OA.hyper_f32(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.t)
    h["lr"] = OA.lr_scheduled(hp.lr, "linear", 2, 20, hp.t)
    for (th, m, v, g), (bt, bm, bv, bg, gdt), g32 in zip(leaves, host, gf32):
        wt, wm, wv = OA.step_leaf(bt, bm, bv, (g32 * scale).astype(np.float32), "f32", h)
        assert np.array_equal(_to_host(th).view(np.uint32), wt.view(np.uint32))
        assert np.array_equal(_to_host(m).view(np.uint32), wm.view(np.uint32))
        assert np.array_equal(_to_host(v).view(np.uint32), wv.view(np.uint32))


def _clip_tree(seed, numels, grad_dtype):
    rng = np.random.default_rng(seed)
    host = []
    for n in numels:
        th = (rng.standard_normal(n) * 0.02).astype(np.float32)
        m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        v = np.abs(rng.standard_normal(n) * 1e-4).astype(np.float32)
        g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
        host.append((th, m, v, f32_to_bf16(g) if grad_dtype == "bf16" else g))
    return host


@pytest.mark.parametrize("world", [2, 3, 5])
@pytest.mark.parametrize("grad_dtype", ["bf16", "f32"])
def test_sharded_clipped_step_equals_one_call(dev, world, grad_dtype):
    """The clipped step of a tree split into `world` ranks' pieces (cut on
    the squared-norm tree's group boundaries), run rank after rank on one
    GPU: each rank's group sums (psk_adamw_group_sqsums), the sums gathered
    in rank order, the scale from them (psk_adamw_clip_scale), each rank's
    pieces updated with it (psk_adamw_tree_scaled) -- the scale and every
    parameter bit for bit those of one psk_adamw_tree_ex call and of the
    oracle."""
    from reduction_groups_gb300 import shard as S

    numels = [200_000, 5, 70_000, 131_072, 0, 65_536 * 3 + 7, 1000]
    host = _clip_tree(17, numels, grad_dtype)
    hp, clip = W.AdamWHyper(lr=1e-3, t=7), 1e-2
    want, wscale = OA.step_tree_scheduled(host, grad_dtype, hp, "cosine", 2, 30, grad_clip=clip)
    # one call
    one = [tuple(_to_dev(a, grad_dtype if k == 3 else "f32") for k, a in enumerate(h)) for h in host]
    ws = _workspace(dev, one, kind="cosine", warmup=2, total=30, grad_clip=clip)
    dev.psk_adamw_tree_ex(one, hp, "cosine", 2, 30, clip, ws)
    # the ranks
    full = [tuple(_to_dev(a, grad_dtype if k == 3 else "f32") for k, a in enumerate(h)) for h in host]
    shares = [[tuple(t[lo:hi] for t in full[i]) for i, lo, hi in S.clip_pieces(numels, world, r)]
              for r in range(world)]
    sums = []
    for r in range(world):
        n_r = S.clip_piece_groups(numels, world, r)
        gs = torch.empty(max(n_r, 1), dtype=torch.float32, device="cuda")
        if n_r:
            dev.psk_adamw_group_sqsums(shares[r], gs[:n_r], _workspace(dev, shares[r], grad_clip=clip))
        sums.append(gs[:n_r])
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    dev.psk_adamw_clip_scale(torch.cat(sums), S.groups_per_leaf(numels), clip, scale)
    for r in range(world):
        dev.psk_adamw_tree_scaled(shares[r], hp, scale, "cosine", 2, 30)
    torch.cuda.synchronize()
    assert scale.cpu().numpy().view(np.uint32)[0] == np.float32(wscale).view(np.uint32)
    assert ws[:4].cpu().numpy().view(np.uint32)[0] == np.float32(wscale).view(np.uint32)
    _check(full, want)
    _check(one, want)


def test_sharded_clip_through_a_one_rank_process_group(dev):
    """reduction_groups_gb300.sharded.adamw_tree_clipped on a one-rank NCCL
    group (the path's collective with nothing to gather) equals the oracle."""
    import datetime
    import os

    import torch.distributed as dist

    from reduction_groups_gb300 import shard as S
    from reduction_groups_gb300 import sharded as SH

    if not dist.is_nccl_available():
        pytest.skip("no NCCL")
    numels = [70_000, 3, 131_072]
    host = _clip_tree(23, numels, "bf16")
    hp, clip = W.AdamWHyper(lr=1e-3, t=3), 1e-2
    want, wscale = OA.step_tree_scheduled(host, "bf16", hp, grad_clip=clip)
    full = [tuple(_to_dev(a, "bf16" if k == 3 else "f32") for k, a in enumerate(h)) for h in host]
    pieces = [tuple(t[lo:hi] for t in full[i]) for i, lo, hi in S.clip_pieces(numels, 1, 0)]
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ.setdefault("MASTER_PORT", "29677")
    dist.init_process_group("nccl", rank=0, world_size=1, timeout=datetime.timedelta(seconds=120))
    try:
        scale = SH.adamw_tree_clipped(pieces, numels, 1, 0, hp, clip, _workspace(dev, pieces, grad_clip=clip))
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert scale.cpu().numpy().view(np.uint32)[0] == np.float32(wscale).view(np.uint32)
    _check(full, want)


def test_sharded_clip_refusals(dev):
    import ctypes

    from reduction_groups_gb300 import _native as N

    L = N.lib()
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    counts = (ctypes.c_int64 * 1)(1)
    assert L.psk_adamw_clip_scale(None, counts, 1, 1.0, scale.data_ptr(), None) == -5         # no group sums
    assert L.psk_adamw_clip_scale(None, counts, 1, 0.0, scale.data_ptr(), None) == -9         # clip must be > 0
    assert L.psk_adamw_clip_scale(None, counts, 600, 1.0, scale.data_ptr(), None) == -9       # too many leaves
    assert L.psk_adamw_tree_scaled(None, 0, None, None, None, None) == -5                    # no scale
