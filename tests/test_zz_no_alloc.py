"""psk_adamw_tree_static (clipping scratch in the library's fixed device
buffer, for callers that cannot hand the library device memory) against
psk_adamw_tree_ex (scratch in a caller workspace): two calls in a row on
copies of one tree give the same bits after each call, and once the first
call has set up the buffer's address, further calls leave the device's free
memory unchanged.  The file sorts last so it also runs after every other GPU
test in one process; it passes alone as well."""

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import reduction_groups_gb300 as R

    return R


def _copy(leaves):
    return [tuple(t.clone() for t in leaf) for leaf in leaves]


def _same(a, b):
    return all(torch.equal(x.view(torch.int32), y.view(torch.int32)) for la, lb in zip(a, b) for x, y in
               zip(la[:3], lb[:3]))


@pytest.mark.parametrize("layers,clip", [(1, 1.0), (1, 1e-3), (0, 0.0)])
def test_static_scratch_equals_caller_workspace_twice(dev, layers, clip):
    tree = W.llama_adamw_leaves(layers=layers) if layers else W.gpt_adamw_leaves()
    base = [tree.device_leaf(i) for i in range(len(tree.leaves))]
    a, b = _copy(base), _copy(base)
    ws = torch.empty(max(16, dev.psk_adamw_workspace(a, "cosine", 10, 500, clip)), dtype=torch.uint8, device="cuda")
    for step in (1, 2):
        hp = W.AdamWHyper(lr=tree.hp.lr, beta1=tree.hp.beta1, beta2=tree.hp.beta2, eps=tree.hp.eps,
                          weight_decay=tree.hp.weight_decay, t=tree.hp.t + step)
        dev.psk_adamw_tree_ex(a, hp, "cosine", 10, 500, clip, ws)
        dev.psk_adamw_tree_static(b, hp, "cosine", 10, 500, clip)
        torch.cuda.synchronize()
        assert _same(a, b), f"call {step}"
    assert not _same(a, base)                      # the steps did update the tree


def test_static_scratch_on_a_side_stream(dev):
    tree = W.gpt_adamw_leaves()
    base = [tree.device_leaf(i) for i in range(len(tree.leaves))]
    a, b = _copy(base), _copy(base)
    ws = torch.empty(max(16, dev.psk_adamw_workspace(a, grad_clip=0.05)), dtype=torch.uint8, device="cuda")
    dev.psk_adamw_tree_ex(a, tree.hp, grad_clip=0.05, workspace=ws)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        dev.psk_adamw_tree_static(b, tree.hp, grad_clip=0.05, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert _same(a, b)


def test_static_calls_take_no_device_memory(dev):
    tree = W.llama_adamw_leaves(layers=1)
    b = [tree.device_leaf(i) for i in range(len(tree.leaves))]
    dev.psk_adamw_tree_static(b, tree.hp, "cosine", 10, 500, 1.0)   # first call: the set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        dev.psk_adamw_tree_static(b, tree.hp, "cosine", 10, 500, 1.0)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
