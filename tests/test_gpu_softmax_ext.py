"""Parity of the masked softmax region and the softmax backward (through the
C ABI) with the CPU oracle, bit for bit (exact exp; the fast exp within the
region's stated tolerance)."""

import numpy as np
import pytest

import oracle.softmax as OS
from oracle.f32 import bf16_to_f32, f32_to_bf16
from synth import workloads as W
from tests.guard import guarded

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


def _same(a, b, dtype):
    if dtype == "bf16":
        a = bf16_to_f32(a)
        b = bf16_to_f32(b)
    return (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))


_GUARDS = []


def _empty(shape, dtype):
    """A NaN-poisoned output with canaries around it (checked at teardown)."""
    g = guarded(shape, torch.bfloat16 if dtype == "bf16" else torch.float32)
    _GUARDS.append(g)
    return g.tensor


@pytest.fixture(autouse=True)
def _canaries_intact():
    _GUARDS.clear()
    yield
    torch.cuda.synchronize()
    assert all(g.intact() for g in _GUARDS), "a store landed outside an output"
    _GUARDS.clear()


ORDERS = [("sequential",), ("interleaved", 8), ("interleaved", 3), ("interleaved", 40)]


@pytest.mark.parametrize("order", ORDERS, ids=lambda o: "-".join(map(str, o)))
@pytest.mark.parametrize("shape,xt,full", [((300, 512), "bf16", True), ((300, 512), "bf16", False),
                                           ((2000, 4096), "bf16", True), ((37, 999), "bf16", True),
                                           ((64, 640), "f32", False), ((5, 10000), "bf16", True)])
def test_masked_softmax_bitwise(dev, order, shape, xt, full):
    rows, cols = shape
    wl = W.softmax_rows(rows, cols)
    x = wl.host_x() if xt == "bf16" else bf16_to_f32(wl.host_x())
    rng = np.random.default_rng(rows + cols)
    mask = (rng.random((rows, cols) if full else (cols,)) < 0.7).astype(np.uint8)
    if full:
        mask[1] = 0                                    # a row the mask empties
        mask[2] = 0
        mask[2, cols - 1] = 1                          # one allowed position, the last
        ii = np.arange(min(rows, cols))
        mask[ii[3:], :] = (np.arange(cols)[None, :] <= ii[3:, None]).astype(np.uint8)   # causal rows
    want = OS.softmax_region(x, xt, "bf16", order, mask=mask)
    y = _empty((rows, cols), "bf16")
    dev.psk_softmax_masked(_to_dev(x, xt), y, torch.from_numpy(mask).cuda(), order, "exact")
    torch.cuda.synchronize()
    ok = _same(_to_host(y), want, "bf16")
    assert ok.all(), f"{(~ok).sum()} of {ok.size} differ"
    assert dev.psk_device_status() == 0


def test_masked_softmax_fast_exp_and_bool_mask(dev):
    wl = W.softmax_rows(256, 4096)
    x = wl.host_x()
    rng = np.random.default_rng(6)
    mask = rng.random((256, 4096)) < 0.5
    mask[7] = False
    for order in (("sequential",), ("interleaved", 8)):
        want = OS.softmax_region(x, "bf16", "f32", order, mask=mask)
        y = _empty((256, 4096), "f32")
        dev.psk_softmax_masked(_to_dev(x, "bf16"), y, torch.from_numpy(mask).cuda(), order, "fast")
        torch.cuda.synchronize()
        got = _to_host(y)
        assert np.all(got[~mask] == 0) and np.all(got[7] == 0)
        rel = np.abs(got.astype(np.float64) - want) / np.maximum(np.abs(want), 1e-38)
        assert rel.max() <= 1e-6


def test_masked_softmax_fast_bf16_out_one_mask_row(dev):
    """The fast masked softmax with bf16 outputs and one mask row for every
    row (a mask stride of 0, the benchmark's form): refused positions 0, the
    rest within one bf16 ulp of the oracle; a mask refusing everything gives
    zero rows."""
    wl = W.softmax_rows(300, 4096)
    x = wl.host_x()
    rng = np.random.default_rng(12)
    for keep in (0.7, 0.0):
        mrow = rng.random(4096) < keep
        mask = np.broadcast_to(mrow, (300, 4096))
        for order in (("sequential",), ("interleaved", 8)):
            want = OS.softmax_region(x, "bf16", "bf16", order, mask=np.ascontiguousarray(mask))
            y = _empty((300, 4096), "bf16")
            dev.psk_softmax_masked(_to_dev(x, "bf16"), y, torch.from_numpy(mrow).cuda(), order, "fast")
            torch.cuda.synchronize()
            got = _to_host(y)
            assert np.all(got[:, ~mrow] == 0)
            d = np.abs(got.astype(np.int32) - want.astype(np.int32))
            assert d.max() <= 1, f"keep {keep}, order {order}: {d.max()} bf16 ulp"


@pytest.mark.parametrize("order", ORDERS, ids=lambda o: "-".join(map(str, o)))
@pytest.mark.parametrize("shape,yt,ct_t,dxt", [((300, 512), "bf16", "bf16", "bf16"), ((2000, 4096), "bf16", "bf16", "f32"),
                                               ((64, 640), "f32", "f32", "f32"), ((37, 999), "bf16", "f32", "bf16"),
                                               ((5, 10000), "f32", "bf16", "f32"), ((600, 16), "bf16", "bf16", "bf16")])
def test_softmax_backward_bitwise(dev, order, shape, yt, ct_t, dxt):
    rows, cols = shape
    rng = np.random.default_rng(cols)
    y32 = OS.softmax_region((rng.standard_normal((rows, cols)) * 2).astype(np.float32), "f32", "f32")
    ct32 = rng.standard_normal((rows, cols)).astype(np.float32)
    y = f32_to_bf16(y32) if yt == "bf16" else y32
    ct = f32_to_bf16(ct32) if ct_t == "bf16" else ct32
    want = OS.softmax_backward(y, ct, yt, ct_t, dxt, order)
    dx = _empty((rows, cols), dxt)
    dev.psk_softmax_backward(_to_dev(y, yt), _to_dev(ct, ct_t), dx, order)
    torch.cuda.synchronize()
    ok = _same(_to_host(dx), want, dxt)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} differ"
    assert dev.psk_device_status() == 0


@pytest.mark.parametrize("cols", [1000, 4096])
def test_softmax_backward_lane_kernel_bitwise(dev, cols):
    """Enough bf16 rows for the lane-per-row kernel (one lane per row, the
    y and ct tiles of each step loaded together): the one-chain orders bit
    for bit against the oracle, a ragged last tile included (1000 columns);
    the interleaved order, on the pipelined kernel, equal to it where its
    sum's order allows (checked against the oracle too)."""
    rows = 10_000
    rng = np.random.default_rng(cols + 1)
    y32 = OS.softmax_region((rng.standard_normal((rows, cols)) * 2).astype(np.float32), "f32", "f32")
    y = f32_to_bf16(y32)
    ct = f32_to_bf16(rng.standard_normal((rows, cols)).astype(np.float32))
    for order in (("sequential",), ("blocked", 64), ("interleaved", 8)):
        want = OS.softmax_backward(y, ct, "bf16", "bf16", "bf16", order)
        dx = _empty((rows, cols), "bf16")
        dev.psk_softmax_backward(_to_dev(y, "bf16"), _to_dev(ct, "bf16"), dx, order)
        torch.cuda.synchronize()
        ok = _same(_to_host(dx), want, "bf16")
        assert ok.all(), f"order {order}: {(~ok).sum()} of {ok.size} differ"
    assert dev.psk_device_status() == 0


def test_softmax_backward_in_place_and_refusals(dev):
    rng = np.random.default_rng(3)
    y = OS.softmax_region((rng.standard_normal((40, 256)) * 2).astype(np.float32), "f32", "f32")
    ct = rng.standard_normal((40, 256)).astype(np.float32)
    want = OS.softmax_backward(y, ct, "f32", "f32", "f32", ("interleaved", 8))
    ctd = _to_dev(ct, "f32")
    dev.psk_softmax_backward(_to_dev(y, "f32"), ctd, ctd, ("interleaved", 8))   # dx written over ct
    torch.cuda.synchronize()
    assert _same(_to_host(ctd), want, "f32").all()
    buf = torch.zeros(40 * 256 + 8, dtype=torch.float32, device="cuda")
    yd = buf[:40 * 256].view(40, 256)
    shifted = buf[8:].view(40, 256)                 # overlaps y, not in place: refused before any launch
    with pytest.raises(dev.PskError) as e:
        dev.psk_softmax_backward(yd, ctd, shifted, ("sequential",))
    assert e.value.name == "PSK_E_ALIAS"
    x = _to_dev(f32_to_bf16(y), "bf16")
    m = torch.ones(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(dev.PskError) as e:
        dev.psk_softmax_masked(x, x.clone(), m, ("interleaved", 65))
    assert e.value.name == "PSK_E_ORDER"


# ---------------------------------------------------- one-chain long rows
# Rows of 2048 < cols <= 4096 summed in one chain (sequential, blocked): partial
# last chain groups, rows past 512-column boundaries, enough rows per CTA that
# the rings wrap many times, both output types and both exp modes.

@pytest.mark.parametrize("rows,cols", [(1, 4096), (3, 2056), (5, 3000), (152 * 2 + 9, 4096), (152 * 40 + 13, 2064),
                                       (152 * 36 + 151, 4096)])
@pytest.mark.parametrize("order", [("sequential",), ("blocked", 64)])
def test_one_chain_long_rows_bitwise(dev, rows, cols, order):
    wl = W.softmax_rows(rows, cols)
    x = wl.host_x()
    dev.psk_device_status(reset=True)
    for yt in ("bf16", "f32"):
        want = OS.softmax_region(x, "bf16", yt, order)
        y = _empty((rows, cols), yt)
        dev.psk_softmax_region(_to_dev(x, "bf16"), y, order, "exact")
        torch.cuda.synchronize()
        ok = _same(_to_host(y), want, yt)
        assert ok.all(), f"{(~ok).sum()} of {ok.size} differ"
        dev.psk_softmax_region(_to_dev(x, "bf16"), y, order, "fast")
        torch.cuda.synchronize()
        got = _to_host(y)
        g = bf16_to_f32(got) if yt == "bf16" else got
        w = bf16_to_f32(want) if yt == "bf16" else want
        tol = 2.0 ** -7 if yt == "bf16" else 4e-6
        assert np.all(np.abs(g.astype(np.float64) - w) <= tol * np.abs(w) + 2.0 ** -140)
    assert dev.psk_device_status() == 0


def test_one_chain_long_rows_specials(dev):
    """-inf entries, a NaN row, an +inf row, an all -inf row and entries far
    below the row max, at 4096 columns in the sequential order."""
    rng = np.random.default_rng(31)
    rows, cols = 40, 4096
    x = (rng.standard_normal((rows, cols)) * 3).astype(np.float32)
    x[0, ::7] = -np.inf
    x[1, 5:400] = np.linspace(-120.0, -80.0, 395)
    x[1, 0] = 10.0
    x[2, :] = -np.inf
    x[3, 3000] = np.nan
    x[4, 4095] = np.inf
    x[5, 511:514] = 50.0
    xs = f32_to_bf16(x)
    want = OS.softmax_region(xs, "bf16", "f32", ("sequential",))
    y = _empty((rows, cols), "f32")
    dev.psk_softmax_region(_to_dev(xs, "bf16"), y, ("sequential",), "exact")
    torch.cuda.synchronize()
    assert _same(_to_host(y), want, "f32").all()


# ------------------------------------------------------ bounded waits
def test_lost_copy_times_out_and_the_device_recovers(dev):
    """The test hook makes every CTA's producer stop at its third row, as if
    the copy were lost: the waits for it run out (about two seconds), the
    kernel records the timeout in the status word and winds down, and the
    next launch on the same context is correct again."""
    rows, cols = 152 * 6, 512
    wl = W.softmax_rows(rows, cols)
    x = wl.host_x()
    xd = _to_dev(x, "bf16")
    y = _empty((rows, cols), "bf16")
    dev.psk_device_status(reset=True)
    try:
        dev.psk_test_drop_row(2)
        dev.psk_softmax_region(xd, y, ("interleaved", 8), "fast")
        torch.cuda.synchronize()
    finally:
        dev.psk_test_drop_row(-1)
    assert dev.psk_device_status(reset=True) & 1
    want = OS.softmax_region(x, "bf16", "bf16", ("sequential",))
    dev.psk_softmax_region(xd, y, ("sequential",), "exact")
    torch.cuda.synchronize()
    assert _same(_to_host(y), want, "bf16").all()
    assert dev.psk_device_status() == 0
