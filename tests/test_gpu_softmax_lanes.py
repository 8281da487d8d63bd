"""Parity of the lane-per-row softmax kernel (one warp lane per row, three
passes over the row, read and written in tiles of 64 columns by up to 32
rows) with the oracle and with the pipelined kernel, through the C ABI.

The kernel takes the fast realization of the one-chain orders (sequential,
blocked) over bf16 rows of 64 to 4096 columns (a multiple of 8), 16-byte
aligned, with at least 64 rows per SM (8 per warp of eight per SM); every case
here has that many rows.  Its outputs must be within the fast realization's tolerance of
the oracle (one bf16 ulp) and bit for bit those of the pipelined kernel
(which takes fewer rows), since both evaluate the same operations on the
same values; with exact exp the same calls take the pipelined kernel and
match the oracle bit for bit.
"""

import numpy as np
import pytest

import oracle.softmax as OS
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


def _lane_rows():
    """The fewest rows the lane kernel takes on this GPU (64 per SM)."""
    return 64 * torch.cuda.get_device_properties(0).multi_processor_count


def _to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _to_host(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _same(a, b):
    from oracle.f32 import bf16_to_f32

    x, y = bf16_to_f32(a), bf16_to_f32(b)
    return (x.view(np.uint32) == y.view(np.uint32)) | (np.isnan(x) & np.isnan(y))


def _within_one_ulp(got, want):
    from oracle.f32 import bf16_to_f32

    g, w = bf16_to_f32(got), bf16_to_f32(want)
    if not np.array_equal(np.isnan(g), np.isnan(w)):
        return False
    fin = ~np.isnan(w)
    return bool(np.all(np.abs(got[fin].astype(np.int64) - want[fin].astype(np.int64)) <= 1))


LANE_ORDERS = [("sequential",), ("blocked", 16)]
PIPE_ROWS = 1024      # too few rows for the lane kernel: the pipelined kernel


def _pipelined(dev, xd, order):
    """The fast realization of the first PIPE_ROWS rows, by the pipelined kernel."""
    y = torch.empty((PIPE_ROWS, xd.shape[1]), dtype=torch.bfloat16, device="cuda")
    dev.psk_softmax_region(xd[:PIPE_ROWS], y, order, "fast")
    torch.cuda.synchronize()
    return _to_host(y)


@pytest.mark.parametrize("order", LANE_ORDERS)
@pytest.mark.parametrize("extra,cols", [(0, 520), (271, 1032), (5, 72), (1, 64)])
def test_lane_kernel_within_tolerance_and_same_as_pipelined(dev, order, extra, cols):
    """Rows whose last tile is ragged (520, 1032 and 72 columns: one group of
    eight past the last full tile of 64), a one-tile row (64 columns), and row
    counts that leave the last batches partly past the tensor's end; the exact
    mode of the same call (the pipelined kernel) bit for bit."""
    rows = _lane_rows() + extra
    x = W.softmax_rows(rows, cols).host_x()
    want = OS.softmax_region(x, "bf16", "bf16", order)
    xd = _to_dev(x)
    gy = guarded((rows, cols), torch.bfloat16)
    dev.psk_device_status(reset=True)
    for mode in ("exact", "fast"):
        dev.psk_softmax_region(xd, gy.tensor, order, mode)
        torch.cuda.synchronize()
        assert gy.intact(), "a store landed outside the output"
        got = _to_host(gy.tensor)
        if mode == "exact":
            ok = _same(got, want)
            assert ok.all(), f"{(~ok).sum()} differ"
        else:
            assert _within_one_ulp(got, want)
            assert np.array_equal(got[:PIPE_ROWS], _pipelined(dev, xd, order))
    assert dev.psk_device_status() == 0


@pytest.mark.parametrize("order", LANE_ORDERS)
@pytest.mark.parametrize("cols", [2048, 4096])
def test_lane_kernel_full_rows(dev, order, cols):
    """Rows of 2048 and 4096 columns (32 and 64 tiles a pass; 4096 is the
    benchmark's row length)."""
    rows = _lane_rows() + 77
    x = W.softmax_rows(rows, cols).host_x()
    want = OS.softmax_region(x, "bf16", "bf16", order)
    xd = _to_dev(x)
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    dev.psk_softmax_region(xd, y, order, "fast")
    torch.cuda.synchronize()
    got = _to_host(y)
    assert _within_one_ulp(got, want)
    assert np.array_equal(got[:PIPE_ROWS], _pipelined(dev, xd, order))


def test_lane_kernel_strided_rows_in_place_and_specials(dev):
    """Rows inside a wider buffer (leading dimension above the row length),
    written in place, with a row of -inf (NaN outputs), a NaN, an inf (NaN
    row), a large shared maximum and values whose exp underflows."""
    rows, cols, ld = _lane_rows() + 9, 1024, 1024 + 24
    rng = np.random.default_rng(31)
    x = (rng.standard_normal((rows, cols)) * 3).astype(np.float32)
    x[2, :] = -np.inf
    x[3, 700] = np.nan
    x[4, 1023] = np.inf
    x[5, 511:514] = 50.0
    x[6, :] = -200.0
    x[6, 17] = 0.0
    x[rows - 1, :] = 0.0
    from oracle.f32 import f32_to_bf16

    xs = f32_to_bf16(x)
    for order in LANE_ORDERS:
        want = OS.softmax_region(xs, "bf16", "bf16", order)
        wide = np.zeros((rows, ld), dtype=np.uint16)
        wide[:, :cols] = xs
        buf = _to_dev(wide)
        pipe = _pipelined(dev, buf[:, :cols], order)
        view = buf[:, :cols]
        dev.psk_softmax_region(view, view, order, "fast")
        torch.cuda.synchronize()
        got = _to_host(buf)
        assert _within_one_ulp(got[:, :cols], want)
        assert np.array_equal(got[:PIPE_ROWS, :cols], pipe)
        assert np.array_equal(got[:, cols:], wide[:, cols:]), "the gap between rows was written"


def test_lane_kernel_lost_copy_times_out_and_the_device_recovers(dev):
    """The test hook withholds each warp's first copy of the batch holding its
    third row (local row 2): the warp's wait runs out (about two seconds), the
    timeout is recorded, the warp waits for its copies in flight and leaves;
    the next launch is correct."""
    rows, cols = _lane_rows() * 2, 512
    x = W.softmax_rows(rows, cols).host_x()
    xd = _to_dev(x)
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    dev.psk_device_status(reset=True)
    try:
        dev.psk_test_drop_row(2)
        dev.psk_softmax_region(xd, y, ("sequential",), "fast")
        torch.cuda.synchronize()
    finally:
        dev.psk_test_drop_row(-1)
    assert dev.psk_device_status(reset=True) & 1
    want = OS.softmax_region(x, "bf16", "bf16", ("sequential",))
    dev.psk_softmax_region(xd, y, ("sequential",), "exact")
    torch.cuda.synchronize()
    assert _same(_to_host(y), want).all()
    assert dev.psk_device_status() == 0
