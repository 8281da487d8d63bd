"""Parity of RMSNorm and LayerNorm on the lane-per-row kernel (one warp lane
per row; the chains, then the output pass, over tiles of 64 columns) with the
oracle, bit for bit, through the C ABI.

The kernel takes the one-chain orders (sequential, blocked) over bf16 rows of
64 to 4096 columns (a multiple of 8), 16-byte aligned, with at least 64 rows
per SM; every case here has that many rows (the interleaved cases take the
pipelined kernel on the same rows and are checked alike).
"""

import numpy as np
import pytest

from tests.test_gpu_norm import _case, _run, _same, _to_dev, _to_host, _want

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import reduction_groups_gb300 as R

    return R


def _lane_rows():
    return 64 * torch.cuda.get_device_properties(0).multi_processor_count


ORDERS = [("sequential",), ("blocked", 16), ("interleaved", 8)]


@pytest.mark.parametrize("kind", ["rms", "layer"])
@pytest.mark.parametrize("order", ORDERS, ids=lambda o: "-".join(map(str, o)))
@pytest.mark.parametrize("extra,cols", [(0, 520), (271, 1032), (5, 72), (1, 64)])
def test_norm_lanes_bitwise(dev, kind, order, extra, cols):
    """Ragged last tiles (520, 1032, 72 columns), a one-tile row, and row
    counts that leave the last batches partly past the tensor's end."""
    wl, x, g, b = _case(_lane_rows() + extra, cols, kind, "bf16", "bf16", "bf16", 5000 + cols)
    dev.psk_device_status(reset=True)
    got = _run(dev, wl, x, g, b, order)
    ok = _same(got, _want(wl, x, g, b, order), "bf16")
    assert ok.all(), f"{(~ok).sum()} of {ok.size} differ"
    assert dev.psk_device_status() == 0


@pytest.mark.parametrize("kind", ["rms", "layer"])
@pytest.mark.parametrize("order", [("sequential",), ("interleaved", 8)], ids=lambda o: "-".join(map(str, o)))
def test_norm_lanes_full_rows(dev, kind, order):
    """Rows of 4096 columns, the benchmark's row length."""
    wl, x, g, b = _case(_lane_rows() + 33, 4096, kind, "bf16", "bf16", "bf16", 5100)
    got = _run(dev, wl, x, g, b, order)
    ok = _same(got, _want(wl, x, g, b, order), "bf16")
    assert ok.all(), f"{(~ok).sum()} differ"


@pytest.mark.parametrize("kind", ["rms", "layer"])
@pytest.mark.parametrize("pt", ["f32", None])
def test_norm_lanes_parameter_types(dev, kind, pt):
    """f32 scale and bias, and none at all."""
    wl, x, g, b = _case(_lane_rows() + 3, 256, kind, "bf16", "bf16", pt, 5200)
    for order in (("sequential",), ("interleaved", 4)):
        got = _run(dev, wl, x, g, b, order)
        assert _same(got, _want(wl, x, g, b, order), "bf16").all()


@pytest.mark.parametrize("kind", ["rms", "layer"])
def test_norm_lanes_strided_in_place_and_specials(dev, kind):
    """Rows inside a wider buffer, normalised in place, with a row of -0 (its
    chains must start at -0, not +0), a row of zeros (zero eps: 0 / 0), a NaN,
    an infinity and large values."""
    rows, cols, ld = _lane_rows() + 9, 512, 512 + 40
    wl, x, g, b = _case(rows, cols, kind, "bf16", "bf16", "bf16", 5300, eps=0.0)
    x = x.copy()
    x[2, :] = 0x8000             # -0
    x[3, :] = 0
    x[4, 100] = 0x7FC0           # NaN
    x[5, 7] = 0x7F80             # inf
    x[6, :] = 0x7F00             # 2^127: the squares overflow
    for order in (("sequential",), ("interleaved", 8)):
        want = _want(wl, x, g, b, order)
        wide = np.zeros((rows, ld), dtype=np.uint16)
        wide[:, :cols] = x
        buf = _to_dev(wide, "bf16")
        view = buf[:, :cols]
        dev.psk_norm_region(view, view, kind, 0.0, _to_dev(g, "bf16"), _to_dev(b, "bf16") if kind == "layer" else None,
                            order)
        torch.cuda.synchronize()
        got = _to_host(buf)
        ok = _same(got[:, :cols], want, "bf16")
        assert ok.all(), f"{(~ok).sum()} differ, rows {np.nonzero(~ok.all(axis=1))[0][:5]}"
        assert np.array_equal(got[:, cols:], wide[:, cols:]), "the gap between rows was written"
