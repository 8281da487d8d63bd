"""The softmax region's fast exp (through the test hook psk_test_fast_exp,
the function the region's fast realization applies to x - max) against the
oracle's correctly rounded exp: within two f32 ulp -- the tolerance stated
for exp nodes -- over every float of the binades [-1, -0.5) and [-104.5,
-64] (the latter's results run through the subnormals down to zero), over
200,000 floats of every other binade of [-104.5, 0), and at the special
values; zero at and below -104.5 and at -inf, NaN kept.  The distribution of
the gaps is printed."""

import numpy as np
import pytest

from oracle.crmath import exp_f32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import reduction_groups_gb300 as R

    return R


def _inputs():
    rng = np.random.default_rng(91)
    parts = [np.arange(0xBF000000, 0xBF800000, dtype=np.uint32),          # [-1, -0.5)
             np.arange(0xC2800000, 0xC2D10001, dtype=np.uint32)]          # [-104.5, -64]
    for e in range(-149, 6):                                              # magnitudes [2^e, 2^(e+1))
        if e in (-1, 6):
            continue
        if e < -126:                                                     # subnormal magnitudes
            lo, hi = 1 << (e + 149), 1 << (e + 150)
        else:
            lo, hi = (e + 127) << 23, (e + 128) << 23
        parts.append((0x80000000 + rng.integers(lo, hi, 200_000, dtype=np.int64)).astype(np.uint32))
    special = np.array([0.0, -0.0, -np.inf, np.nan, -104.5, -104.50001, -104.0, -103.97208, -87.33655,
                        -200.0, -3e38, -1e-45, -0.34657359, -0.6931472, -1.0], dtype=np.float32)
    return np.concatenate([np.concatenate(parts).view(np.float32), special])


def test_fast_exp_within_two_ulp(dev):
    x = _inputs()
    want = exp_f32(x)
    got = np.empty_like(x)
    chunk = 1 << 24
    for i in range(0, x.size, chunk):
        xd = torch.from_numpy(x[i:i + chunk]).cuda()
        yd = torch.empty_like(xd)
        dev.psk_test_fast_exp(xd, yd)
        torch.cuda.synchronize()
        got[i:i + chunk] = yd.cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    d = np.abs(got[fin].view(np.int32).astype(np.int64) - want[fin].view(np.int32).astype(np.int64))
    hist = np.bincount(np.minimum(d, 3), minlength=4)
    print(f"fast exp over {fin.sum()} floats: exact {hist[0]}, 1 ulp {hist[1]}, 2 ulp {hist[2]}, more {hist[3]}")
    assert d.max() <= 2
    assert np.all(got[x <= -104.5] == 0) and got[x == -np.inf][0] == 0


def test_fast_exp_refuses_bad_arguments(dev):
    from reduction_groups_gb300 import _native as N

    L = N.lib()
    assert L.psk_test_fast_exp(None, None, 0, None) == 0
    assert L.psk_test_fast_exp(None, None, 4, None) == -5            # PSK_E_NULL
    x = torch.zeros(4, device="cuda")
    assert L.psk_test_fast_exp(x.data_ptr(), x.data_ptr(), -1, None) == -3   # PSK_E_SHAPE
