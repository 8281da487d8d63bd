"""Parity of the normalization regions (psk_norm_region, through the C ABI)
with the CPU oracle, bit for bit: every operation is IEEE (no transcendental
function), so the kernel and the oracle agree exactly in every order."""

import numpy as np
import pytest

import oracle.norm as ON
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
    if a is None:
        return None
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _to_host(t):
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


def _same(a, b, dtype):
    if dtype == "bf16":
        a = (a.astype(np.uint32) << 16).view(np.float32)
        b = (b.astype(np.uint32) << 16).view(np.float32)
    both_nan = np.isnan(a) & np.isnan(b)
    return (a.view(np.uint32) == b.view(np.uint32)) | both_nan


def _case(rows, cols, kind, xt, yt, pt, seed, eps=None):
    wl = W.NormWorkload("t", seed, rows, cols, kind, eps if eps is not None else (1e-6 if kind == "rms" else 1e-5),
                        xt, yt, pt or "f32")
    x = wl.host_x()
    g = wl.host_gamma() if pt else None
    b = wl.host_beta() if pt else None
    return wl, x, g, b


def _run(dev, wl, x, g, b, order, y=None):
    xd = _to_dev(x, wl.x_dtype)
    gy = None
    if y is None:                # NaN-poisoned, canaries around it
        gy = guarded(x.shape, torch.bfloat16 if wl.y_dtype == "bf16" else torch.float32)
        y = gy.tensor
    dev.psk_norm_region(xd, y, wl.kind, wl.eps, _to_dev(g, wl.param_dtype), _to_dev(b, wl.param_dtype), order)
    torch.cuda.synchronize()
    assert gy is None or gy.intact(), "a store landed outside the output"
    return _to_host(y)


def _want(wl, x, g, b, order):
    return ON.norm_region(x, wl.x_dtype, wl.y_dtype, wl.kind, wl.eps, g, b, wl.param_dtype, order)


ORDERS = [("sequential",), ("interleaved", 2), ("interleaved", 3), ("interleaved", 8), ("interleaved", 32),
          ("interleaved", 40)]


@pytest.mark.parametrize("kind", ["rms", "layer"])
@pytest.mark.parametrize("order", ORDERS, ids=lambda o: "-".join(map(str, o)))
@pytest.mark.parametrize("shape", [(64, 4096), (700, 512), (37, 999), (5, 10000), (3, 1), (600, 16)])
def test_norm_bitwise_orders_and_shapes(dev, kind, order, shape):
    wl, x, g, b = _case(*shape, kind, "bf16", "bf16", "bf16", 2000 + shape[1])
    got = _run(dev, wl, x, g, b, order)
    ok = _same(got, _want(wl, x, g, b, order), "bf16")
    assert ok.all(), f"{(~ok).sum()} of {ok.size} differ"
    assert dev.psk_device_status() == 0


@pytest.mark.parametrize("kind", ["rms", "layer"])
@pytest.mark.parametrize("xt,yt,pt", [("f32", "f32", "f32"), ("bf16", "f32", None), ("f32", "bf16", "bf16"),
                                      ("bf16", "bf16", "f32")])
def test_norm_storage_types_and_optional_params(dev, kind, xt, yt, pt):
    for shape in ((300, 1024), (41, 300)):
        wl, x, g, b = _case(*shape, kind, xt, yt, pt, 3000 + shape[0])
        for order in (("sequential",), ("interleaved", 8)):
            got = _run(dev, wl, x, g, b, order)
            assert _same(got, _want(wl, x, g, b, order), yt).all()


@pytest.mark.parametrize("rows,cols,order", [(2000, 4096, ("sequential",)), (2000, 4096, ("interleaved", 8)),
                                             (3000, 2048, ("interleaved", 2))])
@pytest.mark.parametrize("kind", ["rms", "layer"])
def test_norm_many_rows_per_cta(dev, rows, cols, order, kind):
    """Enough rows that every CTA's rings wrap several times (long and short chains)."""
    wl, x, g, b = _case(rows, cols, kind, "bf16", "bf16", "bf16", 4000 + cols)
    got = _run(dev, wl, x, g, b, order)
    ok = _same(got, _want(wl, x, g, b, order), "bf16")
    assert ok.all(), f"{(~ok).sum()} differ"
    assert dev.psk_device_status() == 0


def test_norm_special_rows(dev):
    """Zero rows (eps 0: 0/0 is NaN; eps > 0: zeros), constant rows (LayerNorm
    gives the bias), NaN and infinite entries, tiny and huge magnitudes (the
    divisor far from 1), in place, in both kinds and paths."""
    rng = np.random.default_rng(8)
    cols = 512
    x = (rng.standard_normal((12, cols)) * 2).astype(np.float32)
    x[0] = 0.0
    x[1] = 3.5
    x[2, 7] = np.nan
    x[3, 9] = np.inf
    x[4] *= np.float32(2.0 ** -70)
    x[5] *= np.float32(2.0 ** 60)
    x[6, ::3] = 0.0
    g = (1 + 0.1 * rng.standard_normal(cols)).astype(np.float32)
    bb = (0.1 * rng.standard_normal(cols)).astype(np.float32)
    for kind in ("rms", "layer"):
        for eps in (0.0, 1e-5):
            for order in (("sequential",), ("interleaved", 8), ("interleaved", 40)):
                beta = bb if kind == "layer" else None
                want = ON.norm_region(x, "f32", "f32", kind, eps, g, beta, "f32", order)
                t = _to_dev(x, "f32")
                dev.psk_norm_region(t, t, kind, eps, _to_dev(g, "f32"), _to_dev(beta, "f32"), order)
                torch.cuda.synchronize()
                assert _same(_to_host(t), want, "f32").all(), (kind, eps, order)


def test_norm_refusals(dev):
    x = torch.zeros((4, 8), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dev.PskError) as e:
        dev.psk_norm_region(x, x.clone(), "rms", 1e-6, g, g.clone())
    assert e.value.name == "PSK_E_ARG"
    with pytest.raises(dev.PskError) as e:
        dev.psk_norm_region(x, x.clone(), "layer", float("nan"))
    assert e.value.name == "PSK_E_ARG"
    with pytest.raises(dev.PskError) as e:
        dev.psk_norm_region(x, x.clone(), "layer", 1e-5, order=("interleaved", 65))
    assert e.value.name == "PSK_E_ORDER"
    big = torch.zeros((2, 49153), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dev.PskError) as e:
        dev.psk_norm_region(big, big.clone(), "rms", 1e-6)
    assert e.value.name == "PSK_E_SHAPE"
    buf = torch.zeros(40, dtype=torch.float32, device="cuda")
    xx = torch.zeros((4, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(dev.PskError) as e:      # y overlaps gamma
        dev.psk_norm_region(xx, buf[:32].view(4, 8), "rms", 1e-6, buf[30:38])
    assert e.value.name == "PSK_E_ALIAS"


@pytest.mark.parametrize("kind", ["rms", "layer"])
@pytest.mark.parametrize("order", [("sequential",), ("interleaved", 8)])
def test_norm_full_size_sampled_rows(dev, kind, order):
    wl = W.norm_rows(kind)
    x = wl.device_x()
    g, b = wl.device_params()
    y = torch.empty_like(x)
    dev.psk_norm_region(x, y, kind, wl.eps, g, b, order)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 16383, 32767] + list(np.random.default_rng(4).integers(0, 32768, 12)))
    idx = torch.from_numpy(rows).cuda()
    gh = wl.host_gamma()
    bh = wl.host_beta()
    want = ON.norm_region(_to_host(x[idx]), "bf16", "bf16", kind, wl.eps, gh, bh, "bf16", order)
    assert _same(_to_host(y[idx]), want, "bf16").all()
    assert dev.psk_device_status() == 0
