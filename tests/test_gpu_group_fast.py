"""The fast math mode of groups (psk_group_run_ex, PSK_EXP_FAST) against the
correctly rounded oracle, within its declared tolerance: EXP within one f32
ulp, EXPC and ERF within two, GELU (correctly rounded in this mode too)
identical, the same NaNs and infinities everywhere; on the 64-node workload
every output within one bf16 ulp of the oracle's and almost all identical.
"""

import numpy as np
import pytest

import oracle.group as OG
from oracle.f32 import bf16_to_f32
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


def _ordinal(bits, sign_bit):
    b = bits.astype(np.int64)
    mag = b & (sign_bit - 1)
    return np.where(b & sign_bit, -mag, mag)


def _ulps32(a, b):
    return np.abs(_ordinal(a.view(np.uint32), 1 << 31) - _ordinal(b.view(np.uint32), 1 << 31))


def _inputs(op, n, rng):
    if op in ("EXP",):
        x = rng.uniform(-110, 95, n)
    elif op == "EXPC":
        x = rng.uniform(-6, 6, n)
    else:
        x = rng.uniform(-6, 6, n)
    x = x.astype(np.float32)
    x[: n // 4] = rng.integers(0, 2 ** 32, n // 4, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x[:16] = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 88.72283935546875, 88.7228317,
                       -103.97208, 3.9192059, 2 ** -60, 2 ** -61, 87.0, -87.0, 1.0], dtype=np.float32)
    return x


@pytest.mark.parametrize("op,ulps", [("EXP", 1), ("EXPC", 2), ("ERF", 2), ("GELU", 0)])
def test_fast_node_within_its_tolerance(dev, op, ulps):
    rng = np.random.default_rng(81)
    n = (1 << 22) + 5
    x = _inputs(op, n, rng)
    toks = W.encode([("IN", 0), (op,)])
    want = OG.evaluate(toks, [], [(x, "f32", (1,))], (n,), "f32")
    g = guarded((n,), torch.float32)
    dev.psk_group_run(toks, [], [(_to_dev(x, "f32"), (1,))], g.tensor, math="fast")
    torch.cuda.synchronize()
    assert g.intact()
    got = _to_host(g.tensor)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    assert np.array_equal(np.isinf(got[fin]), np.isinf(want[fin]))
    u = _ulps32(got[fin], want[fin])
    print(f"{op} fast: max gap {u.max()} f32 ulp over {fin.sum()} inputs")
    assert u.max() <= ulps, f"max {u.max()} ulp at x={x[fin][np.argmax(u)]}"


def test_fast_expc_over_the_clamped_range(dev):
    """The EXP-clamp node's fast exp (the multifunction unit's 2^f after an
    exact split) over every float of [-4, -1) and [1, 4) and 50,000 floats of
    every other binade of (-4, 4), both signs: within two f32 ulp of the
    oracle's correctly rounded exp(clamp(x, -4, 4)); the gaps' distribution is
    printed."""
    rng = np.random.default_rng(83)
    parts = [np.arange(0x3F800000, 0x40800000, dtype=np.uint32)]          # [1, 4)
    for e in range(-149, 0):                                              # magnitudes [2^e, 2^(e+1))
        if e < -126:
            lo, hi = 1 << (e + 149), 1 << (e + 150)
        else:
            lo, hi = (e + 127) << 23, (e + 128) << 23
        parts.append(rng.integers(lo, hi, 50_000, dtype=np.int64).astype(np.uint32))
    mags = np.concatenate(parts)
    x = np.concatenate([mags, mags | np.uint32(0x80000000)]).view(np.float32)
    x = np.concatenate([x, np.array([0.0, -0.0, 4.0, -4.0, 3.9999998, -3.9999998, 0.34657359, -0.34657359,
                                     0.6931472, 2.7725887, -2.7725887], np.float32)])
    n = x.size
    toks = W.encode([("IN", 0), ("EXPC",)])
    want = OG.evaluate(toks, [], [(x, "f32", (1,))], (n,), "f32")
    g = guarded((n,), torch.float32)
    dev.psk_group_run(toks, [], [(_to_dev(x, "f32"), (1,))], g.tensor, math="fast")
    torch.cuda.synchronize()
    assert g.intact()
    got = _to_host(g.tensor)
    u = _ulps32(got, want)
    hist = np.bincount(np.minimum(u, 3), minlength=4)
    print(f"EXPC fast over {n} floats: exact {hist[0]}, 1 ulp {hist[1]}, 2 ulp {hist[2]}, more {hist[3]}")
    assert u.max() <= 2, f"max {u.max()} ulp at x={x[np.argmax(u)]}"


@pytest.mark.parametrize("shape", [(96, 200), (37, 53), (130, 1024)])
def test_fast_cap_group_within_one_bf16_ulp(dev, shape):
    wl = W.cap_group(*shape)
    ins = wl.host_inputs()
    want = OG.evaluate(wl.tokens, wl.imm, [(a, dt, s.strides) for (a, dt), s in zip(ins, wl.inputs)], wl.out_shape,
                       "bf16")
    g = guarded(wl.out_shape, torch.bfloat16)
    dins = [(_to_dev(a, dt), s.strides) for (a, dt), s in zip(ins, wl.inputs)]
    dev.psk_group_run(wl.tokens, wl.imm, dins, g.tensor, math="fast")
    torch.cuda.synchronize()
    assert g.intact()
    got = _to_host(g.tensor)
    both_nan = np.isnan(bf16_to_f32(got)) & np.isnan(bf16_to_f32(want))
    d = np.abs(_ordinal(got, 1 << 15) - _ordinal(want, 1 << 15))
    d[both_nan] = 0
    assert d.max() <= 1 and (d > 0).mean() < 1e-3


def test_fast_cap_group_full_size_sampled_rows(dev):
    """The 64-node workload at full size [8192, 8192] in the fast mode, as the
    benchmark launches it; sampled rows within one bf16 ulp of the oracle."""
    wl = W.cap_group()
    dins = wl.device_inputs()
    out = torch.empty(wl.out_shape, dtype=torch.bfloat16, device="cuda")
    dev.psk_group_run(wl.tokens, wl.imm, [(t, s.strides) for t, s in zip(dins, wl.inputs)], out, math="fast")
    torch.cuda.synchronize()
    rows = np.array([0, 1, 4095, 8191] + list(np.random.default_rng(3).integers(0, 8192, 12)))
    idx = torch.from_numpy(rows).cuda()
    x = _to_host(dins[0][idx])
    ins = [(x, "bf16", (8192, 1)), (_to_host(dins[1]), "bf16", (0, 1)), (_to_host(dins[2]).reshape(-1)[rows], "bf16", (1, 0)),
           (_to_host(dins[3]).reshape(1), "bf16", (0, 0))]
    want = OG.evaluate(wl.tokens, wl.imm, ins, (len(rows), 8192), "bf16")
    got = _to_host(out[idx])
    both_nan = np.isnan(bf16_to_f32(got)) & np.isnan(bf16_to_f32(want))
    d = np.abs(_ordinal(got, 1 << 15) - _ordinal(want, 1 << 15))
    d[both_nan] = 0
    assert d.max() <= 1 and (d > 0).mean() < 1e-3
