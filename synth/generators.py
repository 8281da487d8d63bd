"""Counter-based random draws for the synthetic workloads (no method arithmetic)."""

from __future__ import annotations

import numpy as np

_TWO_NEG53 = 1.0 / 9007199254740992.0


def _stream(seed: int, tensor_id: int) -> np.random.Philox:
    # One Philox4x32-10 stream per (seed, tensor): the key comes from a
    # SeedSequence over both, so streams never overlap and never depend on
    # the order in which tensors are drawn.
    return np.random.Philox(np.random.SeedSequence([int(seed), int(tensor_id)]))


def _uniform53(seed: int, tensor_id: int, n: int) -> np.ndarray:
    """n float64 uniforms in [0, 1) with 53 random bits each."""
    raw = _stream(seed, tensor_id).random_raw(n)
    return (raw >> np.uint64(11)).astype(np.float64) * _TWO_NEG53


def host_normal(shape, std: float, seed: int, tensor_id: int) -> np.ndarray:
    """float32 draws of N(0, std^2): Box-Muller in float64, one rounding to f32."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape, dtype=np.int64))
    m = (n + 1) // 2
    u = _uniform53(seed, tensor_id, 2 * m)
    u1 = 1.0 - u[0::2]  # (0, 1]: log is finite
    u2 = u[1::2]
    rad = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = rad * np.cos(2.0 * np.pi * u2)
    z[1::2] = rad * np.sin(2.0 * np.pi * u2)
    return (z[:n] * float(std)).astype(np.float32).reshape(shape)


def host_uniform(shape, lo: float, hi: float, seed: int, tensor_id: int) -> np.ndarray:
    """float32 draws of U(lo, hi): 24 random bits on [lo, hi), exact in f32 for
    lo, hi powers of two apart (the workloads use [-2, 2))."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape, dtype=np.int64))
    raw = _stream(seed, tensor_id).random_raw(n)
    k = (raw >> np.uint64(40)).astype(np.float64)  # 24-bit integer
    v = lo + (hi - lo) * (k / 16777216.0)
    return v.astype(np.float32).reshape(shape)


def host_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 storage (nearest even), as uint16 bit patterns.

    Used only to store drawn inputs in bf16; the draws themselves are finite."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


# ---------------------------------------------------------------- device draws

def _torch_gen(seed: int, tensor_id: int, device):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(tensor_id)) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def device_normal(shape, std: float, seed: int, tensor_id: int, device="cuda", dtype=None):
    """N(0, std^2) drawn on the device (torch's Philox generator), stored as dtype."""
    import torch

    dtype = dtype or torch.float32
    t = torch.empty(tuple(shape), dtype=torch.float32, device=device)
    t.normal_(0.0, float(std), generator=_torch_gen(seed, tensor_id, device))
    return t if dtype == torch.float32 else t.to(dtype)


def device_abs_normal(shape, std: float, seed: int, tensor_id: int, device="cuda"):
    t = device_normal(shape, std, seed, tensor_id, device)
    return t.abs_()


def device_uniform(shape, lo: float, hi: float, seed: int, tensor_id: int, device="cuda", dtype=None):
    """U(lo, hi) drawn on the device with 24 random bits, stored as dtype."""
    import torch

    dtype = dtype or torch.float32
    g = _torch_gen(seed, tensor_id, device)
    k = torch.randint(0, 1 << 24, tuple(shape), generator=g, device=device, dtype=torch.int32)
    t = k.to(torch.float32).mul_((hi - lo) / 16777216.0).add_(lo)
    return t if dtype == torch.float32 else t.to(dtype)
