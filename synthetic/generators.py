"""Seeded, counter-based synthetic inputs.

This module is the one piece shared by the CUDA-path tests, the bench and the
oracle tests.  It holds none of the optimizer's arithmetic: only an integer
hash, an approximately normal draw built from it, a Bernoulli mask, and
rounding of FP32 values to the 16-bit gradient storage formats.

Why counter-based: value ``i`` of any stream is a pure function of
``(key, i)``.  The device can therefore fill a 1.2e9-element buffer in chunks
with plain torch integer ops, while the host recomputes any sampled index with
numpy and obtains the very same bits.  Every step is exact integer arithmetic
or a single correctly rounded FP32 multiply, so both sides agree bit for bit.

The normal draw is an Irwin-Hall sum of four 22-bit uniforms, centred and
scaled to the requested standard deviation.  Its mean and variance are those
of N(0, sigma^2); its support is bounded at +-2*sqrt(3)*sigma.
"""

from __future__ import annotations

import math

import numpy as np

MASK32 = 0xFFFFFFFF
_MUL_A = 0x7FEB352D  # odd, < 2**31: products with a 32-bit value fit in int64
_MUL_B = 0x2C1B3C6D  # odd, < 2**31
_BITS = 22           # bits kept from each uniform
_NUNI = 4            # uniforms summed per normal draw
_CENTER = _NUNI * ((1 << _BITS) - 1) // 2   # = 2**23 - 2, exact mean of the sum

# Largest index any stream supports: indices are hashed as 32-bit words.
MAX_INDEX = 1 << 32


def _mix32_scalar(x: int) -> int:
    x &= MASK32
    x ^= x >> 16
    x = (x * _MUL_A) & MASK32
    x ^= x >> 15
    x = (x * _MUL_B) & MASK32
    x ^= x >> 16
    return x


def stream_key(*parts: int) -> int:
    """Fold integers (seed, stream id, step, ...) into one 32-bit key."""
    h = 0x9E3779B9
    for p in parts:
        h = _mix32_scalar(h ^ _mix32_scalar(int(p) & MASK32) ^ (int(p) >> 32))
    return h


def _subkeys(key: int, count: int) -> list[tuple[int, int]]:
    return [(_mix32_scalar(key ^ (0x51ED27 * (2 * k + 1))),
             _mix32_scalar(key + 0x2545F491 * (k + 1)))
            for k in range(count)]


# --------------------------------------------------------------------------
# numpy (host) side
# --------------------------------------------------------------------------

def _mix32_np(x: np.ndarray) -> np.ndarray:
    x = x ^ (x >> np.uint64(16))
    x = (x * np.uint64(_MUL_A)) & np.uint64(MASK32)
    x = x ^ (x >> np.uint64(15))
    x = (x * np.uint64(_MUL_B)) & np.uint64(MASK32)
    x = x ^ (x >> np.uint64(16))
    return x


def _uniform32_np(idx: np.ndarray, ka: int, kb: int) -> np.ndarray:
    return _mix32_np(_mix32_np(idx ^ np.uint64(ka)) ^ np.uint64(kb))


def _as_index(idx) -> np.ndarray:
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= MAX_INDEX):
        raise ValueError("synthetic index outside [0, 2**32)")
    return idx.astype(np.uint64)


def normal_scale_f32(sigma: float) -> np.float32:
    """FP32 factor that maps the centred integer sum to standard deviation sigma."""
    return np.float32(sigma * math.sqrt(3.0) / float(1 << _BITS))


def normal_np(idx, sigma: float, key: int) -> np.ndarray:
    """Approximately N(0, sigma^2) FP32 values at the given element indices."""
    u = _as_index(idx)
    s = np.zeros(u.shape, dtype=np.int64)
    for ka, kb in _subkeys(key, _NUNI):
        s += (_uniform32_np(u, ka, kb) >> np.uint64(32 - _BITS)).astype(np.int64)
    z = (s - _CENTER).astype(np.float32)          # |z| < 2**23: exact
    return z * normal_scale_f32(sigma)             # one rounded FP32 multiply


def bernoulli_np(idx, prob_per_10000: int, key: int) -> np.ndarray:
    """Boolean mask, true with probability prob_per_10000 / 10000."""
    u = _as_index(idx)
    (ka, kb), = _subkeys(key, 1)
    return (_uniform32_np(u, ka, kb) % np.uint64(10000)) < np.uint64(prob_per_10000)


def f32_to_bf16_bits_np(x: np.ndarray) -> np.ndarray:
    """Round FP32 to BF16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (b & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    r = np.where(nan, (b >> np.uint64(16)) | np.uint64(0x40), r)
    return r.astype(np.uint16)


def f32_to_f16_bits_np(x: np.ndarray) -> np.ndarray:
    """Round FP32 to IEEE binary16 (nearest, ties to even); uint16 bit patterns."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def bf16_bits_to_f32_np(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f16_bits_to_f32_np(b: np.ndarray) -> np.ndarray:
    return np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float32)


# --------------------------------------------------------------------------
# torch (device) side: same integers, same single FP32 multiply
# --------------------------------------------------------------------------

def _mix32_t(x):
    x ^= x >> 16
    x.mul_(_MUL_A).bitwise_and_(MASK32)
    x ^= x >> 15
    x.mul_(_MUL_B).bitwise_and_(MASK32)
    x ^= x >> 16
    return x


def _uniform32_t(base, ka: int, kb: int):
    x = base ^ ka
    _mix32_t(x)
    x ^= kb
    return _mix32_t(x)


def normal_torch(start: int, count: int, sigma: float, key: int, device):
    """FP32 tensor of indices [start, start+count) of the normal stream ``key``."""
    import torch
    if start < 0 or start + count > MAX_INDEX:
        raise ValueError("synthetic index outside [0, 2**32)")
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    s = torch.zeros_like(idx)
    for ka, kb in _subkeys(key, _NUNI):
        s += _uniform32_t(idx, ka, kb) >> (32 - _BITS)
    del idx
    s -= _CENTER
    z = s.to(torch.float32)
    del s
    scale = torch.tensor(float(normal_scale_f32(sigma)), dtype=torch.float32, device=device)
    return z.mul_(scale)


def bernoulli_torch(start: int, count: int, prob_per_10000: int, key: int, device):
    import torch
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    (ka, kb), = _subkeys(key, 1)
    return (_uniform32_t(idx, ka, kb) % 10000) < prob_per_10000


def f32_to_bf16_bits_torch(x):
    """Round an FP32 tensor to BF16 bits (ties to even); returns int64 holding uint16."""
    import torch
    b = x.contiguous().view(torch.int32).to(torch.int64) & MASK32
    nan = (b & 0x7FFFFFFF) > 0x7F800000
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) & 0xFFFF
    return torch.where(nan, (b >> 16) | 0x40, r)


def store_bits_torch(bits_u16, out_16bit):
    """Write uint16 patterns (held in int64) into a 16-bit tensor of any float type."""
    import torch
    signed = torch.where(bits_u16 >= 0x8000, bits_u16 - 0x10000, bits_u16)
    out_16bit.view(torch.int16).copy_(signed.to(torch.int16))
