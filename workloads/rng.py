"""Counter-based seeded random numbers shared by the oracle side and the GPU side.

This module holds no attention arithmetic. It turns (seed, counter) into numbers:

* ``u64``: output ``n`` of a SplitMix64 stream started at ``seed``, i.e.
  ``mix(seed + (n + 1) * GAMMA)`` with the 64-bit finaliser of Steele, Lea and
  Flood, "Fast splittable pseudorandom number generators" (OOPSLA 2014), with
  the finaliser constants of Vigna's public-domain ``splitmix64.c``.  Because an
  output depends only on its counter, any slice of a stream can be regenerated
  on its own: the oracle side rebuilds exactly the rows it checks.
* ``uniform``: ``(u64 >> 11) * 2**-53`` in [0, 1).
* ``normal``: Box-Muller (cosine branch) on draws ``2e`` and ``2e + 1`` in
  float64, rounded to float32 (nearest) and then to bfloat16 (nearest-even on
  the bit pattern).  One standard normal per element counter ``e``.

Two implementations of the same definition live here: numpy (host) and torch
(host or device, using wrapping int64 arithmetic).  ``tests/test_inputs.py``
checks that they agree bit for bit.
"""
from __future__ import annotations

import math

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1

BF16_NAN_BITS = 0x7FC0


def _fnv1a64(text: str) -> int:
    """FNV-1a 64-bit hash of a stream name (offset basis and prime are the published ones)."""
    h = 0xCBF29CE484222325
    for byte in text.encode("utf-8"):
        h ^= byte
        h = (h * 0x100000001B3) & _MASK64
    return h


def _mix_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * MIX1) & _MASK64
    z = ((z ^ (z >> 27)) * MIX2) & _MASK64
    return z ^ (z >> 31)


def stream_seed(base_seed: int, name: str) -> int:
    """Seed of the named stream under one workload seed (a mixed 64-bit value)."""
    return _mix_int((base_seed & _MASK64) ^ _fnv1a64(name))


# --------------------------------------------------------------------------- numpy
_G = np.uint64(GAMMA)
_M1 = np.uint64(MIX1)
_M2 = np.uint64(MIX2)


def u64_np(seed: int, start: int, count: int) -> np.ndarray:
    n = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _MASK64) + (n + np.uint64(1)) * _G
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def uniform_np(seed: int, start: int, count: int) -> np.ndarray:
    return (u64_np(seed, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal_f64_np(seed: int, start: int, count: int) -> np.ndarray:
    a = u64_np(seed, 2 * start, 2 * count)
    u1 = ((a[0::2] >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)
    u2 = (a[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def f32_to_bf16_bits_np(x32: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32_np(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16_np(seed: int, start: int, count: int) -> np.ndarray:
    """``count`` standard normals from element counter ``start``, as bf16 bits (uint16)."""
    return f32_to_bf16_bits_np(normal_f64_np(seed, start, count).astype(np.float32))


# --------------------------------------------------------------------------- torch
def _signed(v: int) -> int:
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def _srl(x, k: int):
    """Logical right shift of int64 tensors."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def u64_torch(seed: int, start: int, count: int, device):
    import torch

    n = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    z = n * _signed(GAMMA) + _signed(seed)
    z = (z ^ _srl(z, 30)) * _signed(MIX1)
    z = (z ^ _srl(z, 27)) * _signed(MIX2)
    return z ^ _srl(z, 31)


def uniform_torch(seed: int, start: int, count: int, device):
    import torch

    return _srl(u64_torch(seed, start, count, device), 11).to(torch.float64) * (2.0 ** -53)


def normal_f64_torch(seed: int, start: int, count: int, device):
    import torch

    a = u64_torch(seed, 2 * start, 2 * count, device)
    u1 = (_srl(a[0::2], 11) + 1).to(torch.float64) * (2.0 ** -53)
    u2 = _srl(a[1::2], 11).to(torch.float64) * (2.0 ** -53)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)


def f32_to_bf16_torch(x32):
    """Round float32 to bfloat16 (nearest-even on the bit pattern); returns a bfloat16 tensor."""
    import torch

    b = x32.contiguous().view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    r = torch.where(r >= 0x8000, r - 0x10000, r)
    return r.to(torch.int16).view(torch.bfloat16)


def normal_bf16_torch(seed: int, start: int, count: int, device):
    import torch

    return f32_to_bf16_torch(normal_f64_torch(seed, start, count, device).to(torch.float32))
