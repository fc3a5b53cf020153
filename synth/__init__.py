"""Seeded synthetic inputs, shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the all-reduce: it only makes the numbers that
go in. Every value is a pure function of (seed, stream, index), so the host can
regenerate any single element of a multi-gigabyte device buffer bit for bit,
and the CPU oracle never needs to read its inputs back from the GPU.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based hash. Two
implementations of the same definition live here: numpy uint64 for the host
and torch int64 (two's-complement wrap-around) for device tensors. A CPU test
checks that they agree.

Value maps (all exact or IEEE-rounded, hence identical on both sides):
  * uniform(-1, 1): a 24-bit integer k -> (k - 2^23) * 2^-23, exact in fp32.
  * normal(0, sigma): Irwin-Hall sum of four 32-bit uniforms K (exact in int64
    and fp64), centred and scaled in fp64, rounded once to fp32. Same mean and
    variance as N(0, sigma^2); support is +-2*sqrt(3)*sigma.
  * bf16 inputs: the fp32 value converted by torch's round-to-nearest-even cast.
"""
from __future__ import annotations

import math

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _signed(c: int) -> int:
    return c - (1 << 64) if c >= (1 << 63) else c


# --------------------------------------------------------------------------- host (numpy)
def _mix_np(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= np.uint64(_M1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(_M2)
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, stream: int) -> int:
    """64-bit key of one stream (one replica, one buffer) under one seed."""
    z = (seed * GOLDEN + stream + 1) & MASK64
    return int(_mix_np(np.array([z], dtype=np.uint64))[0])


def hash_np(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    key = np.uint64(stream_key(seed, stream))
    with np.errstate(over="ignore"):
        z = key + (idx.astype(np.uint64) + np.uint64(1)) * np.uint64(GOLDEN)
    return _mix_np(z)


def uniform_np(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """fp32 values uniform on [-1, 1) at element indices idx."""
    k = (hash_np(seed, stream, idx) >> np.uint64(40)).astype(np.int64)
    return ((k - (1 << 23)).astype(np.float64) * 2.0 ** -23).astype(np.float32)


def _normal_scale(sigma: float) -> float:
    return sigma * math.sqrt(3.0) / 2.0 ** 32


def normal_np(seed: int, stream: int, idx: np.ndarray, sigma: float) -> np.ndarray:
    """fp32 values with mean 0 and standard deviation sigma at element indices idx."""
    idx = np.asarray(idx, dtype=np.int64)
    h1 = hash_np(seed, stream, 2 * idx)
    h2 = hash_np(seed, stream, 2 * idx + 1)
    lo = np.uint64(0xFFFFFFFF)
    s = ((h1 >> np.uint64(32)).astype(np.int64) + (h1 & lo).astype(np.int64)
         + (h2 >> np.uint64(32)).astype(np.int64) + (h2 & lo).astype(np.int64))
    centred = (s - ((1 << 33) - 2)).astype(np.float64)
    return (centred * _normal_scale(sigma)).astype(np.float32)


def to_bf16_bits_np(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of fp32 x, by torch's round-to-nearest-even cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def values_np(kind: str, seed: int, stream: int, idx: np.ndarray, sigma: float = 1.0,
              dtype: str = "f32") -> np.ndarray:
    """Host values for element indices idx: fp32 array, or uint16 bf16 bits."""
    idx = np.asarray(idx, dtype=np.int64)
    if kind == "uniform":
        v = uniform_np(seed, stream, idx)
    elif kind == "normal":
        v = normal_np(seed, stream, idx, sigma)
    else:
        raise ValueError(kind)
    return to_bf16_bits_np(v) if dtype == "bf16" else v


# --------------------------------------------------------------------------- device (torch)
def _lsr(z, k: int):
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix_t(z):
    z = z ^ _lsr(z, 30)
    z = z * _signed(_M1)
    z = z ^ _lsr(z, 27)
    z = z * _signed(_M2)
    return z ^ _lsr(z, 31)


def hash_t(seed: int, stream: int, idx):
    key = _signed(stream_key(seed, stream))
    return _mix_t(key + (idx + 1) * _signed(GOLDEN))


def fill_(out, kind: str, seed: int, stream: int, start: int = 0, sigma: float = 1.0,
          block: int = 1 << 25):
    """Fill the contiguous 1-D tensor `out` (fp32 or bf16, any device) with the values
    of elements start .. start+out.numel()-1 of the given stream."""
    import torch
    n = out.numel()
    dev = out.device
    for b0 in range(0, n, block):
        b1 = min(n, b0 + block)
        idx = torch.arange(start + b0, start + b1, device=dev, dtype=torch.int64)
        if kind == "uniform":
            k = _lsr(hash_t(seed, stream, idx), 40)
            v = ((k - (1 << 23)).to(torch.float64) * 2.0 ** -23).to(torch.float32)
        elif kind == "normal":
            h1 = hash_t(seed, stream, 2 * idx)
            h2 = hash_t(seed, stream, 2 * idx + 1)
            lo = 0xFFFFFFFF
            s = _lsr(h1, 32) + (h1 & lo) + _lsr(h2, 32) + (h2 & lo)
            del h1, h2
            v = ((s - ((1 << 33) - 2)).to(torch.float64) * _normal_scale(sigma)).to(torch.float32)
        else:
            raise ValueError(kind)
        out[b0:b1].copy_(v.to(out.dtype))
    return out


def host_f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """fp32 values of uint16 bf16 bit patterns (exact widening)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def token_counts(seed: int, p: int, lo: int = 100, hi: int = 10000) -> list[int]:
    """Per-replica non-padding token counts, integers uniform on [lo, hi] inclusive."""
    h = hash_np(seed, 1 << 20, np.arange(p, dtype=np.int64))
    return [int(lo + (int(v) >> 11) % (hi - lo + 1)) for v in h]
