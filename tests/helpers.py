"""Shared helpers of the GPU parity tests: seeded replicas on the device and
the same values on the host (both from the synth generator, never read back
from the device for the oracle)."""
from __future__ import annotations

import numpy as np

import synth


def make_replicas(p, n, dtype="f32", kind="normal", seed=1, sigma=1.0, offsets=None, device="cuda"):
    """p device tensors of n elements (views at element offsets `offsets[r]`
    inside slightly larger allocations, to test misalignment) and the matching
    host arrays (fp32 values, or uint16 bf16 patterns)."""
    import torch
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    offsets = offsets or [0] * p
    devs, hosts, bases = [], [], []
    for r in range(p):
        base = torch.empty(n + offsets[r] + 8, dtype=tdt, device=device)
        v = base[offsets[r]:offsets[r] + n]
        if n:
            synth.fill_(v, kind, seed, r, 0, sigma)
        devs.append(v)
        bases.append(base)
        hosts.append(synth.values_np(kind, seed, r, np.arange(n), sigma, dtype))
    return devs, hosts, bases


def to_host(t) -> np.ndarray:
    """Device tensor -> numpy (fp32 values or uint16 bf16 patterns)."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


def assert_bit_equal(got: np.ndarray, want: np.ndarray, what=""):
    g, w = bits(np.ascontiguousarray(got)), bits(np.ascontiguousarray(want))
    assert g.shape == w.shape, (what, g.shape, w.shape)
    bad = np.flatnonzero(g != w)
    assert bad.size == 0, f"{what}: {bad.size} mismatches, first at {bad[:5]}: got {got[bad[:5]]} want {want[bad[:5]]}"


def assert_bf16_close(got_bits: np.ndarray, want_bits: np.ndarray, what=""):
    """The stated bf16 criterion: |got - want| <= 1e-5 + 1e-6 |want| (values)."""
    from oracle.bf16 import bf16_to_f32
    g = bf16_to_f32(got_bits).astype(np.float64)
    w = bf16_to_f32(want_bits).astype(np.float64)
    assert np.all(np.abs(g - w) <= 1e-5 + 1e-6 * np.abs(w)), what
