"""The oracle's fp32 -> bf16 narrowing against torch's cast on every one of
the 2^32 fp32 bit patterns (CPU only, about a minute and a half).

The oracle's rounding is written from the definition (round to nearest, ties
to even, on the 16 discarded bits, a carry running into the exponent); torch's
CPU cast is an independent implementation of the same IEEE-style conversion.
NaNs are compared as NaN-equal: their payload is not fixed by the definition."""
import numpy as np
import pytest

from oracle.bf16 import bf16_to_f32, f32_to_bf16

torch = pytest.importorskip("torch")

CHUNK = 1 << 24


def test_every_fp32_pattern_rounds_like_torch():
    for c in range((1 << 32) // CHUNK):
        u = np.arange(c * CHUNK, (c + 1) * CHUNK, dtype=np.uint64).astype(np.uint32)
        x = u.view(np.float32)
        mine = f32_to_bf16(x)
        ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(x)
        bad = np.flatnonzero((mine != ref) & ~nan)
        assert bad.size == 0, f"pattern {int(u[bad[0]]):#010x}: oracle {int(mine[bad[0]]):#06x}, torch {int(ref[bad[0]]):#06x}"
        if nan.any():
            assert np.isnan(bf16_to_f32(mine[nan])).all()


def test_every_bf16_pattern_widens_exactly():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    wid = bf16_to_f32(b)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(wid.view(np.uint32)[~np.isnan(wid)], ref.view(np.uint32)[~np.isnan(ref)])
    assert np.array_equal(np.isnan(wid), np.isnan(ref))
    # and narrowing a widened value gives the pattern back (NaNs stay NaN)
    back = f32_to_bf16(wid)
    ok = ~np.isnan(wid)
    assert np.array_equal(back[ok], b[ok])
