"""The device's fp32 -> bf16 round-to-nearest-even conversion (torch's CUDA
cast) against the oracle's integer definition, on every one of the 2^32 fp32
bit patterns, on the GB300 itself. The library's kernels narrow with CUDA's
__float2bfloat16_rn; their bf16 results are compared bit for bit with the
oracle elsewhere, on the values the parity cases reach. NaNs compare as
NaN-equal. Takes a few minutes: the oracle side runs on the host."""
import numpy as np
import pytest

from oracle.bf16 import f32_to_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CHUNK = 1 << 26


def test_device_rounding_equals_the_oracle_on_every_pattern():
    for c in range((1 << 32) // CHUNK):
        lo = c * CHUNK
        bits = torch.arange(lo, lo + CHUNK, dtype=torch.int64, device="cuda").to(torch.int32)  # wraps to the same bits
        got = bits.view(torch.float32).to(torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16)
        u = np.arange(lo, lo + CHUNK, dtype=np.uint64).astype(np.uint32)
        x = u.view(np.float32)
        want = f32_to_bf16(x)
        bad = np.flatnonzero((got != want) & ~np.isnan(x))
        assert bad.size == 0, f"pattern {int(u[bad[0]]):#010x}: device {int(got[bad[0]]):#06x}, oracle {int(want[bad[0]]):#06x}"
        nan = np.isnan(x)
        if nan.any():
            g = got[nan]
            assert ((g & 0x7F80) == 0x7F80).all() and ((g & 0x007F) != 0).all()  # still NaN
