"""The shared input generator: host (numpy) and device (torch) implementations agree bit for bit."""
import numpy as np
import torch

import synth
from synth import shapes


def test_numpy_and_torch_generators_agree():
    idx = np.arange(12345, 12345 + 50000)
    for kind, sigma in (("normal", 1e-3), ("uniform", 1.0), ("normal", 1.0)):
        t = torch.empty(idx.size, dtype=torch.float32)
        synth.fill_(t, kind, 1002, 5, start=12345, sigma=sigma, block=7000)
        assert np.array_equal(t.numpy(), synth.values_np(kind, 1002, 5, idx, sigma))
    tb = torch.empty(idx.size, dtype=torch.bfloat16)
    synth.fill_(tb, "normal", 1004, 2, start=12345, sigma=1e-3)
    host = synth.values_np("normal", 1004, 2, idx, 1e-3, dtype="bf16")
    assert np.array_equal(tb.view(torch.int16).numpy().view(np.uint16), host)


def test_distributions():
    idx = np.arange(400000)
    x = synth.normal_np(1, 0, idx, 1e-3).astype(np.float64)
    assert abs(x.mean()) < 1e-5 and abs(x.std() - 1e-3) < 1e-5
    u = synth.uniform_np(1, 0, idx)
    assert u.min() >= -1 and u.max() < 1 and abs(u.mean()) < 5e-3
    # streams differ
    assert not np.array_equal(synth.normal_np(1, 0, idx[:100], 1.0), synth.normal_np(1, 1, idx[:100], 1.0))


def test_token_counts_in_range():
    c = synth.token_counts(1003, 8)
    assert len(c) == 8 and all(100 <= v <= 10000 for v in c)


def test_shape_sets():
    assert sum(shapes.numel(s) for _, s in shapes.tiny()) == 277421
    assert (len(shapes.resnet50()), sum(shapes.numel(s) for _, s in shapes.resnet50())) == (161, 25557032)
    assert (len(shapes.gpt2_small()), sum(shapes.numel(s) for _, s in shapes.gpt2_small())) == (148, 124439808)
    assert (len(shapes.llama_1b()), sum(shapes.numel(s) for _, s in shapes.llama_1b())) == (147, 1204881408)
    b = shapes.llama_buffers()
    assert len(b) == 64 and all(256 <= v <= 4096 for v in b)


def test_host_buffer_set_matches_the_device_one():
    from synth import workloads as W
    for name in ("resnet50", "llama_1b"):
        cfg = W.CONFIGS[name]
        dev = W.buffer_set(cfg, "cpu", p=2)
        host = W.buffer_set_host(cfg, p=2)
        for r in range(2):
            assert len(dev[r]) == len(host[r])
            for d, h in zip(dev[r], host[r]):
                assert np.array_equal(d.contiguous().view(-1).view(torch.uint8).numpy(), h)
