"""Parameter-shape lists of the gradient sets the workloads are shaped like.

Only shapes are needed (no weights): DDP's buckets, chunks and byte counts
depend on the tensors' element counts and registration order alone. Each list
is in registration order, the order the module defines its parameters.
"""
from __future__ import annotations

import math


def numel(shape) -> int:
    return int(math.prod(shape))


def tiny() -> list[tuple[str, tuple[int, ...]]]:
    """Ten small tensors with odd sizes: 277,421 elements in all."""
    shapes = [(3, 5), (7,), (64, 33), (33,), (128, 64), (128,), (1000, 17), (17,), (4096, 61), (61,)]
    return [(f"t{i}", s) for i, s in enumerate(shapes)]


def resnet50() -> list[tuple[str, tuple[int, ...]]]:
    """ResNet-50 (torchvision layout): 161 tensors, 25,557,032 parameters."""
    out: list[tuple[str, tuple[int, ...]]] = []

    def conv(name, cout, cin, k):
        out.append((f"{name}.weight", (cout, cin, k, k)))

    def bn(name, c):
        out.append((f"{name}.weight", (c,)))
        out.append((f"{name}.bias", (c,)))

    conv("conv1", 64, 3, 7)
    bn("bn1", 64)
    cin = 64
    for li, (blocks, width) in enumerate([(3, 64), (4, 128), (6, 256), (3, 512)], start=1):
        for b in range(blocks):
            pre = f"layer{li}.{b}"
            conv(f"{pre}.conv1", width, cin, 1)
            bn(f"{pre}.bn1", width)
            conv(f"{pre}.conv2", width, width, 3)
            bn(f"{pre}.bn2", width)
            conv(f"{pre}.conv3", width * 4, width, 1)
            bn(f"{pre}.bn3", width * 4)
            if b == 0:
                conv(f"{pre}.downsample.0", width * 4, cin, 1)
                bn(f"{pre}.downsample.1", width * 4)
            cin = width * 4
    out.append(("fc.weight", (1000, 2048)))
    out.append(("fc.bias", (1000,)))
    return out


def resnet50_buffers() -> list[tuple[str, tuple[int, ...], str]]:
    """ResNet-50's BatchNorm buffers (running_mean, running_var: fp32;
    num_batches_tracked: int64 scalar), in registration order."""
    out = []
    for name, shape in resnet50():
        if name.endswith(".bias") and ("bn" in name or "downsample.1" in name):
            base = name[: -len(".bias")]
            c = shape[0]
            out.append((f"{base}.running_mean", (c,), "f32"))
            out.append((f"{base}.running_var", (c,), "f32"))
            out.append((f"{base}.num_batches_tracked", (), "i64"))
    return out


def gpt2_small() -> list[tuple[str, tuple[int, ...]]]:
    """GPT-2 small, 12 layers, d=768, vocab 50257, context 1024, Conv1D layouts,
    head tied to wte: 148 tensors, 124,439,808 parameters."""
    d, v, ctx = 768, 50257, 1024
    out = [("wte", (v, d)), ("wpe", (ctx, d))]
    for i in range(12):
        h = f"h.{i}"
        out += [(f"{h}.ln_1.weight", (d,)), (f"{h}.ln_1.bias", (d,)),
                (f"{h}.attn.c_attn.weight", (d, 3 * d)), (f"{h}.attn.c_attn.bias", (3 * d,)),
                (f"{h}.attn.c_proj.weight", (d, d)), (f"{h}.attn.c_proj.bias", (d,)),
                (f"{h}.ln_2.weight", (d,)), (f"{h}.ln_2.bias", (d,)),
                (f"{h}.mlp.c_fc.weight", (d, 4 * d)), (f"{h}.mlp.c_fc.bias", (4 * d,)),
                (f"{h}.mlp.c_proj.weight", (4 * d, d)), (f"{h}.mlp.c_proj.bias", (d,))]
    out += [("ln_f.weight", (d,)), ("ln_f.bias", (d,))]
    return out


def llama_1b() -> list[tuple[str, tuple[int, ...]]]:
    """Llama-style decoder, 16 layers, d=2048, 32 heads (MHA), SwiGLU MLP 8192,
    vocab 32000, RMSNorm, untied head: 147 tensors, 1,204,881,408 parameters."""
    d, f, v = 2048, 8192, 32000
    out = [("embed_tokens", (v, d))]
    for i in range(16):
        pre = f"layers.{i}"
        out += [(f"{pre}.self_attn.q_proj", (d, d)), (f"{pre}.self_attn.k_proj", (d, d)),
                (f"{pre}.self_attn.v_proj", (d, d)), (f"{pre}.self_attn.o_proj", (d, d)),
                (f"{pre}.mlp.gate_proj", (f, d)), (f"{pre}.mlp.up_proj", (f, d)),
                (f"{pre}.mlp.down_proj", (d, f)),
                (f"{pre}.input_layernorm", (d,)), (f"{pre}.post_attention_layernorm", (d,))]
    out += [("norm", (d,)), ("lm_head", (v, d))]
    return out


def llama_buffers() -> list[int]:
    """Element counts of the 64 fp32 buffer tensors broadcast each forward in the
    Llama-shaped workload: integers uniform on [256, 4096] from a fixed hash."""
    from . import hash_np
    import numpy as np
    h = hash_np(1004, 1 << 21, np.arange(64, dtype=np.int64))
    return [int(256 + (int(x) >> 11) % (4096 - 256 + 1)) for x in h]
