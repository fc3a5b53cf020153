"""The synthetic gradient sets the tests and the bench run on, and host-side
lookup of any of their input values (inputs only: no all-reduce arithmetic).

Each replica r's gradients are one seeded stream (stream r): element e of
tensor t is element tensor_start[t] + e of the stream, tensors in registration
order. On the device each replica's tensors are carved out of one arena at
256-byte-aligned offsets, as a caching allocator would place separate tensors.
"""
from __future__ import annotations

import numpy as np

from . import fill_, token_counts, values_np
from . import shapes as S

MiB = 1 << 20

CONFIGS = {
    # ten odd-sized fp32 tensors, p=4, N(0,1), caps 16 KiB / 256 KiB, fp32 sum then scale 1/p
    "tiny": dict(shapes=S.tiny, p=4, dtype="f32", sigma=1.0, first_cap=16 << 10, cap=256 << 10,
                 divisor="p", seed=1001),
    # ResNet-50's 161 tensors (25.6M fp32), p=8, N(0, 1e-3), caps 1 MiB / 25 MiB, average by 1/8
    "resnet50": dict(shapes=S.resnet50, p=8, dtype="f32", sigma=1e-3, first_cap=1 * MiB, cap=25 * MiB,
                     divisor="p", seed=1002, buffers="resnet50"),
    # GPT-2 small's 148 tensors (124M fp32), p=8, N(0, 1e-3), 25 MiB buckets, divide once by the
    # global token count (per-replica counts uniform on [100, 10000])
    "gpt2_small": dict(shapes=S.gpt2_small, p=8, dtype="f32", sigma=1e-3, first_cap=1 * MiB, cap=25 * MiB,
                       divisor="tokens", seed=1003),
    # Llama-style 1B (147 tensors, 1.2B bf16), p=8, N(0, 1e-3) rounded to bf16, 25 MiB buckets,
    # average by 1/8, plus a per-forward coalesced broadcast of 64 fp32 buffers from replica 0
    "llama_1b": dict(shapes=S.llama_1b, p=8, dtype="bf16", sigma=1e-3, first_cap=1 * MiB, cap=25 * MiB,
                     divisor="p", seed=1004, buffers="llama"),
}


def numels(cfg) -> list[int]:
    return [S.numel(s) for _, s in cfg["shapes"]()]


def tensor_starts(cfg) -> list[int]:
    n = numels(cfg)
    return [int(x) for x in np.concatenate([[0], np.cumsum(n)[:-1]])]


def divisor(cfg) -> float:
    if cfg["divisor"] == "p":
        return float(cfg["p"])
    return float(sum(token_counts(cfg["seed"], cfg["p"])))


def esize(cfg) -> int:
    return 4 if cfg["dtype"] == "f32" else 2


def arena_layout(cfg):
    """Element offset of each tensor inside a replica's arena (256-byte
    aligned, registration order) and the arena's length in elements."""
    align = 256 // esize(cfg)
    offs, pos = [], 0
    for x in numels(cfg):
        offs.append(pos)
        pos += (x + align - 1) // align * align
    return offs, pos


def make_grads(cfg, device="cuda", p=None):
    """p lists of k device tensors holding the seeded gradients."""
    import torch
    p = p or cfg["p"]
    tdt = torch.float32 if cfg["dtype"] == "f32" else torch.bfloat16
    n = numels(cfg)
    starts = tensor_starts(cfg)
    offs, pos = arena_layout(cfg)
    grads, arenas = [], []
    for r in range(p):
        arena = torch.empty(max(pos, 1), dtype=tdt, device=device)
        row = []
        for t, x in enumerate(n):
            v = arena[offs[t]:offs[t] + x]
            fill_(v, "normal", cfg["seed"], r, starts[t], cfg["sigma"])
            row.append(v)
        grads.append(row)
        arenas.append(arena)
    return grads, arenas


def make_grads_from_host(cfg, device="cuda", p=None):
    """As make_grads, with the same values and layout, but every replica's
    arena is generated on the host and copied to the device in one copy, so no
    device kernel runs (for small sets)."""
    import torch
    p = p or cfg["p"]
    n = numels(cfg)
    starts = tensor_starts(cfg)
    offs, pos = arena_layout(cfg)
    host_dt = np.float32 if cfg["dtype"] == "f32" else np.uint16
    grads, arenas = [], []
    for r in range(p):
        h = np.zeros(max(pos, 1), dtype=host_dt)
        for t, x in enumerate(n):
            h[offs[t]:offs[t] + x] = host_values(cfg, r, np.arange(starts[t], starts[t] + x))
        ht = torch.from_numpy(h) if cfg["dtype"] == "f32" else torch.from_numpy(h.view(np.int16)).view(torch.bfloat16)
        arena = ht.to(device)
        grads.append([arena[offs[t]:offs[t] + x] for t, x in enumerate(n)])
        arenas.append(arena)
    return grads, arenas


def host_values(cfg, r: int, flat_idx: np.ndarray) -> np.ndarray:
    """Replica r's input gradient values at registration-order flat indices."""
    return values_np("normal", cfg["seed"], r, flat_idx, cfg["sigma"], cfg["dtype"])


def buffer_set(cfg, device="cuda", p=None):
    """The per-forward buffers of the workload: p lists of tensors, replica r
    filled with its own values (so a broadcast is visible)."""
    import torch
    p = p or cfg["p"]
    kind = cfg.get("buffers")
    out = []
    for r in range(p):
        row = []
        if kind == "llama":
            for j, s in enumerate(S.llama_buffers()):
                t = torch.empty(s, dtype=torch.float32, device=device)
                fill_(t, "uniform", cfg["seed"] + 7, 1000 + r * 64 + j)
                row.append(t)
        elif kind == "resnet50":
            for j, (_, shp, dt) in enumerate(S.resnet50_buffers()):
                if dt == "f32":
                    t = torch.empty(shp, dtype=torch.float32, device=device)
                    fill_(t.view(-1), "uniform", cfg["seed"] + 7, 1000 + r * 1000 + j)
                else:
                    t = torch.full(shp, r * 1000 + j, dtype=torch.int64, device=device)
                row.append(t)
        out.append(row)
    return out


def buffer_set_host(cfg, p=None):
    """The bytes of buffer_set's tensors, generated on the host: p lists of
    uint8 arrays, the same values buffer_set puts on the device."""
    p = p or cfg["p"]
    kind = cfg.get("buffers")
    out = []
    for r in range(p):
        row = []
        if kind == "llama":
            for j, s in enumerate(S.llama_buffers()):
                v = values_np("uniform", cfg["seed"] + 7, 1000 + r * 64 + j, np.arange(s))
                row.append(v.view(np.uint8).copy())
        elif kind == "resnet50":
            for j, (_, shp, dt) in enumerate(S.resnet50_buffers()):
                n = S.numel(shp)
                if dt == "f32":
                    v = values_np("uniform", cfg["seed"] + 7, 1000 + r * 1000 + j, np.arange(n))
                else:
                    v = np.full(n, r * 1000 + j, dtype=np.int64)
                row.append(v.view(np.uint8).copy())
        out.append(row)
    return out
