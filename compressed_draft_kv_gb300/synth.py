"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws numbers: N(0, 1) tensors from a seeded CPU torch
generator, rounded to the element type the library computes in, plus the
workload shapes.  It holds none of the attention or memory arithmetic.
"""
from __future__ import annotations

import hashlib

import torch

# Workload shapes: Llama-3.2-3B / Llama-3.1-8B attention geometry (24q/8kv and
# 32q/8kv heads, head_dim 128), prefixes up to 32K, S sink, W window, r tokens
# per slot, L_draft draft steps per speculative iteration.
WORKLOADS = {
    "tiny_f32": dict(Hq=8, Hkv=2, D=64, layers=1, batch=1, prefix=2048, S=4, W=256, r=256,
                     dtype="f32", seed=0, steps=1),
    "draft3b_1layer_8k": dict(Hq=24, Hkv=8, D=128, layers=1, batch=1, prefix=8192, S=4, W=1024, r=512,
                              dtype="bf16", seed=1, steps=5),
    "draft3b_28l_b8": dict(Hq=24, Hkv=8, D=128, layers=28, batch=8, prefix=32768, S=4, W=1024, r=512,
                           dtype="bf16", seed=2, steps=5),
    # the pages' decoding setting: one sequence at a time
    "draft3b_28l_b1": dict(Hq=24, Hkv=8, D=128, layers=28, batch=1, prefix=32768, S=4, W=1024, r=512,
                           dtype="bf16", seed=7, steps=5),
    "verify8b_32k": dict(Hq=32, Hkv=8, D=128, layers=32, batch=4, prefix=32768, Lq=6,
                         dtype="bf16", seed=3),
    # the pages' own memory configuration: S = W = 128 and nominal 4x / 8x
    # compression (r = 4 / 8), on the 3B-draft attention shape at 32K
    "paper_s128_w128_r4": dict(Hq=24, Hkv=8, D=128, layers=28, batch=8, prefix=32768, S=128, W=128, r=4,
                               dtype="bf16", seed=5, steps=5),
    "paper_s128_w128_r8": dict(Hq=24, Hkv=8, D=128, layers=28, batch=8, prefix=32768, S=128, W=128, r=8,
                               dtype="bf16", seed=6, steps=5),
    # sliding-window attention, the pages' SWA baseline: no sink, no slots (r
    # beyond the longest sequence), a 1,024-token window, on the 3B-draft shape
    "swa_w1024": dict(Hq=24, Hkv=8, D=128, layers=28, batch=8, prefix=32768, S=0, W=1024, r=1 << 20,
                      dtype="bf16", seed=8, steps=5),
    "draft8b_b32_ragged": dict(Hq=32, Hkv=8, D=128, layers=32, batch=32, prefix_lo=16384, prefix_hi=32768,
                               S=4, W=2048, r=1024, dtype="bf16", seed=4, steps=8),
}


def _seed(*parts) -> int:
    h = hashlib.sha256(("/".join(str(p) for p in parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def normal(shape, dtype: str, *stream, scale: float = 1.0) -> torch.Tensor:
    """N(0, scale^2) on the CPU from a generator seeded by ``stream``, rounded
    (round-to-nearest-even) to ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(_seed(*stream))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(torch_dtype(dtype))


def ragged_prefixes(batch: int, lo: int, hi: int, seed) -> list[int]:
    """Prefix lengths uniform on the integers [lo, hi]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(_seed("prefix", seed))
    return [int(x) for x in torch.randint(lo, hi + 1, (batch,), generator=g)]
