"""Seeded synthetic inputs for attention forward/backward (shared by tests, bench, smoke).

Holds no attention arithmetic: it only draws Q, K, V and dO.  The recipe: a CPU
``torch.Generator`` seeded with ``seed`` draws float32 standard normals in the order
Q [B,S,H,D], K [B,S,Hkv,D], V [B,S,Hkv,D], dO [B,S,H,D], each rounded to bfloat16
(round-to-nearest-even).  Layout BSHD, contiguous.
"""
from __future__ import annotations

import torch


def make_qkv_do(B: int, S: int, H: int, Hkv: int, D: int, seed: int = 0,
                dtype: torch.dtype = torch.bfloat16):
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    shapes = [(B, S, H, D), (B, S, Hkv, D), (B, S, Hkv, D), (B, S, H, D)]
    return tuple(torch.randn(s, generator=gen, dtype=torch.float32).to(dtype) for s in shapes)
