"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no attention arithmetic: it only draws Q, K and V.  Recipe (the same
for every caller): a CPU ``torch.Generator`` seeded with ``seed`` draws Q, then K, then
V, each as ``torch.randn(B, H, L, d, dtype=float32) * sigma`` rounded to fp16.  Inputs
are i.i.d. normal, as in the workloads of "An Optimal Mapper Meets a Real GPU",
"Experiment one" (Cases A-D); no dataset is involved.
"""
from __future__ import annotations

import torch


def qkv(B: int, H: int, L: int, d: int, seed: int, sigma: float = 1.0, device="cpu"):
    """Return fp16 (q, k, v), each [B, H, L, d] and contiguous, on `device`."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    out = []
    for _ in range(3):
        t = torch.randn(B, H, L, d, generator=g, dtype=torch.float32) * float(sigma)
        out.append(t.to(torch.float16).to(device).contiguous())
    return tuple(out)
