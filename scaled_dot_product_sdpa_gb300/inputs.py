"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no attention arithmetic: it only draws Q, K and V.  Recipe (the same
for every caller): a CPU ``torch.Generator`` seeded with ``seed`` draws Q, then K, then
V, each as ``torch.randn(B, H, L, d, dtype=float32) * sigma`` rounded to fp16.  Inputs
are i.i.d. normal, as in the workloads of "An Optimal Mapper Meets a Real GPU",
"Experiment one" (Cases A-D); no dataset is involved.

The upstream gradient dO of the backward pass is drawn the same way by
``upstream_grad`` (its own generator, seeded with ``seed``; standard normal, fp16).

Decode inputs (one query row per head, a long key/value sequence) follow the same recipe
with q drawn as [B, H, 1, d]; for very long sequences the draw may run on the GPU (a
CUDA ``torch.Generator`` seeded the same way), so that no multi-GB tensor is drawn on the
host -- every consumer, the oracle included, then reads the values back from the device.
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


def decode_qkv(B: int, H: int, L: int, d: int, seed: int, sigma: float = 1.0, device="cpu", draw_on_device=False):
    """Return fp16 (q [B, H, 1, d], k [B, H, L, d], v [B, H, L, d]) on `device`, drawn in that
    order; on the device's own generator when `draw_on_device`."""
    gdev = torch.device(device) if draw_on_device else torch.device("cpu")
    g = torch.Generator(device=gdev).manual_seed(int(seed))
    out = []
    for shape in ((B, H, 1, d), (B, H, L, d), (B, H, L, d)):
        t = torch.randn(*shape, generator=g, dtype=torch.float32, device=gdev) * float(sigma)
        out.append(t.to(torch.float16).to(device).contiguous())
    return tuple(out)


def upstream_grad(B: int, H: int, L: int, d: int, seed: int, device="cpu"):
    """Return an fp16 upstream gradient dO [B, H, L, d], standard normal, on `device`."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    return torch.randn(B, H, L, d, generator=g, dtype=torch.float32).to(torch.float16).to(device).contiguous()
