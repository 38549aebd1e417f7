"""GPU parity of the backward pass (attn_bwd through the C ABI) against the float64
oracle's gradients ("Validating Memory-Optimal Transformer Kernels on Real Hardware",
section 4).  The forward pass's o and lse come from attn_fwd (as a training step would use
them); the oracle differentiates the exact definition.  Gate: atol = rtol = 2e-2
elementwise on dq, dk, dv (the first page's FP16-in / FP32-accumulate gate): P and dS are
rounded to fp16 before their products, as the forward pass rounds P.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_sdpa_gb300 as gb
from scaled_dot_product_sdpa_gb300 import inputs

pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from scaled_dot_product_sdpa_gb300 import build
    gb.load_library(build.build())
    assert gb.attn_last_device_error() == 0
    yield
    assert gb.attn_last_device_error() == 0, "a kernel recorded a device-side timeout"


def _grads(B, H, L, d, causal, seed, sigma=1.0):
    q, k, v = inputs.qkv(B, H, L, d, seed, sigma)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(B, H, L, d, generator=g).half()
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(d)
    o, lse = gb.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = gb.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    ref = oracle.sdpa_bwd(q, k, v, do, causal, float(np.float32(scale)))
    return (dq, dk, dv), ref


def _check(got, ref, what):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = g.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all(), f"{what} {name}: non-finite"
        err = np.abs(g - r)
        bound = ATOL + RTOL * np.abs(r)
        assert (err <= bound).all(), (f"{what} {name}: max|err| {err.max():.3e} (max|ref| {np.abs(r).max():.3e}), "
                                      f"{(err > bound).sum()} out of tolerance")


@pytest.mark.parametrize("B,H,L,d,causal", [
    (1, 2, 128, 64, False), (1, 2, 128, 64, True), (2, 3, 300, 64, True), (1, 2, 257, 128, True),
    (1, 4, 512, 128, False), (1, 1, 1, 64, False), (1, 2, 77, 128, False), (1, 16, 512, 64, True),
])
def test_bwd_matches_oracle(B, H, L, d, causal):
    got, ref = _grads(B, H, L, d, causal, seed=L + d + int(causal))
    _check(got, ref, f"{B}x{H}x{L}x{d} causal={causal}")


def test_bwd_is_deterministic_and_replays_from_a_graph():
    B, H, L, d = 1, 4, 640, 128
    q, k, v = (t.cuda() for t in inputs.qkv(B, H, L, d, 3))
    do = torch.randn(B, H, L, d, generator=torch.Generator().manual_seed(4)).half().cuda()
    o, lse = gb.attn_fwd(q, k, v, causal=True)
    a = gb.attn_bwd(q, k, v, o, lse, do, causal=True)
    b = gb.attn_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    outs = [torch.empty_like(q) for _ in range(3)]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gb.attn_bwd(q, k, v, o, lse, do, causal=True, dq=outs[0], dk=outs[1], dv=outs[2], stream=s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            gb.attn_bwd(q, k, v, o, lse, do, causal=True, dq=outs[0], dk=outs[1], dv=outs[2], stream=s)
        for t in outs:
            t.zero_()
        g.replay()
    s.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(outs, a))


@pytest.mark.parametrize("B,H,L,d,causal", [
    (2, 40, 512, 64, True),      # 320 items per kernel: every CTA of the persistent grid runs two or more
    (1, 160, 300, 128, False),   # ragged L (300 = 2 x 128 + 44 = 4 x 64 + 44), 480 items
    (2, 48, 1000, 128, True),    # causal, ragged, uneven item lengths across the snake order
])
def test_bwd_many_items_per_cta(B, H, L, d, causal):
    """Workloads with more items than SMs: each persistent CTA carries its pipeline state
    (ring stages, tensor-memory buffers, barrier phases) across items.  Six sampled heads
    are compared with the oracle; every head is checked for finiteness."""
    seed = 97 + L + d
    q, k, v = inputs.qkv(B, H, L, d, seed)
    do = inputs.upstream_grad(B, H, L, d, seed + 1)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(d)
    o, lse = gb.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    got = gb.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert all(torch.isfinite(t).all() for t in got)
    BH = B * H
    heads = sorted(set(np.random.default_rng(seed).integers(0, BH, 6).tolist()) | {0, BH - 1})
    pick = lambda t: t.reshape(BH, L, d)[heads].reshape(1, len(heads), L, d)
    ref = oracle.sdpa_bwd(pick(q), pick(k), pick(v), pick(do), causal, float(np.float32(scale)))
    _check([pick(t.cpu()) for t in got], ref, f"{B}x{H}x{L}x{d} causal={causal}")


def test_bwd_workspace_contents_do_not_matter():
    """The workspace is written before it is read: a caller's workspace full of NaN gives the
    same gradients, bit for bit, as a fresh one."""
    B, H, L, d = 2, 3, 300, 128
    q, k, v = (t.cuda() for t in inputs.qkv(B, H, L, d, 21))
    do = inputs.upstream_grad(B, H, L, d, 22, device="cuda")
    o, lse = gb.attn_fwd(q, k, v, causal=True)
    ref = gb.attn_bwd(q, k, v, o, lse, do, causal=True)
    ws = torch.full((gb.attn_bwd_workspace_bytes(B, H, L) // 4,), float("nan"), device="cuda")
    got = gb.attn_bwd(q, k, v, o, lse, do, causal=True, workspace=ws)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(got, ref))
    with pytest.raises(ValueError):
        gb.attn_bwd(q, k, v, o, lse, do, causal=True, workspace=ws[:16])


def test_bwd_long_sequence_matches_oracle():
    """One head of 4096 rows, causal: the longest items run 32 steps (every ring wraps many
    times within an item, and the dQ items of the last query tiles stream every key tile)."""
    B, H, L, d = 1, 1, 4096, 128
    got, ref = _grads(B, H, L, d, True, seed=4096)
    _check(got, ref, f"{B}x{H}x{L}x{d} causal")
