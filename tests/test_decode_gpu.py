"""GPU parity of decode (attn_decode through the C ABI) against the float64 oracle.

Decode is one query row per (b, h) against all L cached keys ("Validating Memory-Optimal
Transformer Kernels on Real Hardware", section 5, "Paper III: Inference (Decode)").
Tolerances as for the forward pass: O within atol = rtol = 2e-2 elementwise, LSE within
1e-3 absolute.  Shapes cover one key, a ragged last key tile, every head_dim, clusters of
1 to 16 CTAs per head including CTAs whose key range is empty, and the two decode
workloads at full size (sampled heads against the oracle, the rest by properties).
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_sdpa_gb300 as gb
from scaled_dot_product_sdpa_gb300 import inputs
from scaled_dot_product_sdpa_gb300.configs import DECODE_WORKLOADS

pytestmark = pytest.mark.gpu

O_ATOL = O_RTOL = 2e-2
LSE_ATOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from scaled_dot_product_sdpa_gb300 import build
    gb.load_library(build.build())
    assert gb.attn_last_device_error() == 0
    yield
    assert gb.attn_last_device_error() == 0, "a kernel recorded a device-side timeout"


def _check(o, lse, o_ref, lse_ref, what=""):
    o = o.float().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    lse = lse.cpu().numpy().astype(np.float64).reshape(lse_ref.shape)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    bound = O_ATOL + O_RTOL * np.abs(o_ref)
    assert (err <= bound).all(), f"{what}: O max|err| {err.max():.3e}, {(err > bound).sum()} out of tolerance"
    lerr = np.abs(lse - lse_ref)
    assert lerr.max() <= LSE_ATOL, f"{what}: LSE max err {lerr.max():.3e}"


@pytest.mark.parametrize("B,H,L,d", [
    (1, 1, 1, 128),       # one key
    (1, 1, 5, 64),        # one partial key tile
    (2, 3, 300, 64),      # two CTAs per head, ragged last tile
    (1, 4, 777, 128),     # ragged, several CTAs per head
    (1, 1, 65, 512),      # head_dim 512, an empty CTA range
    (1, 2, 1000, 256),    # 16 CTAs per head (or 8 where 16 cannot be launched)
    (4, 8, 4096, 128),    # many heads
    (1, 1, 100000, 64),   # long sequence, the widest cluster
])
def test_decode_matches_oracle(B, H, L, d):
    q, k, v = inputs.decode_qkv(B, H, L, d, seed=31 + L + d)
    scale = 1.0 / np.sqrt(d)
    o, lse = gb.attn_decode(q.cuda(), k.cuda(), v.cuda(), scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(q, k, v, float(np.float32(scale)))
    _check(o, lse, o_ref, lse_ref, f"{B}x{H}x{L}x{d}")


def test_decode_large_logits_and_shifted_keys():
    """sigma 4 inputs (sharp softmax, logits far from zero) and keys shifted by a constant
    vector: the running maximum and the cross-CTA merge must keep the result exact."""
    B, H, L, d = 1, 2, 3000, 128
    q, k, v = inputs.decode_qkv(B, H, L, d, seed=5, sigma=4.0)
    k = (k.float() + 3.0).half()
    o, lse = gb.attn_decode(q.cuda(), k.cuda(), v.cuda(), scale=0.125)
    o_ref, lse_ref = oracle.decode(q, k, v, 0.125)
    _check(o, lse, o_ref, lse_ref, "sharp")


def test_decode_is_deterministic_and_stream_ordered():
    q, k, v = (t.cuda() for t in inputs.decode_qkv(2, 4, 5000, 128, seed=8))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = gb.attn_decode(q, k, v, stream=s)
        o2, l2 = gb.attn_decode(q, k, v, stream=s)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_replays_from_a_cuda_graph():
    q, k, v = (t.cuda() for t in inputs.decode_qkv(1, 4, 9000, 64, seed=9))
    o = torch.empty(1, 4, 64, dtype=torch.float16, device="cuda")
    lse = torch.empty(1, 4, dtype=torch.float32, device="cuda")
    gb.attn_decode(q, k, v, o=o, lse=lse)
    torch.cuda.synchronize()
    ref_o, ref_l = o.clone(), lse.clone()
    o.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            gb.attn_decode(q, k, v, o=o, lse=lse, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


@pytest.mark.parametrize("name", sorted(DECODE_WORKLOADS))
def test_decode_workloads_full_size(name):
    """The decode workloads at full size: six sampled heads against the oracle; every head
    finite with |o| bounded by max |v| (a convex combination of value rows)."""
    w = DECODE_WORKLOADS[name]
    q, k, v = inputs.decode_qkv(w.B, w.H, w.L, w.d, w.seed, w.sigma, device="cuda", draw_on_device=True)
    o, lse = gb.attn_decode(q, k, v, scale=w.scale)
    torch.cuda.synchronize()
    BH = w.B * w.H
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    vmax = v.abs().amax(dim=(2, 3)).float().reshape(BH)
    assert (o.float().abs().reshape(BH, -1).amax(1) <= vmax * (1 + 2e-3) + 1e-6).all()
    heads = sorted(set(np.random.default_rng(w.seed).integers(0, BH, 6).tolist()))
    qh = q.reshape(BH, w.d)[heads].cpu().reshape(1, len(heads), 1, w.d)
    kh = k.reshape(BH, w.L, w.d)[heads].cpu().reshape(1, len(heads), w.L, w.d)
    vh = v.reshape(BH, w.L, w.d)[heads].cpu().reshape(1, len(heads), w.L, w.d)
    o_ref, lse_ref = oracle.decode(qh, kh, vh, float(np.float32(w.scale)))
    _check(o.reshape(BH, w.d)[heads], lse.reshape(BH)[heads], o_ref, lse_ref, name)


@pytest.mark.parametrize("B,H,L,d", [
    (1, 1, 19457, 128),   # 32 clusters of 8 CTAs per head, the last ones without keys
    (1, 2, 40000, 128),   # several clusters per head, ragged last tile
    (1, 1, 70000, 256),   # head_dim 256: clusters of 8
    (1, 12, 5000, 128),   # clusters of two CTAs, 12 per head, ragged last tile
    (2, 3, 7000, 64),     # clusters of two CTAs, 25 per head, ragged last tile
])
def test_decode_grouped_and_single_cluster_agree_with_oracle(B, H, L, d):
    """Few heads: with a workspace each head's keys are split over several clusters and the
    clusters' partials merged by a second kernel; without one, one cluster per head.  Both
    match the oracle."""
    plan = gb.attn_debug_decode_plan(B, H, L, d, torch.cuda.get_device_properties(0).multi_processor_count,
                                     grouped=True)
    assert plan["groups"] > 1
    q, k, v = inputs.decode_qkv(B, H, L, d, seed=77 + L + d)
    scale = 1.0 / np.sqrt(d)
    o_ref, lse_ref = oracle.decode(q, k, v, float(np.float32(scale)))
    for grouped in (True, False):
        o, lse = gb.attn_decode(q.cuda(), k.cuda(), v.cuda(), scale=scale, grouped=grouped)
        torch.cuda.synchronize()
        _check(o, lse, o_ref, lse_ref, f"{B}x{H}x{L}x{d} grouped={grouped}")
