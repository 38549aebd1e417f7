"""GPU parity of the key-range split (FLAG_SPLIT_KV, and the automatic plan where it picks
it) against the float64 oracle, through the C ABI.

A split query tile is computed by the two CTAs of a cluster over disjoint key ranges and
merged with the log-sum-exp weights of the two partial softmaxes -- exact for disjoint key
sets ("An Optimal Mapper Meets a Real GPU", "Experiment one"; STAGE_D.md, section 2,
"Merge"), so the gates are the forward pass's own: O within atol = rtol = 2e-2
elementwise, LSE within 1e-3 absolute.  Shapes put query tiles of 8 or more key tiles in
the schedule (only those are split); few CTAs make one cluster run several split tiles in
a row; ragged L, both masks, every supported head_dim, a forced rescale, other scales.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_sdpa_gb300 as gb
from scaled_dot_product_sdpa_gb300 import inputs

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


def _check(o, lse, o_ref, lse_ref, what):
    o = o.float().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    lse = lse.cpu().numpy().astype(np.float64).reshape(lse_ref.shape)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    bound = O_ATOL + O_RTOL * np.abs(o_ref)
    assert (err <= bound).all(), f"{what}: O max|err| {err.max():.3e}, {(err > bound).sum()} out of tolerance"
    lerr = np.abs(lse - lse_ref)
    assert lerr.max() <= LSE_ATOL, f"{what}: LSE max err {lerr.max():.3e}"


def _n_split(B, H, L, d, causal, grid):
    sched = gb.attn_debug_schedule(B, H, L, d, causal, grid, gb.FLAG_SPLIT_KV)
    n_items = B * H * math.ceil(L / 128) * (d // 256 if d > 256 else 1)
    return len({v for lst in sched for v in lst if v >= n_items})


def _case(B, H, L, d, causal, seed, grid=0, scale=None, q=None, k=None, v=None):
    sigma = 0.5 if d == 512 else 1.0
    if q is None:
        q, k, v = inputs.qkv(B, H, L, d, seed, sigma)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o, lse = gb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, flags=gb.FLAG_SPLIT_KV,
                         grid_limit=grid)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.sdpa_fwd(q, k, v, causal, float(np.float32(scale)))
    _check(o, lse, o_ref, lse_ref, f"split {B}x{H}x{L}x{d} causal={causal} grid={grid}")
    return o, lse


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,L,d", [(1, 2, 1024, 64), (1, 3, 1100, 128), (1, 2, 2048, 512), (2, 1, 1500, 64),
                                      (1, 2, 1537, 128)])
def test_split_matches_oracle(B, H, L, d, causal):
    grid = 152 if d < 512 else 0
    assert _n_split(B, H, L, d, causal, 152) > 0, "the shape must contain split tiles"
    _case(B, H, L, d, causal, seed=L + d + int(causal), grid=grid)


def _max_split_per_cluster(B, H, L, d, causal, grid):
    sched = gb.attn_debug_schedule(B, H, L, d, causal, grid, gb.FLAG_SPLIT_KV)
    n_items = B * H * math.ceil(L / 128) * (d // 256 if d > 256 else 1)
    return max(sum(1 for v in sched[2 * c] if v >= n_items) for c in range(grid // 2))


@pytest.mark.parametrize("B,H,L,d,grid", [(1, 4, 4096, 64, 152), (1, 4, 4096, 128, 152), (1, 1, 4096, 512, 64)])
def test_split_tiles_in_a_row_on_one_cluster(B, H, L, d, grid):
    """Schedules where a cluster runs two split tiles back to back before its plain ones
    (the handover's barrier phases advance twice, the receive area is reused)."""
    assert _max_split_per_cluster(B, H, L, d, True, grid) >= 2
    _case(B, H, L, d, True, seed=grid + d, grid=grid)


@pytest.mark.parametrize("grid", [1, 2, 6])
@pytest.mark.parametrize("d", [64, 128, 512])
def test_split_flag_with_few_ctas(d, grid):
    """Few CTAs (the launch rounds up to an even count): splitting does not pay there, so
    the cluster launch runs plain items only; results must not change."""
    for causal in (True, False):
        _case(1, 2, 640, d, causal, seed=grid * 10 + d, grid=grid)


@pytest.mark.parametrize("d", [64, 128, 512])
def test_split_forced_rescale_and_other_scales(d):
    """Growing logits (the lazy rescale runs in both parts) and scales far from 1/sqrt(d)."""
    B, H, L = 1, 2, 1024
    q, k, v = inputs.qkv(B, H, L, d, seed=99, sigma=0.5 if d == 512 else 1.0)
    q = q.abs()
    ramp = torch.linspace(0, 6 * math.sqrt(64 / d), L).view(1, 1, L, 1)
    k = (k.float() * 0.2 + ramp).half()
    for causal in (False, True):
        _case(B, H, L, d, causal, 0, q=q, k=k, v=v)
    for scale in (1.0, 0.03):
        _case(B, H, L, d, True, seed=7, scale=scale)


def test_split_is_chosen_and_matches_on_a_long_causal_head():
    """4 heads x 4096 causal, head_dim 128: the automatic plan takes the split kernel;
    sampled rows against the oracle, every row finite and bounded by max |v|; repeated
    calls and a CUDA-graph replay give the same bits."""
    B, H, L, d = 1, 4, 4096, 128
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert gb.attn_debug_plan(B, H, L, d, True, sm)["kind"] == 3
    q, k, v = inputs.qkv(B, H, L, d, seed=4242)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = gb.attn_fwd(qd, kd, vd, causal=True)
    o2, l2 = gb.attn_fwd(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    assert torch.isfinite(o).all() and o.float().abs().max() <= v.float().abs().max() * (1 + 2e-3)
    rng = np.random.default_rng(1)
    picks = {0, 127, 128, 1023, 1024, 2047, 2048, L - 129, L - 128, L - 1} | set(rng.integers(0, L, 20).tolist())
    rows = sorted(h * L + i for h in range(B * H) for i in picks)
    o_ref, lse_ref, _ = oracle.sdpa_fwd_rows(q, k, v, True, float(np.float32(1.0 / math.sqrt(d))), rows)
    sel = torch.tensor(rows)
    _check(o.reshape(-1, d).cpu()[sel], lse.reshape(-1).cpu()[sel], o_ref, lse_ref, "auto split, sampled rows")
    og, lg = torch.empty_like(o), torch.empty_like(lse)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gb.attn_fwd(qd, kd, vd, causal=True, o=og, lse=lg, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            gb.attn_fwd(qd, kd, vd, causal=True, o=og, lse=lg, stream=s)
        og.zero_()
        g.replay()
    s.synchronize()
    assert torch.equal(og, o) and torch.equal(lg, lse)
