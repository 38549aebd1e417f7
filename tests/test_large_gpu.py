"""GPU parity on tensors of more than 2^31 elements (more than 4 GiB of fp16 each), so that
every byte offset past the first 2^31 elements needs 64-bit arithmetic: the TMA
coordinates of the query, key and value tiles, the O stores, the LSE rows, (in the
backward pass) the O rows and the row-statistics workspace, and (in decode) the key and
value streams of heads past the 2^31st element.

The inputs repeat one seeded block of 9 heads along the head axis (copies, no
arithmetic), so the oracle needs only that block: head h of the big tensors is head
h % 9 of the block.  A 32-bit wrap of an element offset would move a head by 2^31 / (L d)
heads -- 1024 for the forward shape, 16384 for the backward one, neither a multiple of 9
-- onto different data, so the sampled heads past the 2^31st element fail on it.  O and
the gradients are pre-filled with NaN so that a store sent elsewhere is seen too.
Tolerances are those of the other parity tests ("An Optimal Mapper Meets a Real GPU",
"Ground rules": atol = rtol = 2e-2; LSE 1e-3 absolute).
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
LSE_ATOL = 1e-3
PERIOD = 9


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from scaled_dot_product_sdpa_gb300 import build
    gb.load_library(build.build())
    assert gb.attn_last_device_error() == 0
    yield
    assert gb.attn_last_device_error() == 0, "a kernel recorded a device-side timeout"


def _tile_heads(block: torch.Tensor, H: int) -> torch.Tensor:
    """[1, H, L, d] on the GPU whose head h is head h % PERIOD of the CPU block."""
    assert H % PERIOD == 0
    _, P, L, d = block.shape
    return block.cuda().unsqueeze(1).expand(1, H // PERIOD, P, L, d).reshape(1, H, L, d)


def _check(got, ref, atol, rtol, what):
    got = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite (an unwritten or misplaced store)"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    assert (err <= bound).all(), f"{what}: max|err| {err.max():.3e}, {(err > bound).sum()} out of tolerance"


def test_fwd_beyond_2_31_elements_matches_oracle():
    L, d, H = 16384, 128, 1035  # 1035 * 16384 * 128 = 2.17e9 elements per tensor
    assert H * L * d > 2 ** 31
    seed = 71
    bq, bk, bv = inputs.qkv(1, PERIOD, L, d, seed)
    q, k, v = (_tile_heads(t, H) for t in (bq, bk, bv))
    scale = 1.0 / math.sqrt(d)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((1, H, L), float("nan"), device="cuda")
    gb.attn_fwd(q, k, v, causal=True, scale=scale, o=o, lse=lse)
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed)
    rows_in_head = sorted({0, 127, 128, L - 1} | set(rng.integers(0, L, 8).tolist()))
    for h in (0, 1023, 1024, 1029, H - 1):  # heads from 1024 on start past element 2^31
        ref_rows = [(h % PERIOD) * L + i for i in rows_in_head]
        o_ref, lse_ref, _ = oracle.sdpa_fwd_rows(bq, bk, bv, True, float(np.float32(scale)), ref_rows)
        sel = torch.tensor(rows_in_head, device="cuda")
        _check(o[0, h].index_select(0, sel), o_ref, ATOL, RTOL, f"O of head {h}")
        _check(lse[0, h].index_select(0, sel), lse_ref, LSE_ATOL, 0.0, f"LSE of head {h}")
    del q, k, v, o, lse
    torch.cuda.empty_cache()


def test_bwd_beyond_2_31_elements_matches_oracle():
    L, d, H = 1024, 128, 16389  # 16389 * 1024 * 128 = 2.15e9 elements per tensor
    assert H * L * d > 2 ** 31
    seed = 73
    bq, bk, bv = inputs.qkv(1, PERIOD, L, d, seed)
    bdo = inputs.upstream_grad(1, PERIOD, L, d, seed + 1)
    q, k, v, do = (_tile_heads(t, H) for t in (bq, bk, bv, bdo))
    scale = 1.0 / math.sqrt(d)
    o, lse = gb.attn_fwd(q, k, v, causal=True, scale=scale)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    gb.attn_bwd(q, k, v, o, lse, do, causal=True, scale=scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    heads = (16384, H - 1)  # both start past element 2^31
    ref = oracle.sdpa_bwd(*(t[:, sorted({h % PERIOD for h in heads})] for t in (bq, bk, bv, bdo)), True,
                          float(np.float32(scale)))
    order = sorted({h % PERIOD for h in heads})
    for h in heads:
        j = order.index(h % PERIOD)
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            _check(g[0, h], r[0, j], ATOL, RTOL, f"{name} of head {h}")
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


@pytest.mark.parametrize("grouped", [True, False], ids=["grouped", "one_cluster_per_head"])
def test_decode_beyond_2_31_elements_matches_oracle(grouped):
    """Decode over a key/value cache of 18 heads x 2^20 keys x 128 (2.4e9 elements each).
    The cache tiles a seeded block of 9 heads x 2^17 keys 8 times along the keys and twice
    along the heads: every key of a head appears 8 times, which leaves O unchanged and adds
    ln 8 to the LSE exactly.  A 32-bit wrap moves a head by 16 heads, onto other data."""
    Lb, reps, d, H = 1 << 17, 8, 128, 18
    L = Lb * reps
    assert H * L * d > 2 ** 31
    bq, bk, bv = inputs.decode_qkv(1, PERIOD, Lb, d, seed=79)
    q = _tile_heads(bq, H)
    k, v = (_tile_heads(t, H).view(1, H, 1, Lb, d).expand(1, H, reps, Lb, d).reshape(1, H, L, d) for t in (bk, bv))
    scale = 1.0 / math.sqrt(d)
    o = torch.full((1, H, d), float("nan"), device="cuda", dtype=torch.float16)
    lse = torch.full((1, H), float("nan"), device="cuda")
    gb.attn_decode(q, k, v, scale=scale, o=o, lse=lse, grouped=grouped)
    torch.cuda.synchronize()
    heads = (0, 16, 17)  # heads 16 and 17 start past element 2^31
    o_ref, lse_ref = oracle.decode(bq, bk, bv, float(np.float32(scale)), heads=[h % PERIOD for h in heads])
    for j, h in enumerate(heads):
        _check(o[0, h], o_ref[j], ATOL, RTOL, f"decode O of head {h}")
        _check(lse[0, h:h + 1], lse_ref[j:j + 1] + math.log(reps), LSE_ATOL, 0.0, f"decode LSE of head {h}")
    del q, k, v, o, lse
    torch.cuda.empty_cache()
