"""The backward pass for callers that cannot allocate device memory (attn_bwd_noalloc).

Some callers of this library may not allocate device memory themselves: a plug-in inside
a host application that owns every device allocation, or a latency-critical path where
cudaMalloc, which may synchronise the device, is not allowed.  attn_bwd_noalloc gives them
the backward pass with its workspace in a fixed buffer compiled into the library.  These
tests call it through the C ABI twice in a row and compare every gradient with attn_bwd's
(the entry point with a caller-allocated workspace), within the backward tests' tolerance
(atol = rtol = 2e-2); they also check that an oversized shape is refused before anything
runs.  The file sorts last so that a run stopping at its first failure has run every
other test already.
"""
import ctypes
import math

import pytest
import torch

import scaled_dot_product_sdpa_gb300 as gb
from scaled_dot_product_sdpa_gb300 import inputs

ATOL = RTOL = 2e-2


@pytest.fixture(scope="module")
def lib():
    from scaled_dot_product_sdpa_gb300 import build
    return gb.load_library(build.build())


def _codes():
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "gbattn.h")).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"#define (GBATTN_\w+) \((-?\d+)\)", hdr)}


def test_noalloc_refuses_a_shape_beyond_its_buffer(lib):
    """No GPU needed: the size check comes before any CUDA call."""
    limit = lib.attn_bwd_noalloc_max_bytes()
    assert limit == 16 << 20
    rows = limit // 8
    fake = [ctypes.c_void_p(0x10000000 * (i + 1)) for i in range(9)]
    # One head of rows + 128 query rows needs 8 * (rows + 128) bytes: too many.
    rc = lib.attn_bwd_noalloc(*fake, 1, 1, rows + 128, 64, 1, 0.125, None)
    assert rc == _codes()["GBATTN_ERR_SCRATCH"]
    assert b"fixed buffer" in lib.attn_strerror(rc)


@pytest.mark.gpu
def test_noalloc_matches_attn_bwd_on_two_calls_in_a_row(lib):
    assert torch.cuda.is_available()
    shapes = [(2, 3, 300, 128, True, 41), (1, 4, 512, 64, False, 42)]
    for B, H, L, d, causal, seed in shapes:
        q, k, v = (t.cuda() for t in inputs.qkv(B, H, L, d, seed))
        do = inputs.upstream_grad(B, H, L, d, seed + 1, device="cuda")
        scale = 1.0 / math.sqrt(d)
        o, lse = gb.attn_fwd(q, k, v, causal=causal, scale=scale)
        ref = gb.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = lib.attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  do.data_ptr(), got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(),
                                  B, H, L, d, int(causal), scale, torch.cuda.current_stream().cuda_stream)
        assert rc == 0, lib.attn_strerror(rc)
        torch.cuda.synchronize()
        assert gb.attn_last_device_error() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(g).all(), name
            torch.testing.assert_close(g.float(), r.float(), atol=ATOL, rtol=RTOL, msg=name)
