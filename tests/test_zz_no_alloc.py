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


def _fake_pointers(n=9):
    # Far apart (4 GiB), 16-byte aligned, never dereferenced: every check below fails
    # before any CUDA call.
    return [ctypes.c_void_p((i + 1) << 32) for i in range(n)]


def test_noalloc_refuses_a_shape_beyond_its_buffer(lib):
    """No GPU needed: the size check comes before any CUDA call."""
    limit = lib.attn_bwd_noalloc_max_bytes()
    assert limit == 16 << 20
    rows = limit // 8
    # The largest shape that fits needs the whole buffer, exactly.
    assert lib.attn_bwd_workspace_bytes(1, 1, rows) == limit
    assert lib.attn_bwd_workspace_bytes(1, 512, 4096) == limit
    # One head of rows + 128 query rows needs 8 * (rows + 128) bytes: too many.
    rc = lib.attn_bwd_noalloc(*_fake_pointers(), 1, 1, rows + 128, 64, 1, 0.125, None)
    assert rc == _codes()["GBATTN_ERR_SCRATCH"]
    assert b"fixed buffer" in lib.attn_strerror(rc)


def test_noalloc_reports_argument_errors_before_the_size(lib):
    """No GPU needed: on an oversized shape, a NULL pointer, an unsupported head_dim, a
    misaligned pointer or a bad scale is reported as attn_bwd reports it, not as the
    buffer's size."""
    c = _codes()
    rows = lib.attn_bwd_noalloc_max_bytes() // 8 + 128
    p = _fake_pointers()
    assert lib.attn_bwd_noalloc(None, *p[1:], 1, 1, rows, 64, 1, 0.125, None) == c["GBATTN_ERR_NULL"]
    assert lib.attn_bwd_noalloc(*p[:8], None, 1, 1, rows, 64, 1, 0.125, None) == c["GBATTN_ERR_NULL"]
    assert lib.attn_bwd_noalloc(*p, 1, 1, rows, 96, 1, 0.125, None) == c["GBATTN_ERR_HEAD_DIM"]
    assert lib.attn_bwd_noalloc(*p, 1, 1, rows, 256, 1, 0.125, None) == c["GBATTN_ERR_HEAD_DIM"]
    assert lib.attn_bwd_noalloc(*p, 0, 1, rows, 64, 1, 0.125, None) == c["GBATTN_ERR_DIMS"]
    odd = list(p)
    odd[3] = ctypes.c_void_p((4 << 32) + 8)
    assert lib.attn_bwd_noalloc(*odd, 1, 1, rows, 64, 1, 0.125, None) == c["GBATTN_ERR_ALIGN"]
    assert lib.attn_bwd_noalloc(*p, 1, 1, rows, 64, 1, -1.0, None) == c["GBATTN_ERR_SCALE"]
    same = list(p)
    same[6] = p[0]  # dq over q
    assert lib.attn_bwd_noalloc(*same, 1, 1, rows, 64, 1, 0.125, None) == c["GBATTN_ERR_ALIAS"]


def _noalloc(lib, q, k, v, o, lse, do, got, B, H, L, d, causal, scale):
    return lib.attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                do.data_ptr(), got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(),
                                B, H, L, d, int(causal), scale, torch.cuda.current_stream().cuda_stream)


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
        rc = _noalloc(lib, q, k, v, o, lse, do, got, B, H, L, d, causal, scale)
        assert rc == 0, lib.attn_strerror(rc)
        torch.cuda.synchronize()
        assert gb.attn_last_device_error() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(g).all(), name
            torch.testing.assert_close(g.float(), r.float(), atol=ATOL, rtol=RTOL, msg=name)


@pytest.mark.gpu
def test_noalloc_fills_its_whole_buffer_and_allocates_nothing(lib):
    """A shape whose workspace is the whole buffer (512 heads x 4096 rows: 2,097,152 padded
    query rows, 16 MiB), so the last rows of both halves of the buffer are written and read
    back; gradients against attn_bwd's.  The device's free memory is the same before and
    after a call (the first call, which looks up the buffer's address, is a warm-up)."""
    B, H, L, d, causal = 1, 512, 4096, 64, True
    assert lib.attn_bwd_workspace_bytes(B, H, L) == lib.attn_bwd_noalloc_max_bytes()
    g = torch.Generator(device="cuda").manual_seed(43)  # distinct data in every head
    q, k, v, do = (torch.randn(B, H, L, d, generator=g, device="cuda").half() for _ in range(4))
    scale = 1.0 / math.sqrt(d)
    o, lse = gb.attn_fwd(q, k, v, causal=causal, scale=scale)
    ref = gb.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    got = [torch.full_like(q, float("nan")) for _ in range(3)]
    assert _noalloc(lib, q, k, v, o, lse, do, got, B, H, L, d, causal, scale) == 0
    torch.cuda.synchronize()
    for g in got:
        g.fill_(float("nan"))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    assert _noalloc(lib, q, k, v, o, lse, do, got, B, H, L, d, causal, scale) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "the call changed the device's free memory"
    assert gb.attn_last_device_error() == 0
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert torch.isfinite(g).all(), name
        torch.testing.assert_close(g.float(), r.float(), atol=ATOL, rtol=RTOL, msg=name)
