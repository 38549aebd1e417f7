"""Host-side checks of the C ABI that need no GPU: the library builds for sm_103a, loads,
exports every entry point include/gbattn.h declares, and rejects bad arguments with the
documented codes before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbattn.h")


@pytest.fixture(scope="module")
def lib():
    from scaled_dot_product_sdpa_gb300 import build as b
    path = b.build()
    import scaled_dot_product_sdpa_gb300 as g
    return g.load_library(path)


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:int|const char \*)\s*(\w+)\(", text, re.M)))


def _codes():
    text = open(HEADER).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"#define (GBATTN_\w+) \(?(-?\d+)\)?", text)}


def test_header_declares_the_scope_entry_points():
    names = _declared()
    for required in ("attn_fwd", "attn_last_device_error", "attn_strerror", "attn_debug_scores"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    so = os.path.join(ROOT, "scaled_dot_product_sdpa_gb300", "libgbattn.so")
    out = subprocess.run(["nm", "-D", "--defined-only", so], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, re.M))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    for n in _declared():
        assert hasattr(lib, n)


def test_strerror_covers_every_code(lib):
    for name, code in _codes().items():
        if name.startswith("GBATTN_FLAG"):
            continue
        msg = lib.attn_strerror(code).decode()
        assert msg and "unknown" not in msg, (name, code)
    assert "unknown" in lib.attn_strerror(12345).decode()
    assert lib.attn_version() >= 100


# Fake, 16-byte-aligned, non-overlapping "device" addresses: validation rejects the call
# before any CUDA API is reached, so nothing is dereferenced.
Q, K, V, O, LSE = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def _fwd(lib, q=Q, k=K, v=V, o=O, lse=LSE, B=1, H=2, L=128, d=64, causal=0, scale=0.125, flags=0, grid=0):
    return lib.attn_fwd_ex(q, k, v, o, lse, B, H, L, d, causal, scale, None, flags, grid)


def test_rejects_null_pointers(lib):
    codes = _codes()
    for kw in ("q", "k", "v", "o", "lse"):
        assert _fwd(lib, **{kw: 0}) == codes["GBATTN_ERR_NULL"]


@pytest.mark.parametrize("B,H,L", [(0, 1, 1), (1, 0, 1), (1, 1, 0), (-1, 1, 1), (1 << 16, 1 << 16, 1)])
def test_rejects_bad_dims(lib, B, H, L):
    assert _fwd(lib, B=B, H=H, L=L) == _codes()["GBATTN_ERR_DIMS"]


@pytest.mark.parametrize("d", [0, 16, 32, 96, 100, 192, 1024])
def test_rejects_unsupported_head_dim(lib, d):
    assert _fwd(lib, d=d) == _codes()["GBATTN_ERR_HEAD_DIM"]


def test_smem_p_only_up_to_128(lib):
    assert _fwd(lib, d=256, flags=1) == _codes()["GBATTN_ERR_HEAD_DIM"]


def test_flag_combinations(lib):
    c = _codes()
    assert _fwd(lib, d=512, flags=4) == c["GBATTN_ERR_HEAD_DIM"]
    for bad in (4 | 2, 4 | 1, 32, 64, 16 | 1, 16 | 2, 16 | 4, 16 | 8):
        assert _fwd(lib, flags=bad) == c["GBATTN_ERR_FLAGS"], bad
    assert _fwd(lib, flags=8) == c["GBATTN_ERR_HEAD_DIM"]  # the head_dim split is for d = 512 only
    for bad in (8 | 1, 8 | 2, 8 | 4):
        assert _fwd(lib, d=512, flags=bad) == c["GBATTN_ERR_FLAGS"], bad
    assert _fwd(lib, d=256, flags=16) == c["GBATTN_ERR_HEAD_DIM"]  # no key-range split at d = 256


@pytest.mark.parametrize("kw", ["q", "k", "v", "o", "lse"])
def test_rejects_misaligned(lib, kw):
    base = {"q": Q, "k": K, "v": V, "o": O, "lse": LSE}[kw]
    assert _fwd(lib, **{kw: base + 8}) == _codes()["GBATTN_ERR_ALIGN"]


@pytest.mark.parametrize("scale", [0.0, -0.5, float("inf"), float("nan")])
def test_rejects_bad_scale(lib, scale):
    assert _fwd(lib, scale=scale) == _codes()["GBATTN_ERR_SCALE"]


def test_rejects_aliased_outputs(lib):
    a = _codes()["GBATTN_ERR_ALIAS"]
    assert _fwd(lib, o=Q) == a
    assert _fwd(lib, o=V + 256) == a          # overlaps the tail of v
    assert _fwd(lib, lse=O + 1024) == a       # lse inside o
    assert _fwd(lib, lse=K) == a


def test_valid_call_without_gpu_fails_cleanly(lib):
    """Past validation, a machine without a usable sm_103 device gets an error code.
    Only run where no GPU is visible: the addresses above are fake."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the fake addresses must never reach a launch")
    rc = _fwd(lib)
    assert rc in (_codes()["GBATTN_ERR_LAUNCH"], _codes()["GBATTN_ERR_DEVICE"])


def test_debug_scores_validation(lib):
    c = _codes()
    assert lib.attn_debug_scores(0, K, O, 1, 1, 128, 64, 0.1, None) == c["GBATTN_ERR_NULL"]
    assert lib.attn_debug_scores(Q, K, O, 1, 1, 128, 48, 0.1, None) == c["GBATTN_ERR_HEAD_DIM"]
    assert lib.attn_debug_scores(Q, K, O + 4, 1, 1, 128, 64, 0.1, None) == c["GBATTN_ERR_ALIGN"]
    assert lib.attn_debug_scores(Q, K, Q, 1, 1, 128, 64, 0.1, None) == c["GBATTN_ERR_ALIAS"]


WS = 0x60000000  # fake, 256-byte-aligned device workspace


def _host(lib, q=Q, k=K, v=V, o=O, lse=LSE, B=1, H=2, L=128, d=64, scale=0.125, ws=WS, ws_bytes=1 << 30):
    return lib.attn_fwd_host(q, k, v, o, lse, B, H, L, d, 1, scale, ws, ws_bytes, None)


def test_host_entry_validation(lib):
    c = _codes()
    for kw in ("q", "k", "v", "o", "lse", "ws"):
        assert _host(lib, **{kw: 0}) == c["GBATTN_ERR_NULL"]
    assert _host(lib, d=96) == c["GBATTN_ERR_HEAD_DIM"]
    assert _host(lib, L=0) == c["GBATTN_ERR_DIMS"]
    assert _host(lib, scale=float("nan")) == c["GBATTN_ERR_SCALE"]
    assert _host(lib, ws=WS + 16) == c["GBATTN_ERR_ALIGN"]
    assert _host(lib, ws_bytes=1024) == c["GBATTN_ERR_WORKSPACE"]
    assert _host(lib, o=Q) == c["GBATTN_ERR_ALIAS"]


def test_host_workspace_size(lib):
    lib.attn_fwd_host_workspace_size.restype = ctypes.c_size_t
    # caseD: 256 heads of 512 x 128 -> chunks of 64 heads (24 MB of Q+K+V), two slots of
    # q, k, v, o (4 x 8 MiB) and lse (128 KiB).
    assert lib.attn_fwd_host_workspace_size(8, 32, 512, 128) == 2 * (4 * 64 * 512 * 128 * 2 + 64 * 512 * 4)
    assert lib.attn_fwd_host_workspace_size(1, 1, 0, 64) == 0


DWS = 0xB0000000


def _dec(lib, q=Q, k=K, v=V, o=O, lse=LSE, ws=None, B=1, H=2, L=128, d=64, scale=0.125):
    return lib.attn_decode(q, k, v, o, lse, ws, B, H, L, d, scale, None)


def test_decode_workspace_bytes(lib):
    for B, H, d in [(1, 1, 64), (1, 8, 128), (8, 32, 512)]:
        assert lib.attn_decode_workspace_bytes(B, H, d) == B * H * 32 * (d + 2) * 4
    c = _codes()
    assert lib.attn_decode_workspace_bytes(0, 1, 64) == c["GBATTN_ERR_DIMS"]
    assert lib.attn_decode_workspace_bytes(1, 1, 96) == c["GBATTN_ERR_HEAD_DIM"]


def test_decode_workspace_validation(lib):
    c = _codes()
    assert _dec(lib, ws=DWS + 8) == c["GBATTN_ERR_ALIGN"]
    assert _dec(lib, ws=O) == c["GBATTN_ERR_ALIAS"]
    assert _dec(lib, ws=K + 4096) == c["GBATTN_ERR_ALIAS"]  # inside k


def test_decode_validation(lib):
    c = _codes()
    for kw in ("q", "k", "v", "o", "lse"):
        assert _dec(lib, **{kw: 0}) == c["GBATTN_ERR_NULL"]
    for B, H, L in [(0, 1, 1), (1, 0, 1), (1, 1, 0), (1 << 16, 1 << 16, 1)]:
        assert _dec(lib, B=B, H=H, L=L) == c["GBATTN_ERR_DIMS"]
    for d in (0, 32, 96, 1024):
        assert _dec(lib, d=d) == c["GBATTN_ERR_HEAD_DIM"]
    for kw in ("q", "k", "v", "o", "lse"):
        base = {"q": Q, "k": K, "v": V, "o": O, "lse": LSE}[kw]
        assert _dec(lib, **{kw: base + 8}) == c["GBATTN_ERR_ALIGN"]
    for scale in (0.0, -1.0, float("inf"), float("nan")):
        assert _dec(lib, scale=scale) == c["GBATTN_ERR_SCALE"]
    assert _dec(lib, o=Q) == c["GBATTN_ERR_ALIAS"]
    assert _dec(lib, o=K + 1024) == c["GBATTN_ERR_ALIAS"]      # inside k
    assert _dec(lib, lse=O + 64) == c["GBATTN_ERR_ALIAS"]      # inside o (2*64*2 bytes)
    assert _dec(lib, lse=V) == c["GBATTN_ERR_ALIAS"]


def test_decode_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the fake addresses must never reach a launch")
    assert _dec(lib) in (_codes()["GBATTN_ERR_LAUNCH"], _codes()["GBATTN_ERR_DEVICE"])


DO_, DQ, DK, DV, WS = 0x60000000, 0x70000000, 0x80000000, 0x90000000, 0xA0000000


def _bwd(lib, q=Q, k=K, v=V, o=O, lse=LSE, do=DO_, dq=DQ, dk=DK, dv=DV, ws=WS, B=1, H=2, L=128, d=64, causal=0,
         scale=0.125):
    return lib.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, B, H, L, d, causal, scale, None)


def test_bwd_workspace_bytes(lib):
    """8 bytes per query row, rows padded to a multiple of 128."""
    for B, H, L in [(1, 1, 1), (1, 2, 128), (2, 3, 129), (8, 32, 512), (1, 1, 1000)]:
        assert lib.attn_bwd_workspace_bytes(B, H, L) == 8 * B * H * (-(-L // 128) * 128)
    c = _codes()
    for B, H, L in [(0, 1, 1), (1, 0, 1), (1, 1, 0), (1 << 16, 1 << 14, 1 << 10)]:
        assert lib.attn_bwd_workspace_bytes(B, H, L) == c["GBATTN_ERR_DIMS"]


def test_bwd_validation(lib):
    c = _codes()
    for kw in ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv", "ws"):
        assert _bwd(lib, **{kw: 0}) == c["GBATTN_ERR_NULL"], kw
    for B, H, L in [(0, 1, 1), (1, 0, 1), (1, 1, 0)]:
        assert _bwd(lib, B=B, H=H, L=L) == c["GBATTN_ERR_DIMS"]
    for d in (32, 96, 256, 512):
        assert _bwd(lib, d=d) == c["GBATTN_ERR_HEAD_DIM"], d
    for kw in ("q", "do", "dq", "dv", "lse", "ws"):
        base = {"q": Q, "do": DO_, "dq": DQ, "dv": DV, "lse": LSE, "ws": WS}[kw]
        assert _bwd(lib, **{kw: base + 8}) == c["GBATTN_ERR_ALIGN"], kw
    for scale in (0.0, float("nan")):
        assert _bwd(lib, scale=scale) == c["GBATTN_ERR_SCALE"]
    assert _bwd(lib, dq=Q) == c["GBATTN_ERR_ALIAS"]
    assert _bwd(lib, dk=DO_ + 64) == c["GBATTN_ERR_ALIAS"]
    assert _bwd(lib, dv=DK) == c["GBATTN_ERR_ALIAS"]
    assert _bwd(lib, dq=LSE) == c["GBATTN_ERR_ALIAS"]
    assert _bwd(lib, ws=DV + 1024) == c["GBATTN_ERR_ALIAS"]  # inside dv
    assert _bwd(lib, ws=O) == c["GBATTN_ERR_ALIAS"]
    assert _bwd(lib, dk=WS + 2048 - 16) == c["GBATTN_ERR_ALIAS"]  # workspace is 2048 bytes here
