"""ctypes binding of libgbattn.so: argument marshalling only.

Every function here converts torch tensors to raw device pointers and sizes, calls the
C entry point of the same name (include/gbattn.h), and turns a nonzero return code into
a GbattnError.  There is no fallback: if the library is missing or the tensors are not
on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgbattn.so")
_lib = None

FLAG_P_SMEM = 1
FLAG_SINGLE_TILE = 2
FLAG_TWO_TILE = 4
FLAG_DSPLIT = 8
FLAG_SPLIT_KV = 16


class GbattnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: gbattn error {code}: {attn_strerror(code)}")


def load_library(path: str | None = None):
    """Load libgbattn.so (built by scaled_dot_product_sdpa_gb300.build).  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libgbattn.so not built ({path} missing); run "
                           "`python -m scaled_dot_product_sdpa_gb300.build` or __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.attn_fwd.restype = i
    lib.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, i, i]
    lib.attn_fwd_ex.restype = i
    lib.attn_debug_scores.argtypes = [vp, vp, vp, i, i, i, i, f, vp]
    lib.attn_debug_scores.restype = i
    lib.attn_last_device_error.argtypes = []
    lib.attn_last_device_error.restype = i
    lib.attn_debug_wait_probe.argtypes = [ctypes.c_longlong, vp]
    lib.attn_debug_wait_probe.restype = i
    lib.attn_strerror.argtypes = [i]
    lib.attn_strerror.restype = ctypes.c_char_p
    ip = ctypes.POINTER(ctypes.c_int)
    lib.attn_debug_schedule.argtypes = [i, i, i, i, i, i, i, ip, ip, i]
    lib.attn_debug_schedule.restype = i
    sz = ctypes.c_size_t
    lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.attn_fwd_host.restype = i
    lib.attn_fwd_host_workspace_size.argtypes = [i, i, i, i]
    lib.attn_fwd_host_workspace_size.restype = sz
    lib.attn_debug_plan.argtypes = [i, i, i, i, i, i, i, i, ip]
    lib.attn_debug_plan.restype = i
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.attn_bwd.restype = i
    lib.attn_bwd_workspace_bytes.argtypes = [i, i, i]
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_longlong
    lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.attn_bwd_noalloc.restype = i
    lib.attn_bwd_noalloc_max_bytes.argtypes = []
    lib.attn_bwd_noalloc_max_bytes.restype = ctypes.c_longlong
    lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, vp]
    lib.attn_decode.restype = i
    lib.attn_decode_workspace_bytes.argtypes = [i, i, i]
    lib.attn_decode_workspace_bytes.restype = ctypes.c_longlong
    lib.attn_debug_decode_plan.argtypes = [i, i, i, i, i, i, i, ip]
    lib.attn_debug_decode_plan.restype = i
    lib.attn_version.argtypes = []
    lib.attn_version.restype = i
    _lib = lib
    return lib


def attn_strerror(code: int) -> str:
    return load_library().attn_strerror(int(code)).decode()


def attn_version() -> int:
    return load_library().attn_version()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check_qkv(q, k, v=None):
    ts = [q, k] + ([v] if v is not None else [])
    for t in ts:
        if not t.is_cuda:
            raise ValueError("gbattn: tensors must be on a CUDA device (no CPU path exists)")
        if t.dtype != torch.float16:
            raise ValueError("gbattn: q, k, v must be float16")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError("gbattn: q, k, v must be contiguous [B, H, L, d]")
        if t.shape != q.shape:
            raise ValueError("gbattn: q, k, v must have the same shape")
    return q.shape


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None, stream=None,
             flags: int = 0, grid_limit: int = 0):
    """O, LSE = SDPA forward of fp16 [B, H, L, d] q, k, v.  Outputs are allocated by torch
    on q's device unless given.  Enqueued on `stream` (default: torch's current stream)."""
    B, H, L, d = _check_qkv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    if o.shape != q.shape or o.dtype != torch.float16 or not o.is_contiguous():
        raise ValueError("gbattn: o must be contiguous float16 like q")
    if lse.shape != (B, H, L) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("gbattn: lse must be contiguous float32 [B, H, L]")
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                             B, H, L, d, int(bool(causal)), float(scale), _stream_handle(stream),
                             int(flags), int(grid_limit))
    if rc != 0:
        raise GbattnError(rc, "attn_fwd")
    return o, lse


def attn_bwd_workspace_bytes(B: int, H: int, L: int) -> int:
    """Bytes of device workspace attn_bwd needs (8 per query row, rows padded to 128)."""
    n = load_library().attn_bwd_workspace_bytes(int(B), int(H), int(L))
    if n < 0:
        raise GbattnError(int(n), "attn_bwd_workspace_bytes")
    return int(n)


def attn_bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
             stream=None, workspace=None):
    """Gradients (dq, dk, dv) of O = SDPA(q, k, v) for the upstream gradient dout, from the
    forward pass's o and lse (as attn_fwd returns them).  fp16 [B, H, L, d] tensors, d 64 or
    128; outputs allocated by torch on q's device unless given, and so is the workspace
    (attn_bwd_workspace_bytes(B, H, L) bytes) unless `workspace` (a contiguous CUDA tensor
    at least that large) is given.  Enqueued on `stream`."""
    B, H, L, d = _check_qkv(q, k, v)
    for t in (o, dout):
        if not t.is_cuda or t.dtype != torch.float16 or t.shape != q.shape or not t.is_contiguous():
            raise ValueError("gbattn: o and dout must be contiguous float16 like q")
    if not lse.is_cuda or lse.dtype != torch.float32 or lse.shape != (B, H, L) or not lse.is_contiguous():
        raise ValueError("gbattn: lse must be contiguous float32 [B, H, L]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t in (dq, dk, dv):
        if t.shape != q.shape or t.dtype != torch.float16 or not t.is_contiguous():
            raise ValueError("gbattn: dq, dk, dv must be contiguous float16 like q")
    lib = load_library()
    nbytes = attn_bwd_workspace_bytes(B, H, L)
    if workspace is None:
        workspace = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device)
        if isinstance(stream, torch.cuda.Stream):
            workspace.record_stream(stream)  # freed only once the kernels on `stream` are done
    elif (not workspace.is_cuda or not workspace.is_contiguous()
          or workspace.numel() * workspace.element_size() < nbytes):
        raise ValueError(f"gbattn: workspace must be a contiguous CUDA tensor of at least {nbytes} bytes")
    with torch.cuda.device(q.device):
        rc = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), B, H, L, d,
                          int(bool(causal)), float(scale), _stream_handle(stream))
    if rc != 0:
        raise GbattnError(rc, "attn_bwd")
    return dq, dk, dv


def attn_decode(q, k, v, scale: float | None = None, o=None, lse=None, stream=None, grouped: bool = True):
    """Decode: O [B, H, d] and LSE [B, H] for one fp16 query row q ([B, H, d] or
    [B, H, 1, d]) per head against fp16 k, v [B, H, L, d], every key visible.  Outputs are
    allocated by torch on q's device unless given, and so is the small workspace that lets
    a head's keys be split over several clusters (`grouped`; without it, one cluster per
    head).  Enqueued on `stream`."""
    for t in (q, k, v):
        if not t.is_cuda:
            raise ValueError("gbattn: tensors must be on a CUDA device (no CPU path exists)")
        if t.dtype != torch.float16 or not t.is_contiguous():
            raise ValueError("gbattn: q, k, v must be contiguous float16")
    if k.dim() != 4 or v.shape != k.shape:
        raise ValueError("gbattn: k and v must share one [B, H, L, d] shape")
    B, H, L, d = k.shape
    if tuple(q.shape) not in ((B, H, d), (B, H, 1, d)):
        raise ValueError("gbattn: q must be [B, H, d] or [B, H, 1, d]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty((B, H, d), dtype=torch.float16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if o.numel() != B * H * d or o.dtype != torch.float16 or not o.is_contiguous():
        raise ValueError("gbattn: o must be contiguous float16 with B*H*d elements")
    if lse.numel() != B * H or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("gbattn: lse must be contiguous float32 [B, H]")
    lib = load_library()
    ws = None
    if grouped:
        nbytes = lib.attn_decode_workspace_bytes(B, H, d)
        if nbytes < 0:
            raise GbattnError(int(nbytes), "attn_decode_workspace_bytes")
        ws = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device)
        if isinstance(stream, torch.cuda.Stream):
            ws.record_stream(stream)  # freed only once the kernels on `stream` are done
    with torch.cuda.device(q.device):
        rc = lib.attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                             ws.data_ptr() if ws is not None else None, B, H, L, d, float(scale),
                             _stream_handle(stream))
    if rc != 0:
        raise GbattnError(rc, "attn_decode")
    return o, lse


def attn_debug_decode_plan(B: int, H: int, L: int, d: int, sm_count: int, max_ranks: int = 16,
                           grouped: bool = False) -> dict:
    """The split attn_decode uses (host-only): CTAs per cluster, keys per CTA and clusters
    per head (more than one only with a workspace, `grouped`)."""
    out = (ctypes.c_int * 3)()
    rc = load_library().attn_debug_decode_plan(B, H, L, d, sm_count, max_ranks, int(bool(grouped)), out)
    if rc != 0:
        raise GbattnError(rc, "attn_debug_decode_plan")
    return {"ranks": out[0], "keys_per_rank": out[1], "groups": out[2]}


def attn_debug_scores(q, k, scale: float | None = None, s=None, stream=None):
    """Raw scaled logits scale * Q K^T as fp32 [B, H, L, L] (test hook, no mask)."""
    B, H, L, d = _check_qkv(q, k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if s is None:
        s = torch.empty((B, H, L, L), dtype=torch.float32, device=q.device)
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.attn_debug_scores(q.data_ptr(), k.data_ptr(), s.data_ptr(), B, H, L, d, float(scale),
                                   _stream_handle(stream))
    if rc != 0:
        raise GbattnError(rc, "attn_debug_scores")
    return s


def attn_last_device_error() -> int:
    """Synchronise the current device, then read and clear its device status word."""
    return load_library().attn_last_device_error()


def attn_debug_wait_probe(limit_cycles: int, stream=None) -> None:
    rc = load_library().attn_debug_wait_probe(int(limit_cycles), _stream_handle(stream))
    if rc != 0:
        raise GbattnError(rc, "attn_debug_wait_probe")


def attn_debug_schedule(B: int, H: int, L: int, d: int, causal: bool, grid: int, flags: int = 0):
    """The static work schedule attn_fwd would use (host-only): a list with, per CTA, the
    work-item indices it runs in order; None when the kernels use their fixed order.  With
    FLAG_SPLIT_KV an index >= the item count names a query tile whose key range the two
    CTAs of a cluster (CTAs 2c, 2c + 1) share."""
    max_items = 1 << 16
    start = (ctypes.c_int * (grid + 1))()
    items = (ctypes.c_int * max_items)()
    n = load_library().attn_debug_schedule(B, H, L, d, int(bool(causal)), grid, flags, start, items, max_items)
    if n < 0:
        raise GbattnError(n, "attn_debug_schedule")
    if n == 0:
        return None
    return [list(items[start[c]:start[c + 1]]) for c in range(grid)]


def attn_debug_plan(B: int, H: int, L: int, d: int, causal: bool, sm_count: int, flags: int = 0,
                    grid_limit: int = 0) -> dict:
    """The kernel attn_fwd would launch on a GPU with `sm_count` SMs (host-only):
    kind 0 single-tile, 1 two-tile, 2 single-tile with the head_dim split, 3 single-tile
    with key-range splits (CTAs in clusters of two)."""
    out = (ctypes.c_int * 4)()
    rc = load_library().attn_debug_plan(B, H, L, d, int(bool(causal)), sm_count, flags, grid_limit, out)
    if rc != 0:
        raise GbattnError(rc, "attn_debug_plan")
    return {"kind": out[0], "items": out[1], "grid": out[2], "makespan": out[3] / 100.0}


# Device workspaces of attn_fwd_host, one per (device, stream): calls on one stream never
# overlap on the GPU, calls on different streams may.
_host_workspaces: dict = {}


def attn_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None,
                  device=None, stream=None):
    """O, LSE = SDPA forward of fp16 [B, H, L, d] CPU tensors q, k, v (pin them for the
    copies to overlap), computed on `device` (default: the current CUDA device) in
    chunks whose host<->device copies overlap the kernels.  Outputs are CPU tensors
    (pinned, allocated here unless given).  Enqueued on `stream` (default: the device's
    current stream); synchronise it before reading the outputs."""
    for t in (q, k, v):
        if t.is_cuda:
            raise ValueError("gbattn: attn_fwd_host takes CPU tensors (use attn_fwd for CUDA tensors)")
        if t.dtype != torch.float16 or t.dim() != 4 or not t.is_contiguous() or t.shape != q.shape:
            raise ValueError("gbattn: q, k, v must be contiguous float16 [B, H, L, d] of one shape")
    B, H, L, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q).pin_memory()
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32).pin_memory()
    if o.is_cuda or o.shape != q.shape or o.dtype != torch.float16 or not o.is_contiguous():
        raise ValueError("gbattn: o must be a contiguous float16 CPU tensor like q")
    if lse.is_cuda or lse.shape != (B, H, L) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("gbattn: lse must be a contiguous float32 CPU tensor [B, H, L]")
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    lib = load_library()
    with torch.cuda.device(device):
        sh = _stream_handle(stream)
        need = int(lib.attn_fwd_host_workspace_size(B, H, L, d))
        key = (device.index, sh)
        ws = _host_workspaces.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
            _host_workspaces[key] = ws
        rc = lib.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               B, H, L, d, int(bool(causal)), float(scale), ws.data_ptr(), ws.numel(), sh)
    if rc != 0:
        raise GbattnError(rc, "attn_fwd_host")
    return o, lse
