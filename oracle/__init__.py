"""float64 CPU oracle for the scaled-dot-product attention forward pass.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s cpu_baseline / reference leg may import this package.  It shares
no code with the CUDA path: it builds its own C library (``sdpa_oracle.c``) with gcc
and talks to it through ctypes; it imports nothing from the product package.

Definitions followed (cited by page title and section):

* "An Optimal Mapper Meets a Real GPU", "Ground rules" and "Experiment one":
  SDPA O = softmax(scale * Q K^T + causal mask) V with FP16 inputs, query length equal
  to key/value length, gated against PyTorch SDPA; its three stages are QK, softmax
  (max, exp, sum, divide) and AV.
* STAGE_D.md (nvfp4-megamoe-kernel), section 4: the row log-sum-exp (LSE) output;
  section 2: head_dim sub-tiles are additive in logit space (S = S_0 + S_1) and an
  "external merge" of softmax outputs over partial dot products is not the attention.
* "Validating Memory-Optimal Transformer Kernels on Real Hardware", section 4 ("Paper
  II: Backward Pass and Fused Forward+Backward"): the gradients of the attention output
  with respect to Q, K and V (GQ, GK, GV, through the score gradient GS); ``sdpa_bwd``
  computes them for a given upstream gradient dO by differentiating the definition.
* "Validating Memory-Optimal Transformer Kernels on Real Hardware", section 5 ("Paper
  III: Inference (Decode)"): decoding, one new query row per sequence against the whole
  cached key/value sequence; ``decode`` computes it by the same definition with every key
  visible.

Every function takes arrays of shape [B, H, L, d] (anything numpy can view, including
CPU torch tensors), converts them to float64 (exact for fp16 values) and returns numpy
float64 arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile sdpa_oracle.c into oracle/liboracle.so with gcc (OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", _LIB, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.oracle_sdpa_fwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, ctypes.c_double, i]
        lib.oracle_sdpa_fwd.restype = i
        lib.oracle_sdpa_fwd_rows.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, ctypes.c_double,
                                             ctypes.POINTER(ctypes.c_int64), ctypes.c_long, i]
        lib.oracle_sdpa_fwd_rows.restype = i
        lib.oracle_scores.argtypes = [dp, dp, dp, i, i, i, i, ctypes.c_double, i, i]
        lib.oracle_scores.restype = None
        lib.oracle_softmax.argtypes = [dp, dp, dp, i, i, i, i]
        lib.oracle_softmax.restype = None
        lib.oracle_pv.argtypes = [dp, dp, dp, i, i, i, i]
        lib.oracle_pv.restype = None
        lib.oracle_sdpa_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, ctypes.c_double, i]
        lib.oracle_sdpa_bwd.restype = i
        u16p = ctypes.POINTER(ctypes.c_uint16)
        lib.oracle_f16_to_f64.argtypes = [u16p, dp, ctypes.c_long]
        lib.oracle_f16_to_f64.restype = None
        lib.oracle_decode_f16.argtypes = [u16p, u16p, u16p, dp, dp, ctypes.c_long, ctypes.c_long, i,
                                          ctypes.c_double, ctypes.POINTER(ctypes.c_int64), ctypes.c_long, i]
        lib.oracle_decode_f16.restype = i
        _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: exact fp16 -> fp64 via numpy
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape4(q):
    if q.ndim != 4:
        raise ValueError("expected [B, H, L, d]")
    return q.shape


def sdpa_fwd(q, k, v, causal: bool, scale: float, nthreads: int = 0):
    """Full forward pass by the plain definition.  Returns (O [B,H,L,d], LSE [B,H,L])
    in float64.  `scale` is used as given (pass the same fp32 value the kernel gets)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, L, d = _shape4(q)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, L, d] shape")
    o = np.empty((B, H, L, d), np.float64)
    lse = np.empty((B, H, L), np.float64)
    rc = _load().oracle_sdpa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, L, d,
                                 int(bool(causal)), float(scale), int(nthreads))
    if rc < 0:
        raise MemoryError("oracle scratch allocation failed")
    return o, lse


def sdpa_fwd_rows(q, k, v, causal: bool, scale: float, rows, nthreads: int = 0):
    """The forward pass for a sample of flat rows (row = (b*H + h)*L + i) only.
    Returns (O [n, d], LSE [n]) in float64, plus the thread count used."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, L, d = _shape4(q)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    rc = _load().oracle_sdpa_fwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, L, d,
                                      int(bool(causal)), float(scale),
                                      rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
                                      int(nthreads))
    if rc == -2:
        raise IndexError("row index out of range")
    if rc < 0:
        raise MemoryError("oracle scratch allocation failed")
    return o, lse, rc


def scores(q, k, scale: float, t0: int = 0, t1: int | None = None):
    """Stage QK alone: scale * sum_{t0 <= t < t1} q_i,t k_j,t for all i, j (no mask)."""
    q, k = _f64(q), _f64(k)
    B, H, L, d = _shape4(q)
    t1 = d if t1 is None else t1
    if not (0 <= t0 <= t1 <= d):
        raise ValueError("bad head_dim range")
    s = np.empty((B, H, L, L), np.float64)
    _load().oracle_scores(_ptr(q), _ptr(k), _ptr(s), B, H, L, d, float(scale), int(t0), int(t1))
    return s


def softmax(s, causal: bool):
    """Stage softmax alone on logits [B,H,L,L]: returns (P [B,H,L,L], LSE [B,H,L])."""
    s = _f64(s)
    B, H, L, L2 = s.shape
    if L2 != L:
        raise ValueError("logits must be [B, H, L, L]")
    p = np.empty_like(s)
    lse = np.empty((B, H, L), np.float64)
    _load().oracle_softmax(_ptr(s), _ptr(p), _ptr(lse), B, H, L, int(bool(causal)))
    return p, lse


def pv(p, v):
    """Stage AV alone: O = P V for P [B,H,L,L] and V [B,H,L,d]."""
    p, v = _f64(p), _f64(v)
    B, H, L, d = _shape4(v)
    o = np.empty((B, H, L, d), np.float64)
    _load().oracle_pv(_ptr(p), _ptr(v), _ptr(o), B, H, L, d)
    return o


def _u16(x) -> np.ndarray:
    """Raw fp16 bits of x (a float16 numpy array or a CPU fp16 torch tensor), contiguous."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != np.float16:
        raise TypeError("decode takes fp16 inputs")
    return x.view(np.uint16)


def f16_to_f64(h) -> np.ndarray:
    """The oracle's own binary16 -> float64 conversion of raw bits h (uint16 array)."""
    h = np.ascontiguousarray(np.asarray(h, dtype=np.uint16))
    out = np.empty(h.shape, np.float64)
    _load().oracle_f16_to_f64(h.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), _ptr(out), h.size)
    return out


def decode(q, k, v, scale: float, heads=None, nthreads: int = 0):
    """Decode by the plain definition: q [B, H, d] (or [B, H, 1, d]), k, v [B, H, L, d], all
    fp16; every key visible.  Returns (O [n, d], LSE [n]) in float64 for the flat heads
    (b*H + h) listed in `heads` (default: all B*H heads, in order)."""
    qu, ku, vu = _u16(q), _u16(k), _u16(v)
    if ku.ndim != 4 or vu.shape != ku.shape:
        raise ValueError("k and v must share one [B, H, L, d] shape")
    B, H, L, d = ku.shape
    if qu.size != B * H * d:
        raise ValueError("q must hold one d-vector per (b, h)")
    BH = B * H
    if heads is None:
        hp, n = None, BH
    else:
        hs = np.ascontiguousarray(np.asarray(heads, dtype=np.int64))
        hp, n = hs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), hs.size
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    rc = _load().oracle_decode_f16(qu.ctypes.data_as(u16p), ku.ctypes.data_as(u16p), vu.ctypes.data_as(u16p),
                                   _ptr(o), _ptr(lse), BH, L, d, float(scale), hp, n, int(nthreads))
    if rc == -2:
        raise IndexError("head index out of range")
    if rc < 0:
        raise MemoryError("oracle scratch allocation failed")
    return o, lse


def sdpa_bwd(q, k, v, dout, causal: bool, scale: float, nthreads: int = 0):
    """Gradients (dQ, dK, dV), each [B, H, L, d] float64, of O = SDPA(q, k, v) for the
    upstream gradient dout, by differentiating the plain definition (the full L x L
    score, probability and score-gradient matrices of each head are formed)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, L, d = _shape4(q)
    if k.shape != q.shape or v.shape != q.shape or dout.shape != q.shape:
        raise ValueError("q, k, v, dout must share one [B, H, L, d] shape")
    dq, dk, dv = (np.empty((B, H, L, d), np.float64) for _ in range(3))
    rc = _load().oracle_sdpa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, H, L, d,
                                 int(bool(causal)), float(scale), int(nthreads))
    if rc < 0:
        raise MemoryError("oracle scratch allocation failed")
    return dq, dk, dv
