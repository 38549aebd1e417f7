"""Pins for the oracle's decode function (one query row per sequence against all of its
cached keys, "Validating Memory-Optimal Transformer Kernels on Real Hardware", section 5
"Paper III: Inference (Decode)") and for its fp16 -> float64 conversion.

As for the forward pass, the pages print no decode values, so the pins are closed forms
worked by hand (tests/golden/decode_examples.json), special cases with closed forms,
invariants, PyTorch's SDPA in float64 (the library routine the first page gates
against), the oracle's own forward pass (pinned separately), and mutation tests that
plant a plausible mistake in a copy of the oracle and check that a pin catches it.
"""
import ctypes
import json
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "decode_examples.json")
_ENV = {"e": math.e, "exp": math.exp, "log": math.log, "__builtins__": {}}


def _examples():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


def _inputs(ex):
    q = np.asarray(ex["q"], np.float16)[None, None, :]
    k = np.asarray(ex["k"], np.float16)[None, None]
    v = np.asarray(ex["v"], np.float16)[None, None]
    for name, a in (("q", q), ("k", k), ("v", v)):
        assert np.array_equal(a.astype(np.float64).ravel(), np.asarray(ex[name], np.float64).ravel()), name
    return q, k, v


def _expected(ex):
    return (np.array([eval(s, _ENV) for s in ex["O"]], np.float64), eval(ex["LSE"], _ENV))


def test_f16_conversion_exhaustive():
    """Every one of the 65536 binary16 bit patterns against numpy's conversion."""
    h = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_to_f64(h)
    ref = h.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("ex", _examples(), ids=lambda e: e["name"])
def test_worked_examples(ex):
    q, k, v = _inputs(ex)
    o, lse = oracle.decode(q, k, v, ex["scale"])
    o_ref, lse_ref = _expected(ex)
    np.testing.assert_allclose(o[0], o_ref, rtol=1e-15, atol=1e-15)
    assert abs(lse[0] - lse_ref) <= 1e-14


def _rand(B, H, L, d, seed, sigma=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, 1, d, generator=g) * sigma).half()
    k = (torch.randn(B, H, L, d, generator=g) * sigma).half()
    v = (torch.randn(B, H, L, d, generator=g) * sigma).half()
    return q, k, v


def test_single_key_returns_that_value():
    q, k, v = _rand(2, 3, 1, 64, 11)
    o, lse = oracle.decode(q, k, v, 0.125)
    np.testing.assert_array_equal(o, v.double().numpy().reshape(6, 64))
    s = (q.double() * k.double()).sum(-1).reshape(6) * 0.125
    np.testing.assert_allclose(lse, s.numpy(), rtol=0, atol=1e-13)


def test_zero_query_gives_mean_and_log_length():
    _, k, v = _rand(1, 4, 37, 128, 12)
    q = torch.zeros(1, 4, 1, 128, dtype=torch.float16)
    o, lse = oracle.decode(q, k, v, 0.088388)
    np.testing.assert_allclose(o, v.double().mean(2).numpy().reshape(4, 128), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.full(4, math.log(37)), rtol=0, atol=1e-13)


def test_constant_values_give_constant_output():
    q, k, _ = _rand(1, 2, 50, 64, 13)
    v = torch.empty(1, 2, 50, 64, dtype=torch.float16)
    v[:] = torch.linspace(-3, 3, 64).half()
    o, _ = oracle.decode(q, k, v, 0.125)
    np.testing.assert_allclose(o, np.tile(v[0, 0, 0].double().numpy(), (2, 1)), rtol=0, atol=1e-12)


def test_key_permutation_invariance():
    q, k, v = _rand(1, 2, 40, 64, 14)
    perm = torch.randperm(40, generator=torch.Generator().manual_seed(3))
    o1, l1 = oracle.decode(q, k, v, 0.125)
    o2, l2 = oracle.decode(q, k[:, :, perm], v[:, :, perm], 0.125)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("B,H,L,d", [(2, 3, 37, 64), (1, 2, 300, 128), (1, 1, 65, 512)])
def test_matches_torch_sdpa_float64(B, H, L, d):
    q, k, v = _rand(B, H, L, d, 15 + L)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    o, lse = oracle.decode(q, k, v, scale)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), k.double(), v.double(), scale=scale)
    np.testing.assert_allclose(o, ref.numpy().reshape(B * H, d), rtol=0, atol=1e-12)
    s = (q.double() @ k.double().transpose(-1, -2)) * scale
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy().reshape(B * H), rtol=0, atol=1e-12)


def test_equals_last_row_of_causal_forward():
    """Decode of query q against keys 0..L-1 is row L-1 of the causal forward pass whose
    last query row is q (the forward oracle is pinned on its own)."""
    B, H, L, d = 1, 3, 45, 64
    qf, k, v = _rand(B, H, L, d, 16)
    qfull = torch.randn(B, H, L, d, generator=torch.Generator().manual_seed(17)).half()
    qfull[:, :, L - 1] = qf[:, :, 0]
    o_f, lse_f = oracle.sdpa_fwd(qfull, k, v, True, 0.125)
    o, lse = oracle.decode(qf, k, v, 0.125)
    np.testing.assert_allclose(o, o_f[:, :, L - 1].reshape(B * H, d), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_f[:, :, L - 1].reshape(B * H), rtol=0, atol=1e-13)


def test_head_subset_matches_full():
    q, k, v = _rand(2, 4, 33, 64, 18)
    o, lse = oracle.decode(q, k, v, 0.125)
    heads = [7, 0, 3, 3]
    o2, lse2 = oracle.decode(q, k, v, 0.125, heads=heads)
    np.testing.assert_array_equal(o2, o[heads])
    np.testing.assert_array_equal(lse2, lse[heads])
    with pytest.raises(IndexError):
        oracle.decode(q, k, v, 0.125, heads=[8])


# ---------------------------------------------------------------------------------------
# Mutation tests (on the CPU): a plausible mistake planted in a copy of the decode
# function or the conversion must make a pin fail.
# ---------------------------------------------------------------------------------------
_SRC = os.path.join(os.path.dirname(oracle.__file__), "sdpa_oracle.c")
MUTANTS = {
    "dropped_scale": ("srow[j] = scale * dot;", "srow[j] = dot;"),
    "half_length_dot": ("for (int t = 0; t < d; ++t)\n                dot += qf[t]",
                        "for (int t = 0; t < d / 2; ++t)\n                dot += qf[t]"),
    "last_key_dropped": ("for (long j = 0; j < L; ++j) {\n            const uint16_t *kj",
                         "for (long j = 0; j < L - 1; ++j) {\n            const uint16_t *kj"),
    "no_max_subtraction": ("srow[j] = exp(srow[j] - m);\n            l += srow[j];",
                           "srow[j] = exp(srow[j]);\n            l += srow[j];"),
    "lse_without_max": ("lse[i] = m + log(l);", "lse[i] = log(l);"),
    "missing_divide": ("o[i * d + c] = acc[c] / l;", "o[i * d + c] = acc[c];"),
    "values_read_from_keys": ("const uint16_t *vj = v + ", "const uint16_t *vj = k + "),
    "f16_exponent_bias": ("mag = ldexp((double)(f + 1024), e - 25);", "mag = ldexp((double)(f + 1024), e - 24);"),
    "f16_subnormal_scale": ("mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);"),
    "f16_sign_dropped": ("return (h >> 15) ? -mag : mag;", "return mag;"),
}


def _decode_with(lib, ex):
    q, k, v = _inputs(ex)
    L, d = k.shape[2], k.shape[3]
    o = np.empty((1, d))
    lse = np.empty((1,))
    u16 = lambda a: np.ascontiguousarray(a).view(np.uint16).ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    qa, ka, va = (np.ascontiguousarray(a) for a in (q, k, v))
    lib.oracle_decode_f16(u16(qa), u16(ka), u16(va), P(o), P(lse), 1, L, d, ex["scale"], None, 0, 1)
    return o[0], lse[0]


def _load_lib(path):
    lib = ctypes.CDLL(str(path))
    u16p = ctypes.POINTER(ctypes.c_uint16)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_decode_f16.argtypes = [u16p, u16p, u16p, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                      ctypes.c_double, ctypes.POINTER(ctypes.c_int64), ctypes.c_long, ctypes.c_int]
    lib.oracle_decode_f16.restype = ctypes.c_int
    return lib


def _pins_pass(lib):
    for ex in _examples():
        o, lse = _decode_with(lib, ex)
        o_ref, lse_ref = _expected(ex)
        if not (np.allclose(o, o_ref, rtol=1e-12, atol=1e-15) and abs(lse - lse_ref) <= 1e-12):
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(_SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so), str(path), "-lm"],
                   check=True)
    with np.errstate(all="ignore"):
        assert not _pins_pass(_load_lib(so)), f"the decode worked examples did not catch mutant {name}"


def test_unmutated_copy_passes():
    for old, _ in MUTANTS.values():
        assert open(_SRC).read().count(old) == 1
    assert _pins_pass(_load_lib(oracle.build()))
