"""Pins for the oracle's backward pass (the gradients GQ, GK, GV of the attention output,
through the score gradient GS: "Validating Memory-Optimal Transformer Kernels on Real
Hardware", section 4, "Paper II: Backward Pass and Fused Forward+Backward").

The pages print no gradient values.  The pins: PyTorch autograd through
scaled_dot_product_attention in float64 (the library routine the first page gates the
forward pass against); central finite differences of the oracle's own forward pass (pinned
on its own) against the oracle's gradients; closed forms (one key: dQ = dK = 0, dV = dO;
constant values: dQ = dK = 0); the invariant sum_j dK_j = 0 (every row of the score
gradient sums to zero); and mutation tests that plant plausible mistakes in a copy of the
backward code and check that the autograd pin catches each one.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle


def _rand(B, H, L, d, seed, dtype=torch.float64):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(B, H, L, d, generator=g, dtype=dtype) for _ in range(4)]


def _autograd(q, k, v, do, causal, scale):
    qq, kk, vv = (t.clone().double().requires_grad_() for t in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=causal, scale=scale)
    o.backward(do.double())
    return qq.grad.numpy(), kk.grad.numpy(), vv.grad.numpy()


@pytest.mark.parametrize("B,H,L,d,causal", [(1, 2, 37, 16, False), (2, 1, 64, 32, True), (1, 1, 130, 64, True),
                                            (1, 3, 5, 128, False)])
def test_matches_torch_autograd_float64(B, H, L, d, causal):
    q, k, v, do = _rand(B, H, L, d, L + d)
    scale = 1.0 / np.sqrt(d)
    got = oracle.sdpa_bwd(q, k, v, do, causal, scale)
    want = _autograd(q, k, v, do, causal, scale)
    for g, w in zip(got, want):
        np.testing.assert_allclose(g, w, rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences_of_the_forward_oracle(causal):
    """d/dx sum(O * dO) by central differences of oracle.sdpa_fwd, for a few entries of each
    of q, k, v, against the oracle's gradients."""
    q, k, v, do = (t.numpy() for t in _rand(1, 1, 6, 4, 3))
    scale, h = 0.7, 1e-6
    dq, dk, dv = oracle.sdpa_bwd(q, k, v, do, causal, scale)
    rng = np.random.default_rng(1)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(5):
            idx = (0, 0, int(rng.integers(6)), int(rng.integers(4)))
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            fp = (oracle.sdpa_fwd(*args, causal, scale)[0] * do).sum()
            args[which][idx] -= 2 * h
            fm = (oracle.sdpa_fwd(*args, causal, scale)[0] * do).sum()
            assert abs((fp - fm) / (2 * h) - grad[idx]) < 1e-7, (which, idx)


def test_one_key_closed_form():
    q, k, v, do = _rand(2, 2, 1, 32, 5)
    dq, dk, dv = oracle.sdpa_bwd(q, k, v, do, False, 0.5)
    assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0
    np.testing.assert_array_equal(dv, do.numpy())


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_give_zero_q_and_k_gradients(causal):
    q, k, _, do = _rand(1, 2, 40, 16, 6)
    v = torch.ones(1, 2, 40, 16, dtype=torch.float64) * torch.linspace(-1, 2, 16, dtype=torch.float64)
    dq, dk, _ = oracle.sdpa_bwd(q, k, v, do, causal, 0.25)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_key_gradients_sum_to_zero(causal):
    q, k, v, do = _rand(2, 3, 50, 32, 7)
    _, dk, _ = oracle.sdpa_bwd(q, k, v, do, causal, 0.2)
    assert np.abs(dk.sum(axis=2)).max() < 1e-12


# ---------------------------------------------------------------------------------------
# Mutation tests (on the CPU): a plausible mistake planted in a copy of the backward code
# must make the autograd pin fail.
# ---------------------------------------------------------------------------------------
_SRC = os.path.join(os.path.dirname(oracle.__file__), "sdpa_oracle.c")
MUTANTS = {
    "dq_without_scale": ("dqh[i * d + t] = scale * aq;", "dqh[i * d + t] = aq;"),
    "dk_without_scale": ("dkh[j * d + t] = scale * ak;", "dkh[j * d + t] = ak;"),
    "no_rowsum_term": ("dS[i * L + j] = P[i * L + j] * (dS[i * L + j] - rs);",
                       "dS[i * L + j] = P[i * L + j] * dS[i * L + j];"),
    "dv_with_score_gradient": ("av += P[i * L + j] * doh[i * d + t];", "av += dS[i * L + j] * doh[i * d + t];"),
    "dv_transposed_p": ("av += P[i * L + j] * doh[i * d + t];", "av += P[j * L + i] * doh[i * d + t];"),
    "dq_with_queries": ("aq += dS[i * L + j] * kh[j * d + t];", "aq += dS[i * L + j] * qh[j * d + t];"),
    "dk_untransposed": ("ak += dS[i * L + j] * qh[i * d + t];", "ak += dS[j * L + i] * qh[i * d + t];"),
    "dp_with_keys": ("acc += doh[i * d + t] * vh[j * d + t];", "acc += doh[i * d + t] * kh[j * d + t];"),
}


def _mutant(name, tmp_path):
    src = open(_SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so), str(path), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    dp = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.oracle_sdpa_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, ctypes.c_double, i]
    lib.oracle_sdpa_bwd.restype = i
    return lib


def _pin_passes(lib):
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    for causal in (False, True):
        q, k, v, do = (np.ascontiguousarray(t.numpy()) for t in _rand(1, 2, 24, 8, 9))
        out = [np.empty_like(q) for _ in range(3)]
        lib.oracle_sdpa_bwd(P(q), P(k), P(v), P(do), *(P(a) for a in out), 1, 2, 24, 8, int(causal), 0.4, 1)
        want = _autograd(*(torch.from_numpy(a) for a in (q, k, v, do)), causal, 0.4)
        if not all(np.allclose(g, w, rtol=0, atol=1e-9) for g, w in zip(out, want)):
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    assert not _pin_passes(_mutant(name, tmp_path)), f"the autograd pin did not catch mutant {name}"


def test_unmutated_copy_passes():
    for old, _ in MUTANTS.values():
        assert open(_SRC).read().count(old) == 1
    lib = ctypes.CDLL(oracle.build())
    dp = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.oracle_sdpa_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, ctypes.c_double, i]
    lib.oracle_sdpa_bwd.restype = i
    assert _pin_passes(lib)
