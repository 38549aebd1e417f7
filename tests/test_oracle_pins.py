"""Pins for the float64 CPU oracle: checks against things other than the oracle itself.

Each pin follows the SDPA definition of "An Optimal Mapper Meets a Real GPU" ("Ground
rules", "Experiment one") and the STAGE_D.md notes (sections 2 and 4: logit additivity
over head_dim sub-tiles, the LSE output, the wrong external merge).  The pages print no
numeric worked example, so the pins are hand-worked closed forms (tests/golden/),
special cases with closed forms, invariants, the library routine the first page gates
against (PyTorch SDPA, here in float64 on the CPU), and mutation tests that plant a
plausible mistake in a copy of the oracle and check that a pin catches it.
"""
import json
import math
import os
import subprocess

import ctypes
import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
_ENV = {"e": math.e, "exp": math.exp, "log": math.log, "__builtins__": {}}


def _examples():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


def _expected(ex):
    o = np.array([[eval(s, _ENV) for s in row] for row in ex["O"]], dtype=np.float64)
    lse = np.array([eval(s, _ENV) for s in ex["LSE"]], dtype=np.float64)
    return o, lse


def _as4(x):
    return np.asarray(x, dtype=np.float64)[None, None]


@pytest.mark.parametrize("ex", _examples(), ids=lambda e: e["name"])
def test_worked_example_full_forward(ex):
    o, lse = oracle.sdpa_fwd(_as4(ex["q"]), _as4(ex["k"]), _as4(ex["v"]), ex["causal"], ex["scale"])
    o_ref, lse_ref = _expected(ex)
    np.testing.assert_allclose(o[0, 0], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], lse_ref, rtol=1e-15, atol=1e-12)


@pytest.mark.parametrize("ex", _examples(), ids=lambda e: e["name"])
def test_worked_example_staged(ex):
    """The three stages (QK, softmax, AV) run one by one give the same closed forms."""
    s = oracle.scores(_as4(ex["q"]), _as4(ex["k"]), ex["scale"])
    p, lse = oracle.softmax(s, ex["causal"])
    o = oracle.pv(p, _as4(ex["v"]))
    o_ref, lse_ref = _expected(ex)
    np.testing.assert_allclose(o[0, 0], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], lse_ref, rtol=1e-15, atol=1e-12)


def _rand(B, H, L, d, seed, sigma=1.0):
    g = np.random.default_rng(seed)
    mk = lambda: (g.standard_normal((B, H, L, d)) * sigma).astype(np.float16).astype(np.float64)
    return mk(), mk(), mk()


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one(causal):
    q, k, _ = _rand(2, 3, 37, 16, 11)
    p, _ = oracle.softmax(oracle.scores(q, k, 0.25), causal)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-13)
    assert (p >= 0).all()
    if causal:
        upper = np.triu(np.ones((37, 37), bool), k=1)
        assert (p[..., upper] == 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(causal):
    q, k, _ = _rand(1, 2, 50, 8, 3)
    kappa = np.arange(8, dtype=np.float64) - 3.5
    v = np.broadcast_to(kappa, (1, 2, 50, 8)).copy()
    o, _ = oracle.sdpa_fwd(q, k, v, causal, 0.3)
    np.testing.assert_allclose(o, np.broadcast_to(kappa, o.shape), atol=1e-12)


def test_q_zero_causal_gives_prefix_mean():
    _, k, v = _rand(1, 2, 40, 8, 5)
    q = np.zeros_like(k)
    o, lse = oracle.sdpa_fwd(q, k, v, True, 0.7)
    prefix = np.cumsum(v, axis=2) / np.arange(1, 41)[None, None, :, None]
    np.testing.assert_allclose(o, prefix, atol=1e-12)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, 41)), lse.shape), atol=1e-12)


def test_q_zero_noncausal_gives_mean():
    _, k, v = _rand(2, 1, 33, 4, 6)
    o, lse = oracle.sdpa_fwd(np.zeros_like(k), k, v, False, 1.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-12)
    np.testing.assert_allclose(lse, math.log(33), atol=1e-12)


def test_causal_row0_is_v0():
    q, k, v = _rand(2, 2, 19, 16, 7)
    o, lse = oracle.sdpa_fwd(q, k, v, True, 0.125)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-12)
    dot0 = (q[:, :, 0] * k[:, :, 0]).sum(-1)
    np.testing.assert_allclose(lse[:, :, 0], 0.125 * dot0, atol=1e-12)


def test_subtile_logit_additivity():
    """head_dim 512 split into two 256-wide sub-tiles: S = S_0 + S_1 (STAGE_D.md, section 2)."""
    q, k, _ = _rand(1, 2, 24, 512, 8, sigma=0.5)
    s = oracle.scores(q, k, 1 / math.sqrt(512))
    s0 = oracle.scores(q, k, 1 / math.sqrt(512), 0, 256)
    s1 = oracle.scores(q, k, 1 / math.sqrt(512), 256, 512)
    np.testing.assert_allclose(s0 + s1, s, atol=1e-12)
    assert np.abs(s0).max() > 0.1 and np.abs(s1).max() > 0.1


@pytest.mark.parametrize("causal", [False, True])
def test_external_merge_is_not_attention(causal):
    """Negative test (STAGE_D.md, section 2): softmax each partial dot product, then merge
    the two outputs with LSE weights.  That merge is valid only for disjoint key sets, so
    on random data it must differ from the true O by far more than the O tolerance."""
    q, k, v = _rand(1, 2, 64, 512, 9, sigma=1.0)
    sc = 1 / math.sqrt(512)
    o_true, _ = oracle.sdpa_fwd(q, k, v, causal, sc)
    p0, l0 = oracle.softmax(oracle.scores(q, k, sc, 0, 256), causal)
    p1, l1 = oracle.softmax(oracle.scores(q, k, sc, 256, 512), causal)
    o0, o1 = oracle.pv(p0, v), oracle.pv(p1, v)
    w0, w1 = np.exp(l0)[..., None], np.exp(l1)[..., None]
    o_ext = (w0 * o0 + w1 * o1) / (w0 + w1)
    excess = np.abs(o_ext - o_true) / (2e-2 + 2e-2 * np.abs(o_true))
    assert excess.max() > 10.0


def test_disjoint_key_merge_is_attention():
    """The same LSE-weighted merge is exact when the two parts hold disjoint keys."""
    q, k, v = _rand(1, 1, 48, 16, 10)
    sc = 0.25
    o_true, lse_true = oracle.sdpa_fwd(q, k, v, False, sc)
    parts = [(0, 20), (20, 48)]
    outs, lses = [], []
    # Logits over all keys, then restricted to each disjoint key range.
    s_all = oracle.scores(q, k, sc)
    for a, b in parts:
        s = s_all[..., a:b]
        m = s.max(-1, keepdims=True)
        e = np.exp(s - m)
        outs.append((e @ v[:, :, a:b]) / e.sum(-1, keepdims=True))
        lses.append(m[..., 0] + np.log(e.sum(-1)))
    w = [np.exp(l - lse_true)[..., None] for l in lses]
    np.testing.assert_allclose(w[0] * outs[0] + w[1] * outs[1], o_true, atol=1e-12)


def test_key_shift_invariance():
    """k_j <- k_j + w for every j leaves O unchanged and shifts LSE_i by scale*q_i.w."""
    q, k, v = _rand(1, 3, 30, 8, 12)
    w = np.array([0.5, -1.0, 0.25, 0.0, 2.0, -0.75, 1.5, 0.125])
    o, lse = oracle.sdpa_fwd(q, k, v, False, 0.4)
    o2, lse2 = oracle.sdpa_fwd(q, k + w, v, False, 0.4)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2 - lse, 0.4 * (q @ w), atol=1e-12)


def test_noncausal_permutation_equivariance():
    q, k, v = _rand(2, 2, 27, 8, 13)
    perm = np.random.default_rng(0).permutation(27)
    o, lse = oracle.sdpa_fwd(q, k, v, False, 0.35)
    o2, lse2 = oracle.sdpa_fwd(q, k[:, :, perm], v[:, :, perm], False, 0.35)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, atol=1e-12)


@pytest.mark.parametrize("B,H,L,d,causal", [
    (1, 2, 1, 64, False), (1, 2, 17, 64, True), (2, 3, 129, 64, False), (1, 2, 200, 128, True),
    (1, 1, 96, 256, True), (1, 1, 70, 512, True), (1, 1, 70, 512, False),
])
def test_matches_torch_sdpa_float64(B, H, L, d, causal):
    """Library special case: PyTorch SDPA in float64 on the CPU (the first page's gate)
    and torch.logsumexp of explicitly masked logits for the LSE."""
    q, k, v = _rand(B, H, L, d, 100 + L + d)
    sc = 1.0 / math.sqrt(d)
    o, lse = oracle.sdpa_fwd(q, k, v, causal, sc, nthreads=3)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    o_t = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=sc)
    s_t = torch.matmul(tq, tk.transpose(-1, -2)) * sc
    if causal:
        s_t = s_t.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), float("-inf"))
    lse_t = torch.logsumexp(s_t, dim=-1)
    np.testing.assert_allclose(o, o_t.numpy(), atol=1e-10)
    np.testing.assert_allclose(lse, lse_t.numpy(), atol=1e-10)


def test_rows_entry_matches_full():
    q, k, v = _rand(2, 2, 45, 32, 14)
    o, lse = oracle.sdpa_fwd(q, k, v, True, 0.2)
    rows = np.array([0, 1, 44, 45, 100, 179])
    o_r, lse_r, nt = oracle.sdpa_fwd_rows(q, k, v, True, 0.2, rows)
    assert nt >= 1
    np.testing.assert_array_equal(o_r, o.reshape(-1, 32)[rows])
    np.testing.assert_array_equal(lse_r, lse.reshape(-1)[rows])
    with pytest.raises(IndexError):
        oracle.sdpa_fwd_rows(q, k, v, True, 0.2, [180])


def test_thread_count_does_not_change_results():
    q, k, v = _rand(1, 4, 65, 16, 15)
    o1, l1 = oracle.sdpa_fwd(q, k, v, True, 0.3, nthreads=1)
    o4, l4 = oracle.sdpa_fwd(q, k, v, True, 0.3, nthreads=4)
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(l1, l4)


# ---------------------------------------------------------------------------------------
# Mutation tests: plant a plausible mistake in a copy of the oracle's C source (on the
# CPU), build it, and check that the pins above would have caught it.
# ---------------------------------------------------------------------------------------
_SRC = os.path.join(os.path.dirname(oracle.__file__), "sdpa_oracle.c")
MUTANTS = {
    "dropped_scale": ("srow[j] = scale * acc;", "srow[j] = acc;"),
    "transposed_qk": ("const double *qi = q + (bh * L + i) * d;\n    const double *kh = k + bh * L * d;",
                      "const double *qi = k + (bh * L + i) * d;\n    const double *kh = q + bh * L * d;"),
    "half_length_dot": ("for (long t = 0; t < d; ++t)\n            acc += qi[t] * kj[t];",
                        "for (long t = 0; t < d / 2; ++t)\n            acc += qi[t] * kj[t];"),
    "causal_excludes_diagonal": ("long jmax = causal ? i + 1 : L; /* keys j <= i",
                                 "long jmax = causal ? i : L; /* keys j <= i"),
    "causal_mask_ignored": ("long jmax = causal ? i + 1 : L; /* keys j <= i",
                            "long jmax = L; /* keys j <= i"),
    "lse_without_max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "exp_sign_flipped": ("srow[j] = exp(srow[j] - m);\n        l += srow[j];",
                         "srow[j] = exp(m - srow[j]);\n        l += srow[j];"),
    "no_max_subtraction": ("srow[j] = exp(srow[j] - m);\n        l += srow[j];",
                           "srow[j] = exp(srow[j]);\n        l += srow[j];"),
    "missing_divide": ("o_row[c] = acc / l;", "o_row[c] = acc;"),
    "v_index_transposed": ("acc += srow[j] * vh[j * d + c];", "acc += srow[j] * vh[(c * d + j) % (L * d)];"),
}


def _build_mutant(name, tmp_path):
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
    lib.oracle_sdpa_fwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, ctypes.c_double, i]
    lib.oracle_sdpa_fwd.restype = i
    return lib


def _run_lib(lib, ex):
    q, k, v = (np.ascontiguousarray(_as4(ex[n])) for n in ("q", "k", "v"))
    L, d = ex["L"], ex["d"]
    o = np.empty((1, 1, L, d))
    lse = np.empty((1, 1, L))
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    lib.oracle_sdpa_fwd(P(q), P(k), P(v), P(o), P(lse), 1, 1, L, d, int(ex["causal"]), ex["scale"], 1)
    return o[0, 0], lse[0, 0]


def _pins_pass(lib):
    for ex in _examples():
        o, lse = _run_lib(lib, ex)
        o_ref, lse_ref = _expected(ex)
        if not (np.allclose(o, o_ref, rtol=0, atol=1e-9) and np.allclose(lse, lse_ref, rtol=0, atol=1e-9)):
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    lib = _build_mutant(name, tmp_path)
    with np.errstate(all="ignore"):
        assert not _pins_pass(lib), f"the worked examples did not catch mutant {name}"


def test_unmutated_copy_passes(tmp_path):
    """Control for the mutation tests: the anchors exist and the clean source passes."""
    for name in MUTANTS:
        old, _ = MUTANTS[name]
        assert open(_SRC).read().count(old) == 1
    lib = ctypes.CDLL(oracle.build())
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_sdpa_fwd.argtypes = [dp, dp, dp, dp, dp] + [ctypes.c_int] * 5 + [ctypes.c_double, ctypes.c_int]
    lib.oracle_sdpa_fwd.restype = ctypes.c_int
    assert _pins_pass(lib)
