"""Pins for the oracle's backward pass (the gradient of <y, dy> with respect to q, k,
v, u): every check compares it with something other than itself -- central finite
differences of the forward oracle (pinned on its own), the closed-form gradient of
causal linear attention for the Residual aggregation, and invariants.  A planted
mistake in a copy of the oracle must make one of them fail.

Pages cited:
  [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
  [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
           (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
"""
import ctypes
import os
import re
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from mc_inputs import GRM, MEAN, RESIDUAL, SOUP, SSC, make_inputs

NAMES = ("dq", "dk", "dv", "du")


def _inputs(B, H, L, d, seed):
    q, k, v, u = [t.double().numpy() for t in make_inputs(B, H, L, d, seed, "f32")]
    dy = np.random.default_rng(seed + 100).standard_normal(q.shape)
    return q, k, v, u, dy


def _finite_differences(args, dy, C, mode, topk, eps=1e-6, given_sel=None):
    """d<y, dy>/dX for X in q, k, v, u, element by element (central differences)."""
    out = {}
    for j, name in enumerate(NAMES):
        X = args[j]
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            val = []
            for sgn in (1.0, -1.0):
                a = list(args)
                a[j] = X.copy()
                a[j][idx] += sgn * eps
                val.append(np.sum(oracle.forward(*a, C, mode, topk, given_sel=given_sel)["y"] * dy))
            fd[idx] = (val[0] - val[1]) / (2 * eps)
        out[name] = fd
    return out


@pytest.mark.parametrize("mode,topk", [(RESIDUAL, 0), (GRM, 0), (SOUP, 0), (SSC, 1), (SSC, 0), (MEAN, 0)])
@pytest.mark.parametrize("L,C", [(10, 4), (9, 3)])
def test_backward_matches_finite_differences(mode, topk, L, C):
    """The gradient is the derivative of the (separately pinned) forward: central
    differences in fp64 agree to ~1e-10; the bound leaves room for the O(eps^2) term."""
    q, k, v, u, dy = _inputs(1, 1, L, 3, 3 + L)
    g = oracle.backward(q, k, v, u, dy, C, mode, topk)
    fd = _finite_differences([q, k, v, u], dy, C, mode, topk)
    for n in NAMES:
        scale = max(np.abs(fd[n]).max(), 1e-12)
        assert np.abs(g[n] - fd[n]).max() <= 1e-7 * scale + 1e-12, (n, mode, topk)


def test_backward_on_a_given_selection():
    """With the SSC selection given (as the forward takes it), the backward is the
    derivative of the forward evaluated on that selection: central differences of the
    forward with the same given selection agree.  The selection here is the router's
    choice reversed (the lowest-scoring cached segment instead of the highest), so it is
    not the one the router would make; and giving the router's own choice reproduces
    the ungiven backward exactly."""
    L, C, topk = 10, 3, 1
    q, k, v, u, dy = _inputs(1, 1, L, 3, 41)
    fwd = oracle.forward(q, k, v, u, C, SSC, topk)
    base = oracle.backward(q, k, v, u, dy, C, SSC, topk)
    same = oracle.backward(q, k, v, u, dy, C, SSC, topk, given_sel=fwd["sel"])
    for n in NAMES:
        np.testing.assert_array_equal(same[n], base[n])
    # the lowest-scoring cached segment of every token (-1 where there is none)
    kbar = np.stack([k[0, 0, n * C:min(L, n * C + C)].mean(0) for n in range((L + C - 1) // C)])
    other = np.full((1, 1, L, topk), -1, np.int32)
    for t in range(L):
        s = t // C
        if s > 0:
            other[0, 0, t, 0] = int(np.argmin(kbar[:s] @ u[0, 0, t]))
    assert np.any(other != fwd["sel"])
    g = oracle.backward(q, k, v, u, dy, C, SSC, topk, given_sel=other)
    fd = _finite_differences([q, k, v, u], dy, C, SSC, topk, given_sel=other)
    for n in NAMES:
        scale = max(np.abs(fd[n]).max(), 1e-12)
        assert np.abs(g[n] - fd[n]).max() <= 1e-7 * scale + 1e-12, n
        assert np.abs(g[n] - base[n]).max() > 1e-6 * scale, n  # a different function of the inputs


def _causal_la_grads(q, k, v, dy):
    """Gradients of <LA(q, k, v), dy>, LA_t = sum_{j<=t} v_j (k_j . q_t) ([MC-ja §2 eq. 2],
    phi = id, no 1/Z), in matrix form: A = tril(Q K^T), Y = A V."""
    L = q.shape[-2]
    mask = np.tril(np.ones((L, L)))
    dA = np.einsum("...td,...jd->...tj", dy, v) * mask
    dq = np.einsum("...tj,...jd->...td", dA, k)
    dk = np.einsum("...tj,...td->...jd", dA, q)
    A = np.einsum("...td,...jd->...tj", q, k) * mask
    dv = np.einsum("...tj,...td->...jd", A, dy)
    return dq, dk, dv


@pytest.mark.parametrize("C", [64, 16, 5, 1])
def test_residual_backward_is_causal_la_backward(C):
    """Residual MC collapses to causal linear attention for every segmentation
    ([MC-ja §3.1 GRM paragraph]), so its gradient is that of linear attention."""
    q, k, v, u, dy = _inputs(1, 2, 64, 8, 5)
    g = oracle.backward(q, k, v, u, dy, C, RESIDUAL)
    dq, dk, dv = _causal_la_grads(q, k, v, dy)
    for a, b in ((g["dq"], dq), (g["dk"], dk), (g["dv"], dv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-10)
    assert not g["du"].any()


@pytest.mark.parametrize("C", [16, 7])
def test_mean_backward_is_scaled_causal_la_backward(C):
    """Mean: y_t = LA_t / (s_t + 1), the gradient of LA with dy_t scaled by 1 / (s_t + 1)."""
    q, k, v, u, dy = _inputs(1, 1, 48, 8, 6)
    g = oracle.backward(q, k, v, u, dy, C, MEAN)
    w = 1.0 / (np.arange(48) // C + 1)
    dq, dk, dv = _causal_la_grads(q, k, v, dy * w[:, None])
    for a, b in ((g["dq"], dq), (g["dk"], dk), (g["dv"], dv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("mode,topk", [(RESIDUAL, 0), (GRM, 0), (SOUP, 0), (SSC, 2), (MEAN, 0)])
def test_backward_euler_identities(mode, topk):
    # y is homogeneous of degree one in q and in v (the gates depend on neither, every memory is
    # linear in v: [MC-ja §3 eq. 4b-5, §3.1 eq. 7-10]), so <dq, q> = <dv, v> = <dy, y> per (b, h);
    # with constant gates (Residual, Mean) y is also linear in k and <dk, k> = <dy, y>.
    q, k, v, u, dy = _inputs(1, 2, 300, 16, 5)
    y = oracle.forward(q, k, v, u, 64, mode, topk)["y"]
    g = oracle.backward(q, k, v, u, dy, 64, mode, topk)
    ref = (dy * y).sum(axis=(2, 3))
    pairs = [("dq", q), ("dv", v)] + ([("dk", k)] if mode in (RESIDUAL, MEAN) else [])
    for name, x in pairs:
        got = (g[name] * x).sum(axis=(2, 3))
        assert np.abs(got - ref).max() <= 1e-10 * np.abs(ref).max(), (mode, name)


def test_backward_is_linear_in_dy():
    q, k, v, u, dy = _inputs(1, 2, 40, 6, 7)
    dy2 = np.random.default_rng(1).standard_normal(dy.shape)
    a = oracle.backward(q, k, v, u, dy, 8, GRM)
    b = oracle.backward(q, k, v, u, dy2, 8, GRM)
    c = oracle.backward(q, k, v, u, dy - 2.0 * dy2, 8, GRM)
    for n in NAMES:
        np.testing.assert_allclose(c[n], a[n] - 2.0 * b[n], rtol=1e-9, atol=1e-11)


def test_ssc_backward_limits():
    """topk >= N-1 selects every cached segment (GRM); Soup is GRM for a linear memory."""
    q, k, v, u, dy = _inputs(1, 1, 40, 6, 8)
    ref = oracle.backward(q, k, v, u, dy, 8, GRM)
    for mode, topk in ((SSC, 4), (SSC, 10), (SOUP, 0)):
        g = oracle.backward(q, k, v, u, dy, 8, mode, topk)
        for n in NAMES:
            np.testing.assert_allclose(g[n], ref[n], rtol=1e-10, atol=1e-12)


_MUTATIONS = [
    ("softmax backward misses the mean term", r"const double dr = g\[c\] \* \(dg\[c\] - sgd\);",
     "const double dr = g[c] * dg[c];"),
    ("online pool gradient not divided by the count", r"J->dk\[\(size_t\)j \* d \+ b\] \+= dr \* ut\[b\] / cnt;",
     "J->dk[(size_t)j * d + b] += dr * ut[b];"),
    ("cached gradient transposed", r"Gi\[\(size_t\)a \* d \+ b\] \+= g\[c\] \* dyt\[a\] \* qt\[b\];",
     "Gi[(size_t)a * d + b] += g[c] * dyt[b] * qt[a];"),
    ("pooled key gradient dropped", r"dkj\[b\] \+= dkbar\[\(size_t\)n \* d \+ b\] / \(double\)\(t1 - t0\);", ";"),
    ("online read skips the current token", r"for \(int j = t0; j <= t; \+\+j\) \{\n                const double \*kj",
     "for (int j = t0; j < t; ++j) {\n                const double *kj"),
    ("dq reads M instead of M^T", r"dqt\[b\] \+= g\[c\] \* M\[\(size_t\)a \* d \+ b\] \* dyt\[a\];",
     "dqt[b] += g[c] * M[(size_t)b * d + a] * dyt[a];"),
]


@pytest.mark.parametrize("desc,pat,rep", _MUTATIONS, ids=[m[0] for m in _MUTATIONS])
def test_backward_pins_catch_planted_mistake(desc, pat, rep):
    """Plant one plausible mistake in a copy of the oracle's backward (on the CPU) and
    check that a pin fails."""
    oracle._load()
    src = open(oracle._SRC).read()
    mutated, n = re.subn(pat, rep, src)
    assert n >= 1, f"mutation pattern not found: {desc}"
    tmpd = tempfile.mkdtemp(prefix="mc_oracle_bmut_")
    try:
        c = os.path.join(tmpd, "m.c")
        so = os.path.join(tmpd, "libm.so")
        open(c, "w").write(mutated)
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                        "-ffp-contract=off", c, "-o", so, "-lm"], check=True)
        saved = oracle._lib
        lib = ctypes.CDLL(so)
        for fn in ("mc_oracle_forward", "mc_oracle_backward"):
            getattr(lib, fn).argtypes = getattr(saved, fn).argtypes
            getattr(lib, fn).restype = ctypes.c_int
        oracle._lib = lib
        failed = 0
        try:
            for pin in (lambda: test_backward_matches_finite_differences(GRM, 0, 10, 4),
                        lambda: test_residual_backward_is_causal_la_backward(5)):
                try:
                    pin()
                except AssertionError:
                    failed += 1
        finally:
            oracle._lib = saved
        assert failed >= 1, f"no pin caught: {desc}"
    finally:
        shutil.rmtree(tmpd, ignore_errors=True)
