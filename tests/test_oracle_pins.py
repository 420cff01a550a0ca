"""Pins for the fp64 oracle: each test checks it against something other than
itself -- a hand-worked example, a closed form, a special case that reduces to
a textbook routine (causal linear attention, gated token-level attention, a
plain matrix product), an invariant of the mathematics, or brute force.

Pages cited:
  [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
  [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
           (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
The SWLA pins (sliding-window linear attention, c = 2, [MC-ja §3.1 eq. 28-29])
reduce it to closed forms written here with numpy: a constant decay (a decayed
causal linear attention), alpha = 0 (a two-token window), alpha = beta = lambda
= 1 (each past token counted twice, once within its own segment's window).
"""
import os
import re
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from mc_inputs import GRM, MEAN, RESIDUAL, SOUP, SSC, make_inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def _inputs(B, H, L, d, seed, dtype="f32"):
    return [t.double().numpy() for t in make_inputs(B, H, L, d, seed, dtype)]


def causal_la(q, k, v):
    """Plain causal linear attention, y_t = sum_{j<=t} v_j (k_j . q_t) -- [MC-ja §2 eq. 2], phi = id, no 1/Z."""
    L = q.shape[-2]
    scores = np.einsum("...td,...jd->...tj", q, k)
    scores = scores * np.tril(np.ones((L, L)))
    return np.einsum("...tj,...jd->...td", scores, v)


def blockwise_la(q, k, v, C):
    """Causal linear attention restricted to each segment (block-diagonal causal mask)."""
    L = q.shape[-2]
    t = np.arange(L)
    mask = (t[:, None] >= t[None, :]) & (t[:, None] // C == t[None, :] // C)
    scores = np.einsum("...td,...jd->...tj", q, k) * mask
    return np.einsum("...tj,...jd->...td", scores, v)


def seg_number(L, C):
    return (np.arange(L) // C + 1).astype(np.float64)


# ---------------------------------------------------------------- worked example

def _load_golden(name):
    vals = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            vals[key.strip()] = np.array([float(x) for x in rest.split()], np.float64)
    return vals


def test_hand_worked_example():
    """Hand-derived d=2 example (tests/golden/hand_example_d2.txt): Residual [MC-ja §3.1 eq. 7],
    GRM [MC-ja §3.1 eq. 9-10], SSC [MC-sum §3.4], the cached states [MC-ja §3 eq. 4b]."""
    g = _load_golden("hand_example_d2.txt")
    q, k, v, u = (g[n].reshape(1, 1, 3, 2) for n in "qkvu")
    res = oracle.forward(q, k, v, u, 2, RESIDUAL)
    np.testing.assert_allclose(res["y"].reshape(-1), g["residual"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(res["states"][0, 0, 0].reshape(-1), g["state0"], atol=1e-12)
    np.testing.assert_allclose(res["states"][0, 0, 1].reshape(-1), g["state1"], atol=1e-12)
    for mode in (GRM, SOUP):
        y = oracle.forward(q, k, v, u, 2, mode)["y"]
        np.testing.assert_allclose(y.reshape(-1), g["grm"], rtol=0, atol=1e-12)
    y0 = oracle.forward(q, k, v, u, 2, SSC, topk=0)["y"]
    np.testing.assert_allclose(y0.reshape(-1), g["ssc_top0"], atol=1e-12)
    y1 = oracle.forward(q, k, v, u, 2, SSC, topk=1)["y"]
    np.testing.assert_allclose(y1.reshape(-1), g["ssc_top1"], atol=1e-12)


# ---------------------------------------------------------------- states

@pytest.mark.parametrize("L,C", [(96, 32), (100, 32), (64, 64), (50, 7)])
def test_states_are_segment_gemms(L, C):
    """Cached state of segment n is V_n^T K_n (a plain matrix product) [MC-ja §3 eq. 4b]."""
    q, k, v, u = _inputs(2, 2, L, 8, 11)
    st = oracle.forward(q, k, v, u, C, GRM)["states"]
    N = (L + C - 1) // C
    assert st.shape == (2, 2, N, 8, 8)
    for n in range(N):
        sl = slice(n * C, min(L, n * C + C))
        ref = np.einsum("bhta,bhtc->bhac", v[:, :, sl], k[:, :, sl])
        np.testing.assert_allclose(st[:, :, n], ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- collapse invariants

@pytest.mark.parametrize("C", [128, 32, 8, 2, 37, 1])
def test_residual_equals_causal_la_for_any_segmentation(C):
    """Residual MC over a linear memory collapses to plain linear attention
    ([MC-ja §3.1, GRM paragraph]; [MC-sum §3.1])."""
    q, k, v, u = _inputs(1, 2, 128, 16, 1)
    y = oracle.forward(q, k, v, u, C, RESIDUAL)["y"]
    np.testing.assert_allclose(y, causal_la(q, k, v), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("mode,topk", [(GRM, 0), (SOUP, 0), (SSC, 3), (SSC, 0), (RESIDUAL, 0)])
def test_single_segment_is_plain_recurrent_model(mode, topk):
    """N = 1: nothing is cached, MC is the plain recurrent model [MC-sum §2.2]."""
    q, k, v, u = _inputs(1, 2, 64, 16, 2)
    for C in (64, 100):
        y = oracle.forward(q, k, v, u, C, mode, topk)["y"]
        np.testing.assert_allclose(y, causal_la(q, k, v), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("C", [16, 5])
def test_grm_with_constant_gates(C):
    """u = 0 gives equal gates 1/s over the s memories: y_t = LA_t / s_t
    ([MC-ja §3.1]: constant gates make GRM the Residual variant, up to the softmax scale)."""
    q, k, v, u = _inputs(1, 1, 80, 8, 3)
    u = np.zeros_like(u)
    y = oracle.forward(q, k, v, u, C, GRM)["y"]
    ref = causal_la(q, k, v) / seg_number(80, C)[:, None]
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("C", [16, 5, 1, 80])
def test_mean_is_linear_attention_over_the_memory_count(C):
    """Memory caching added after training averages the s + 1 memories with equal
    weights ([MC-ja, variants appendix, post-training MC]); for a linear memory their
    sum is plain causal linear attention, so y_t = LA_t / (s_t + 1) whatever u is."""
    q, k, v, u = _inputs(1, 2, 80, 8, 4)
    y = oracle.forward(q, k, v, u, C, MEAN)["y"]
    ref = causal_la(q, k, v) / seg_number(80, C)[:, None]
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)
    y0 = oracle.forward(q, k, v, np.zeros((0,)), C, MEAN)["y"]  # u is not read
    np.testing.assert_array_equal(y0, y)


def test_log_segmentation_worked_example():
    """The pages' worked example of the logarithmic segmentation (tests/golden/log_segments.txt)."""
    vals = _load_golden("log_segments.txt")
    for L, lens in vals.items():
        off = oracle.log_segments(int(L))
        assert list(np.diff(off)) == [int(x) for x in lens]


@pytest.mark.parametrize("L", [1, 2, 37, 64, 100, 1000, 65535])
def test_log_segmentation_properties(L):
    """One segment per set bit of L, distinct powers of two, longest first, N <= log2 L + 1."""
    lens = np.diff(oracle.log_segments(L))
    assert lens.sum() == L and len(lens) == bin(L).count("1")
    assert all(x & (x - 1) == 0 for x in lens) and list(lens) == sorted(lens, reverse=True)
    assert len(lens) <= int(np.log2(L)) + 1


VAR_SEGS = [[0, 40, 56, 60, 61, 64], [0, 1, 2, 3, 64], [0, 64]]


@pytest.mark.parametrize("off", VAR_SEGS + [None])
def test_variable_segments_residual_is_causal_la(off):
    """Residual collapses to causal LA for ANY segmentation, constant or not."""
    q, k, v, u = _inputs(1, 2, 64, 8, 21)
    off = off if off is not None else oracle.log_segments(64 - 1) + []
    L = off[-1]
    q, k, v, u = (x[..., :L, :] for x in (q, k, v, u))
    y = oracle.forward(q, k, v, u, None, RESIDUAL, seg_off=off)["y"]
    np.testing.assert_allclose(y, causal_la(q, k, v), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("off", VAR_SEGS)
def test_variable_segments_constant_gates(off):
    """u = 0 (GRM) or Mean: equal gates over the s + 1 memories, y_t = LA_t / (s_t + 1)."""
    q, k, v, u = _inputs(1, 1, 64, 8, 22)
    s_of = np.searchsorted(np.asarray(off), np.arange(64), side="right")  # s_t + 1
    ref = causal_la(q, k, v) / s_of[:, None]
    for mode, uu in ((GRM, np.zeros_like(u)), (MEAN, u)):
        y = oracle.forward(q, k, v, uu, None, mode, seg_off=off)["y"]
        np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("mode,topk", [(GRM, 0), (SSC, 1), (SOUP, 0), (MEAN, 0)])
@pytest.mark.parametrize("off", VAR_SEGS)
def test_variable_segments_state_form_matches_twin(off, mode, topk):
    q, k, v, u = _inputs(1, 2, 64, 8, 23)
    a = oracle.forward(q, k, v, u, None, mode, topk, seg_off=off)
    b = oracle.bruteforce(q, k, v, u, None, mode, topk, seg_off=off)
    np.testing.assert_allclose(a["y"], b, rtol=1e-10, atol=1e-11)
    for n in range(len(off) - 1):  # the cached states are the segments' V^T K
        K, V = k[..., off[n]:off[n + 1], :], v[..., off[n]:off[n + 1], :]
        np.testing.assert_allclose(a["states"][:, :, n], np.einsum("bhta,bhtc->bhac", V, K), rtol=1e-12,
                                   atol=1e-12)


def test_constant_boundaries_match_the_segment_length():
    q, k, v, u = _inputs(1, 2, 70, 8, 24)
    off = list(range(0, 70, 16)) + [70]
    for mode, topk in ((GRM, 0), (SSC, 2)):
        a = oracle.forward(q, k, v, u, 16, mode, topk)
        b = oracle.forward(q, k, v, u, None, mode, topk, seg_off=off)
        np.testing.assert_array_equal(a["y"], b["y"])


def test_one_token_segments_are_gated_attention():
    """N = L: every token is its own segment, the pool of a one-token segment is its
    key, and GRM becomes y_t = sum_{i<=t} softmax_i(u_t . k_i) v_i (k_i . q_t)
    ([MC-sum §2.2 and §4.1]); written here as a dense masked softmax."""
    q, k, v, u = _inputs(1, 2, 40, 8, 4)
    y = oracle.forward(q, k, v, u, 1, GRM)["y"]
    L = 40
    logits = np.einsum("...td,...id->...ti", u, k)
    logits = np.where(np.tril(np.ones((L, L), bool)), logits, -np.inf)
    w = np.exp(logits - logits.max(-1, keepdims=True))
    w /= w.sum(-1, keepdims=True)
    kq = np.einsum("...td,...id->...ti", q, k)
    ref = np.einsum("...ti,...id->...td", w * kq, v)
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("C", [16, 7])
def test_soup_equals_grm_for_linear_memory(C):
    """Memory Soup and GRM coincide for a linear memory ([MC-ja §3.1, SWLA paragraph];
    [MC-sum §3.3]).  The oracle forms the soup matrix literally, so this is a real cross-check."""
    q, k, v, u = _inputs(2, 1, 96, 8, 5)
    a = oracle.forward(q, k, v, u, C, GRM)["y"]
    b = oracle.forward(q, k, v, u, C, SOUP)["y"]
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_ssc_limits():
    """SSC with topk >= N-1 selects every cached memory (= GRM); topk = 0 keeps only the
    online memory, i.e. linear attention inside each segment ([MC-sum §3.4])."""
    q, k, v, u = _inputs(1, 2, 96, 8, 6)
    C = 12
    N = 8
    grm = oracle.forward(q, k, v, u, C, GRM)["y"]
    for kk in (N - 1, N + 5):
        np.testing.assert_allclose(oracle.forward(q, k, v, u, C, SSC, kk)["y"], grm, rtol=1e-11, atol=1e-12)
    y0 = oracle.forward(q, k, v, u, C, SSC, 0)["y"]
    np.testing.assert_allclose(y0, blockwise_la(q, k, v, C), rtol=1e-10, atol=1e-12)


def test_ssc_selection_matches_a_sort():
    """The router's top-k ([MC-sum §3.4]) equals a stable sort of the fp32 scores, descending,
    lower index first on ties; the pooled keys are plain means of each segment's keys."""
    q, k, v, u = _inputs(1, 2, 120, 8, 7)
    C, topk = 10, 3
    out = oracle.forward(q, k, v, u, C, SSC, topk)
    sel = out["sel"]
    kbar = k.reshape(1, 2, 12, 10, 8).mean(axis=3)
    for h in range(2):
        for t in range(120):
            s = t // C
            r = (u[0, h, t] @ kbar[0, h, :s].T).astype(np.float32)
            order = sorted(range(s), key=lambda i: (-r[i], i))[:topk]
            got = [int(x) for x in sel[0, h, t] if x >= 0]
            assert got == order, (h, t)


def test_ssc_ties_go_to_lower_index():
    """Equal router scores: the lower segment index wins (deterministic tie rule)."""
    q, k, v, u = _inputs(1, 1, 40, 4, 8)
    C = 10
    k[0, 0, 10:20] = k[0, 0, 0:10]  # segments 0 and 1 have equal pooled keys
    k[0, 0, 20:30] = -k[0, 0, 0:10]
    out = oracle.forward(q, k, v, u, C, SSC, 1)
    sel = out["sel"][0, 0, 30:40, 0]
    kb0 = k[0, 0, 0:10].mean(0)
    for j, t in enumerate(range(30, 40)):
        r0 = np.float32(u[0, 0, t] @ kb0)
        r2 = np.float32(u[0, 0, t] @ (-kb0))
        assert sel[j] == (0 if r0 >= r2 else 2)


def _router_case(a):
    """d = 2, one token per segment (so each cached pooled key is that token's key),
    k_i = (a_i, 0) and u_t = (1, 0): the router score of token t against cached segment
    i < t is exactly a_i."""
    L = len(a) + 1
    rng = np.random.default_rng(21)
    q = rng.standard_normal((1, 1, L, 2))
    v = rng.standard_normal((1, 1, L, 2))
    k = np.zeros((1, 1, L, 2))
    k[0, 0, :len(a), 0] = a
    k[0, 0, len(a), 0] = 0.375
    u = np.zeros((1, 1, L, 2))
    u[..., 0] = 1.0
    return q, k, v, u


def test_ssc_gap_hand_case():
    """The router's near-tie record, worked by hand ([MC-sum §3.4]: the k largest cached
    scores).  Scores a_i of the cached segments, exact binary fractions:
      a = [1/2, 1/4, 1/2 + 2^-10, 1/4 + 2^-10, 1/8, 1/2 + 2^-11, 1/2 + 2^-30].
    Ranking is in fp32, where 1/2 + 2^-30 rounds to 1/2 and ties with segment 0 (the lower
    index wins); the gap is the fp64 distance between the last chosen score and the best
    left out, infinite when nothing is left out.  Token t sees segments 0..t-1.
      topk 2: t=3 [2,0] gap 1/4; t=4,5 [2,0] gap 1/4 - 2^-10; t=6,7 [2,5] gap 2^-11.
      topk 3: t=3 [2,0,1] inf; t=4,5 [2,0,3] gap 2^-10; t=6 [2,5,0] gap 1/4 - 2^-10;
              t=7 [2,5,0] gap 2^-30 (fp64 would have ranked segment 6 third)."""
    a = [0.5, 0.25, 0.5 + 2**-10, 0.25 + 2**-10, 0.125, 0.5 + 2**-11, 0.5 + 2**-30]
    q, k, v, u = _router_case(a)
    inf = np.inf
    want = {2: {3: ([2, 0], 0.25), 4: ([2, 0], 0.25 - 2**-10), 5: ([2, 0], 0.25 - 2**-10),
                6: ([2, 5], 2**-11), 7: ([2, 5], 2**-11)},
            3: {3: ([2, 0, 1], inf), 4: ([2, 0, 3], 2**-10), 5: ([2, 0, 3], 2**-10),
                6: ([2, 5, 0], 0.25 - 2**-10), 7: ([2, 5, 0], 2**-30)}}
    for topk, rows in want.items():
        out = oracle.forward(q, k, v, u, 1, SSC, topk)
        for t, (sel, gap) in rows.items():
            assert [int(x) for x in out["sel"][0, 0, t]] == sel, (topk, t)
            assert out["gap"][0, 0, t] == gap, (topk, t, out["gap"][0, 0, t], gap)
        # fewer cached segments than topk: all of them, nothing left out
        assert np.isinf(out["gap"][0, 0, :3]).all()


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("mode,topk", [(RESIDUAL, 0), (GRM, 0), (SOUP, 0), (SSC, 2)])
def test_causality(mode, topk):
    """y_t depends on tokens j <= t only: changing later tokens leaves it unchanged.
    (This pins the online pool to keys seen so far and the online memory to the
    update before the read.)"""
    q, k, v, u = _inputs(1, 1, 60, 8, 9)
    C, t = 8, 27
    a = oracle.forward(q, k, v, u, C, mode, topk)["y"]
    q2, k2, v2, u2 = (x.copy() for x in (q, k, v, u))
    rng = np.random.default_rng(0)
    for x in (q2, k2, v2, u2):
        x[..., t + 1:, :] = rng.standard_normal(x[..., t + 1:, :].shape)
    b = oracle.forward(q2, k2, v2, u2, C, mode, topk)["y"]
    np.testing.assert_array_equal(a[..., : t + 1, :], b[..., : t + 1, :])
    assert not np.allclose(a[..., t + 1:, :], b[..., t + 1:, :])


def test_linear_in_values():
    """The gates do not depend on v, so y is linear in v."""
    q, k, v, u = _inputs(1, 1, 48, 8, 10)
    v2 = _inputs(1, 1, 48, 8, 12)[2]
    C = 8
    for mode, topk in ((GRM, 0), (SSC, 2)):
        a = oracle.forward(q, k, v, u, C, mode, topk)["y"]
        b = oracle.forward(q, k, v2, u, C, mode, topk)["y"]
        c = oracle.forward(q, k, 2.0 * v - 3.0 * v2, u, C, mode, topk)["y"]
        np.testing.assert_allclose(c, 2.0 * a - 3.0 * b, rtol=1e-10, atol=1e-10)


def test_completed_segment_permutation():
    """A cached segment enters only through its final state and its key mean, both
    invariant to the order of its tokens; later outputs cannot see the order."""
    q, k, v, u = _inputs(1, 1, 64, 8, 13)
    C = 16
    perm = np.random.default_rng(1).permutation(16)
    q2, k2, v2, u2 = (x.copy() for x in (q, k, v, u))
    for x in (q2, k2, v2, u2):
        x[..., 0:16, :] = x[..., perm, :]
    for mode in (GRM, SSC):
        a = oracle.forward(q, k, v, u, C, mode, 1)["y"]
        b = oracle.forward(q2, k2, v2, u2, C, mode, 1)["y"]
        np.testing.assert_allclose(a[..., 16:, :], b[..., 16:, :], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("mode,topk", [(RESIDUAL, 0), (GRM, 0), (SOUP, 0), (SSC, 2), (SSC, 0), (MEAN, 0)])
@pytest.mark.parametrize("C", [16, 9, 1])
def test_state_form_matches_token_level_twin(mode, topk, C):
    """The state form equals the same sum regrouped by token (the twin never forms a memory)."""
    q, k, v, u = _inputs(1, 2, 48, 8, 14)
    a = oracle.forward(q, k, v, u, C, mode, topk)["y"]
    b = oracle.bruteforce(q, k, v, u, C, mode, topk)
    np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


def test_seg_mask_and_given_selection():
    """Partial evaluation and an externally given SSC selection reproduce the full run."""
    q, k, v, u = _inputs(1, 2, 64, 8, 15)
    C = 8
    full = oracle.forward(q, k, v, u, C, SSC, 2)
    mask = np.zeros(8, bool)
    mask[[2, 5]] = True
    part = oracle.forward(q, k, v, u, C, SSC, 2, seg_mask=mask)
    for n in (2, 5):
        np.testing.assert_array_equal(part["y"][..., n * C:(n + 1) * C, :], full["y"][..., n * C:(n + 1) * C, :])
    again = oracle.forward(q, k, v, u, C, SSC, 2, given_sel=full["sel"])
    np.testing.assert_array_equal(again["y"], full["y"])


# ---------------------------------------------------------------- the pins have teeth

# ---------------------------------------------------------------- SWLA (c = 2)

def _swla_scalars(B, H, L, seed, lo=0.5):
    rng = np.random.default_rng(seed)
    return (rng.uniform(lo, 1.0, (B, H, L)), rng.uniform(0.0, 1.0, (B, H, L)), rng.uniform(0.0, 1.0, (B, H, L)))


@pytest.mark.parametrize("mode,topk", [(RESIDUAL, 0), (GRM, 0), (SOUP, 0), (SSC, 2), (MEAN, 0)])
@pytest.mark.parametrize("C", [12, 5, 1])
def test_swla_state_form_matches_token_level_twin(mode, topk, C):
    """The recurrence of eq. 28 and its unrolled per-token weights agree."""
    q, k, v, u = _inputs(1, 2, 36, 6, 41)
    sw = _swla_scalars(1, 2, 36, 7)
    ref = oracle.forward(q, k, v, u, C, mode, topk, swla=sw)["y"]
    twin = oracle.bruteforce(q, k, v, u, C, mode, topk, swla=sw)
    assert np.max(np.abs(ref - twin)) <= 1e-12 * max(1.0, np.max(np.abs(twin)))


@pytest.mark.parametrize("mode,topk", [(RESIDUAL, 0), (GRM, 0), (SSC, 1)])
def test_swla_with_unit_decay_and_no_window_is_plain_mc(mode, topk):
    """alpha = lambda = 1, beta = 0 is the plain update M += v k^T."""
    q, k, v, u = _inputs(1, 2, 40, 8, 42)
    one, zero = np.ones((1, 2, 40)), np.zeros((1, 2, 40))
    a = oracle.forward(q, k, v, u, 10, mode, topk)
    b = oracle.forward(q, k, v, u, 10, mode, topk, swla=(one, zero, one))
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["states"], b["states"])


def test_swla_constant_decay_is_decayed_linear_attention():
    """beta = 0, lambda = 1, alpha = a: y_t = sum_{j<=t} a^(t-j) v_j (k_j . q_t) (one segment)."""
    q, k, v, u = _inputs(1, 1, 30, 5, 43)
    L, a = 30, 0.83
    t = np.arange(L)
    decay = np.where(t[:, None] >= t[None, :], a ** (t[:, None] - t[None, :]).clip(min=0), 0.0)
    want = np.einsum("tj,jd->td", np.einsum("td,jd->tj", q[0, 0], k[0, 0]) * decay, v[0, 0])
    sw = (np.full((1, 1, L), a), np.zeros((1, 1, L)), np.ones((1, 1, L)))
    got = oracle.forward(q, k, v, u, L, RESIDUAL, swla=sw)["y"][0, 0]
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))


def test_swla_zero_decay_is_a_two_token_window():
    """alpha = 0: y_t = lambda_t v_t (k_t . q_t) + beta_t v_{t-1} (k_{t-1} . q_t) (one segment)."""
    q, k, v, u = _inputs(1, 1, 25, 4, 44)
    _, be, la = _swla_scalars(1, 1, 25, 8)
    sw = (np.zeros((1, 1, 25)), be, la)
    got = oracle.forward(q, k, v, u, 25, RESIDUAL, swla=sw)["y"][0, 0]
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    want = la[0, 0][:, None] * np.sum(K * Q, 1)[:, None] * V
    want[1:] += be[0, 0, 1:][:, None] * np.sum(K[:-1] * Q[1:], 1)[:, None] * V[:-1]
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))


@pytest.mark.parametrize("C", [7, 1, 30])
def test_swla_window_does_not_cross_segments(C):
    """alpha = beta = lambda = 1, Residual: token j counts twice for every later token of its
    segment's window reach (j + 1 in the same segment), once otherwise."""
    q, k, v, u = _inputs(1, 1, 30, 4, 45)
    L = 30
    t = np.arange(L)
    twice = (t[:, None] > t[None, :]) & ((t[None, :] + 1) // C == t[None, :] // C)
    w = np.where(t[:, None] >= t[None, :], 1.0, 0.0) + twice
    want = np.einsum("tj,jd->td", np.einsum("td,jd->tj", q[0, 0], k[0, 0]) * w, v[0, 0])
    one = np.ones((1, 1, L))
    got = oracle.forward(q, k, v, u, C, RESIDUAL, swla=(one, one, one))["y"][0, 0]
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))


def test_swla_states_are_the_segments_last_memory():
    """The cached state of a segment is its memory after the segment's last token: with
    alpha = 0 that is beta_T v_{T-1} k_{T-1}^T + lambda_T v_T k_T^T."""
    q, k, v, u = _inputs(1, 1, 24, 3, 46)
    _, be, la = _swla_scalars(1, 1, 24, 9)
    st = oracle.forward(q, k, v, u, 8, GRM, swla=(np.zeros((1, 1, 24)), be, la))["states"][0, 0]
    K, V = k[0, 0], v[0, 0]
    for n in range(3):
        T = 8 * n + 7
        want = be[0, 0, T] * np.outer(V[T - 1], K[T - 1]) + la[0, 0, T] * np.outer(V[T], K[T])
        assert np.max(np.abs(st[n] - want)) <= 1e-13 * np.max(np.abs(want))


_MUTATIONS = [
    # (description, regex pattern, replacement)
    ("state transposed", r"M\[\(size_t\)a \* d \+ b\] \+= vt\[a\] \* kt\[b\];",
     "M[(size_t)a * d + b] += vt[b] * kt[a];"),
    ("swla window uses the current token", r"be \* vp\[a\] \* kp\[b\]", "be * vt[a] * kt[b]"),
    ("swla decays the new terms too", r"M\[\(size_t\)a \* d \+ b\] = al \* M\[\(size_t\)a \* d \+ b\] \+ be",
     "M[(size_t)a * d + b] = al * (M[(size_t)a * d + b]) * 1.0 + al * be"),
    ("swla window crosses segments", r"const double al = J->alpha\[t\], be = t > t0 \? J->beta\[t\] : 0\.0",
     "const double al = J->alpha[t], be = t > 0 ? J->beta[t] : 0.0"),
    ("pool not averaged", r"kbar\[\(size_t\)n \* d \+ b\] /= \(double\)\(t1 - t0\);", ";"),
    ("online pool over a wrong count", r"r\[s\] = dot\(ut, ksum, d\) / cnt;",
     "r[s] = dot(ut, ksum, d) / (cnt + 1.0);"),
    ("softmax sign", r"r\[i\] = exp\(r\[i\] - m\);", "r[i] = exp(m - r[i]);"),
    ("online gate index", r"add_matvec\(yt, g\[s\], Mon, qt, d\);", "add_matvec(yt, g[0], Mon, qt, d);"),
    ("dropped last cached term",
     r"for \(int i = 0; i < s; \+\+i\) add_matvec\(yt, g\[i\]",
     "for (int i = 0; i + 1 < s; ++i) add_matvec(yt, g[i]"),
    ("residual drops cached", r"for \(int i = 0; i < s; \+\+i\) add_matvec\(yt, 1\.0,",
     "for (int i = 1; i < s; ++i) add_matvec(yt, 1.0,"),
    ("ssc ties to higher index", r"if \(best < 0 \|\| fi > bv\) \{ /\* strict",
     "if (best < 0 || fi >= bv) { /* strict"),
    ("gap from the first chosen score", r"\*gap = fabs\(r\[idx\[want - 1\]\] - r\[best\]\);",
     "*gap = fabs(r[idx[0]] - r[best]);"),
    ("router ranks in fp64", r"float fi = \(float\)r\[i\];", "double fi = r[i];"),
    ("soup uses online twice", r"Mstar\[e\] \+= g\[i\] \* Mi\[e\];", "Mstar[e] += g[s] * Mi[e];"),
    ("segment end one token early", r"if \(J->seg_off\) return J->seg_off\[n \+ 1\];",
     "if (J->seg_off) return J->seg_off[n + 1] - (n + 2 < J->nseg ? 1 : 0);"),
    ("mean over the cached memories only", r"const double w = 1\.0 / \(double\)\(s \+ 1\);",
     "const double w = 1.0 / (double)(s > 0 ? s : 1);"),
]


def _run_pins_against(libpath):
    """Re-run a representative subset of the pins against a mutated oracle build."""
    import ctypes
    saved = oracle._lib
    try:
        lib = ctypes.CDLL(libpath)
        lib.mc_oracle_forward.argtypes = saved.mc_oracle_forward.argtypes
        lib.mc_oracle_forward.restype = ctypes.c_int
        lib.mc_oracle_bruteforce.argtypes = saved.mc_oracle_bruteforce.argtypes
        lib.mc_oracle_bruteforce.restype = ctypes.c_int
        lib.mc_oracle_forward_swla.argtypes = saved.mc_oracle_forward_swla.argtypes
        lib.mc_oracle_forward_swla.restype = ctypes.c_int
        lib.mc_oracle_bruteforce_swla.argtypes = saved.mc_oracle_bruteforce_swla.argtypes
        lib.mc_oracle_bruteforce_swla.restype = ctypes.c_int
        for fn in ("mc_oracle_forward_segments", "mc_oracle_bruteforce_segments"):
            getattr(lib, fn).argtypes = getattr(saved, fn).argtypes
            getattr(lib, fn).restype = ctypes.c_int
        oracle._lib = lib
        pins = [
            test_hand_worked_example,
            lambda: test_states_are_segment_gemms(96, 32),
            lambda: test_residual_equals_causal_la_for_any_segmentation(8),
            lambda: test_one_token_segments_are_gated_attention(),
            lambda: test_soup_equals_grm_for_linear_memory(7),
            lambda: test_ssc_limits(),
            lambda: test_ssc_ties_go_to_lower_index(),
            test_ssc_gap_hand_case,
            lambda: test_causality(GRM, 0),
            lambda: test_single_segment_is_plain_recurrent_model(GRM, 0),
            lambda: test_mean_is_linear_attention_over_the_memory_count(5),
            lambda: test_variable_segments_constant_gates(VAR_SEGS[0]),
            lambda: test_variable_segments_state_form_matches_twin(VAR_SEGS[0], GRM, 0),
            test_swla_constant_decay_is_decayed_linear_attention,
            test_swla_zero_decay_is_a_two_token_window,
            lambda: test_swla_window_does_not_cross_segments(7),
        ]
        failed = 0
        for p in pins:
            try:
                p()
            except AssertionError:
                failed += 1
        return failed
    finally:
        oracle._lib = saved


@pytest.mark.parametrize("desc,pat,rep", _MUTATIONS, ids=[m[0] for m in _MUTATIONS])
def test_pins_catch_planted_mistake(desc, pat, rep):
    """Plant one plausible mistake in a copy of the oracle (on the CPU) and check that at
    least one pin fails."""
    oracle._load()
    src = open(oracle._SRC).read()
    mutated, n = re.subn(pat, rep, src)
    assert n >= 1, f"mutation pattern not found: {desc}"
    tmpd = tempfile.mkdtemp(prefix="mc_oracle_mut_")
    try:
        csrc = os.path.join(tmpd, "m.c")
        so = os.path.join(tmpd, "m.so")
        with open(csrc, "w") as f:
            f.write(mutated)
        subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", csrc, "-o", so, "-lm"],
                       check=True)
        assert _run_pins_against(so) >= 1, f"no pin caught: {desc}"
    finally:
        shutil.rmtree(tmpd, ignore_errors=True)
