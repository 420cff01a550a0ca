"""Validity of an SSC selection near fp32 ties, for the GPU parity tests.

The router keeps, for every token, the topk cached segments with the largest scores
r_{t,i} = <u_t, mean of segment i's keys> ([MC-sum §3.4], "给 RNN 装上“会增长的记忆”：
解读 Google 的 Memory Caching"), ranked in fp32.  Where two scores lie closer than the
precision the method is specified to (GAP = 1e-5 in fp32), more than one set is a
correct top-k.  A set is accepted when it has the right size and no score left out
exceeds a chosen one by more than GAP; y is then compared with the oracle evaluated on
that set (the oracle's ``given_sel``).

This module only checks results: the scores are recomputed here in fp64 from the
inputs to judge a set, never to produce an expected output.
"""
from __future__ import annotations

import itertools

import numpy as np

GAP = 1e-5


def _f64(x):
    if hasattr(x, "detach"):  # a torch tensor (bf16 widens exactly through fp32)
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, np.float64)


def cached_scores(k, u, seg_off):
    """fp64 scores r[b, h, t, i] = <u_t, mean of segment i's keys> for every segment i
    (the caller restricts them to the segments before the token's own)."""
    kf = _f64(k)
    uf = _f64(u)
    kbar = np.stack([kf[:, :, a:b].mean(2) for a, b in zip(seg_off[:-1], seg_off[1:])], 2)
    return np.einsum("bhtd,bhnd->bhtn", uf, kbar)


def is_valid(r, chosen, topk):
    """Is `chosen` (segment indices, -1 ignored) a top-`topk` of the scores r within GAP?"""
    chosen = [int(i) for i in chosen if i >= 0]
    n = len(r)
    if len(chosen) != min(topk, n) or len(set(chosen)) != len(chosen) or any(i >= n for i in chosen):
        return False
    rest = [i for i in range(n) if i not in set(chosen)]
    if not chosen or not rest:
        return True
    return max(r[rest]) <= min(r[chosen]) + GAP


def alternatives(r, topk, limit=64):
    """Every valid top-k set of the scores r (sorted index lists), at most `limit`."""
    n = len(r)
    want = min(topk, n)
    if want == 0:
        return [[]]
    kth = np.sort(r)[::-1][want - 1]
    cand = [i for i in range(n) if r[i] >= kth - GAP]
    out = []
    for c in itertools.combinations(cand, want):
        if is_valid(r, list(c), topk):
            out.append(sorted(c))
            if len(out) >= limit:
                break
    return out


def seg_starts(L, C):
    """Boundaries [0, C, 2C, ..., L] of the constant segmentation."""
    return list(range(0, L, C)) + [L]


def check_y_over_valid_sets(y, q, k, v, u, seg_off, topk, ref, run_oracle, tol):
    """y from a path whose selection is not observable (decode, given boundaries):
    tokens whose oracle gap is >= GAP must match the oracle as is; every near-tie token
    must match the oracle evaluated on one of its valid top-k sets.  `run_oracle(sel)`
    returns the oracle's y for a given selection [B, H, L, topk].  Returns the number
    of near-tie tokens checked this way."""
    yref = ref["y"]
    scale = np.abs(yref).max()
    err = np.abs(np.asarray(y, np.float64) - yref).max(-1) / scale
    gap = ref["gap"]
    tie = gap < GAP
    assert np.all(err[~tie] <= tol), float(err[~tie].max())
    if not tie.any():
        return 0
    r = cached_scores(k, u, seg_off)
    seg_of = np.searchsorted(np.asarray(seg_off), np.arange(yref.shape[2]), side="right") - 1
    alts = {}
    for b, h, t in zip(*np.nonzero(tie)):
        s = int(seg_of[t])
        alts[(b, h, t)] = alternatives(r[b, h, t, :s], topk)
        assert alts[(b, h, t)], (b, h, t)
    depth = max(len(a) for a in alts.values())
    ok = {key: False for key in alts}
    for j in range(depth):
        sel = np.array(ref["sel"], copy=True)
        for (b, h, t), a in alts.items():
            pick = a[min(j, len(a) - 1)]
            sel[b, h, t] = -1
            sel[b, h, t, :len(pick)] = pick
        yj = run_oracle(sel)
        for (b, h, t) in alts:
            e = np.abs(np.asarray(y[b, h, t], np.float64) - yj[b, h, t]).max() / scale
            ok[(b, h, t)] |= bool(e <= tol)
    bad = [key for key, good in ok.items() if not good]
    assert not bad, f"near-tie tokens matching no valid selection: {bad[:5]}"
    return len(alts)
