"""Parity of the backward pass (mc_backward / mc_backward_f32, through the C ABI)
with the oracle's backward: the gradients dq, dk, dv, du of <y, dy>, element by
element, at sizes that span several tiles and a ragged tail.

Tolerance per gradient tensor: max|g - g_ref| <= 1e-4 * max|g_ref| for fp32
inputs, <= 1e-2 * max|g_ref| for bf16 inputs and outputs (fp32 accumulation) --
the forward's bounds.  SSC: the selection passes no gradient, so where the GPU's
router and the oracle's part on an fp32 near-tie (gap < 1e-5), the GPU's set must be
a valid top-k and the oracle's backward is evaluated on that set.
"""
import zlib

import numpy as np
import pytest
import torch

import memory_caching_linear_gb300 as mcl
import oracle
from mc_inputs import GRM, LONG_GRM, MEAN, RESIDUAL, SOUP, SSC, make_inputs, workload_inputs
from ssc_valid import GAP, cached_scores, is_valid, seg_starts

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}
NAMES = ("dq", "dk", "dv", "du")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from memory_caching_linear_gb300 import build
    build.build()
    mcl.load_library()


def rel_err(got, ref):
    scale = np.abs(ref).max()
    return float(np.abs(np.asarray(got, np.float64) - ref).max() / (scale if scale > 0 else 1.0))


def _case(name, B, H, L, d, dtype):
    seed = zlib.crc32(name.encode()) % 1000
    q, k, v, u = make_inputs(B, H, L, d, seed=seed, dtype=dtype)
    g = torch.Generator().manual_seed(seed + 7)
    dy = torch.randn(B, H, L, d, generator=g).to(q.dtype)
    return q, k, v, u, dy


def run_backward(q, k, v, u, dy, C, mode, topk=0):
    dev = torch.device("cuda")
    out = mcl.mc_backward(*(t.to(dev) if t is not None else None for t in (q, k, v, u, dy)), C, mode, topk)
    assert mcl.mc_check_device() == mcl.MC_OK
    return {n: (t.float().cpu().numpy() if t is not None else None) for n, t in zip(NAMES, out)}


CASES = [
    # (name, B, H, L, d, C, dtype)
    ("b-tiny", 1, 1, 256, 16, 64, "f32"),
    ("b-N1", 1, 1, 200, 16, 256, "f32"),
    ("b-ragged", 1, 2, 200, 32, 64, "f32"),
    ("b-C1", 1, 1, 40, 16, 1, "f32"),
    ("b-C37", 2, 1, 150, 64, 37, "f32"),
    ("b-d128", 1, 1, 300, 128, 128, "f32"),
    ("b-d64-bf16", 1, 2, 512, 64, 128, "bf16"),
    ("b-d128-bf16", 1, 1, 777, 128, 256, "bf16"),
    # shapes of the tensor-core path (G on tcgen05): d = 64 / 128, seg_len % 128 == 0, L % seg_len == 0
    ("b-tc-d128", 1, 2, 1024, 128, 256, "bf16"),
    ("b-tc-d128-N8", 2, 1, 1024, 128, 128, "bf16"),
]


def gpu_selection(q, k, v, u, C, topk):
    """The GPU router's selection (mc_ssc_select runs the same router as the backward's
    gates), checked against the oracle's: equal except on fp32 near-ties, where it must be
    a valid top-k.  Returns it, or None when it equals the oracle's everywhere."""
    dev = torch.device("cuda")
    fwd = oracle.forward(q, k, v, u, C, SSC, topk)
    sel = mcl.mc_ssc_select(k.to(dev), u.to(dev), C, topk).cpu().numpy()
    differ = np.any(np.sort(sel, -1) != np.sort(fwd["sel"], -1), axis=-1)
    if not differ.any():
        return None
    assert np.all(fwd["gap"][differ] < GAP), "selections differ outside near-ties"
    r = cached_scores(k, u, seg_starts(q.shape[2], C))
    for b, h, t in zip(*np.nonzero(differ)):
        assert is_valid(r[b, h, t, :t // C], sel[b, h, t], topk), (b, h, t)
    print(f"near-tie tokens where the GPU chose another valid set: {int(differ.sum())}")
    return sel


def check_backward(q, k, v, u, dy, C, mode, topk, dtype, label):
    given = None
    if mode == SSC and 0 < topk < (q.shape[2] + C - 1) // C - 1:
        given = gpu_selection(q, k, v, u, C, topk)
    ref = oracle.backward(q, k, v, u, dy, C, mode, topk, given_sel=given)
    got = run_backward(q, k, v, u, dy, C, mode, topk)
    for n in NAMES:
        if got[n] is None:
            assert mode in (RESIDUAL, MEAN)
            continue
        err = rel_err(got[n], ref[n])
        assert err <= TOL[dtype], (label, mode, topk, n, err)
        assert np.isfinite(got[n]).all()


@pytest.mark.parametrize("mode,topk", [(RESIDUAL, 0), (GRM, 0), (SOUP, 0), (SSC, 0), (SSC, 2), (SSC, 100),
                                       (MEAN, 0)])
@pytest.mark.parametrize("name,B,H,L,d,C,dtype", CASES, ids=[c[0] for c in CASES])
def test_backward_parity(name, B, H, L, d, C, dtype, mode, topk):
    q, k, v, u, dy = _case(name, B, H, L, d, dtype)
    check_backward(q, k, v, u, dy, C, mode, topk, dtype, name)


@pytest.mark.slow
@pytest.mark.parametrize("mode,topk", [(GRM, 0), (RESIDUAL, 0), (SSC, 4), (MEAN, 0)])
def test_backward_parity_tensor_core_n64(mode, topk):
    """Element by element at 64 segments, the bench's segment count: every cached-state
    kernel of the tensor-core backward (the cached pass, G, dk / dv) reads 63 cached
    states for the last segment's tokens.  One head keeps the oracle to seconds."""
    q, k, v, u, dy = _case("b-tc-N64", 1, 1, 8192, 128, "bf16")
    check_backward(q, k, v, u, dy, 128, mode, topk, "bf16", "b-tc-N64")


def test_backward_without_u_for_unrouted_modes():
    q, k, v, u, dy = _case("b-nou", 1, 2, 300, 32, "f32")
    for mode in (RESIDUAL, MEAN):
        ref = oracle.backward(q, k, v, u, dy, 64, mode)
        got = run_backward(q, k, v, None, dy, 64, mode)
        assert got["du"] is None
        for n in ("dq", "dk", "dv"):
            assert rel_err(got[n], ref[n]) <= TOL["f32"], (mode, n)


def test_autograd_wrapper_matches_the_entry_point():
    dev = torch.device("cuda")
    q, k, v, u, dy = (t.to(dev) for t in _case("b-autograd", 1, 2, 256, 64, "f32"))
    leaves = [t.clone().requires_grad_(True) for t in (q, k, v, u)]
    y = mcl.MemoryCaching.apply(*leaves, 64, GRM, 0)
    grads = torch.autograd.grad(y, leaves, dy)
    direct = mcl.mc_backward(q, k, v, u, dy, 64, GRM)
    for a, b in zip(grads, direct):
        torch.testing.assert_close(a, b, rtol=0, atol=0)


# ------------------------------------------------------------------ full size: homogeneity identities
# y_t = sum_i g_{t,i} M_i q_t, where the gates depend on neither q nor v and every memory M_i is
# linear in v ("メモリキャッシング：メモリ容量が増大する RNN", §3 eq. 4b-5 and §3.1 eq. 7-10), so y is
# homogeneous of degree one in q and in v, and Euler's theorem gives <dq, q> = <dv, v> = <dy, y>
# for every (b, h) problem; with constant gates (Residual, Mean) also <dk, k> = <dy, y>.  These hold
# at any size: they check the whole tensor-core gradient path at the long workload's full size,
# where the oracle cannot run.  Tolerance: 1e-2 of the sum of the terms' magnitudes (bf16 outputs).

def _identities(w, mode, topk=0):
    dev = torch.device("cuda")
    q, k, v, u = (t.to(dev) for t in workload_inputs(w))
    g = torch.Generator().manual_seed(w.seed + 7)
    dy = torch.randn(w.B, w.H, w.L, w.d, generator=g).to(q.dtype).to(dev)
    y, _ = mcl.mc_forward(q, k, v, u, w.seg_len, mode, topk, want_states=False)
    dq, dk, dv, du = mcl.mc_backward(q, k, v, u, dy, w.seg_len, mode, topk)
    assert mcl.mc_check_device() == mcl.MC_OK

    def dot(a, b):  # per (b, h): the sum of a * b and the sum of |a * b|, in fp64
        p = a.double() * b.double()
        return p.sum(dim=(2, 3)), p.abs().sum(dim=(2, 3))

    ref, ref_abs = dot(dy, y)
    pairs = [("dq", dq, q), ("dv", dv, v)] + ([("dk", dk, k)] if mode in (RESIDUAL, MEAN) else [])
    for name, grad, x in pairs:
        assert torch.isfinite(grad).all(), name
        got, got_abs = dot(grad, x)
        err = ((got - ref).abs() / (0.5 * (got_abs + ref_abs))).max().item()
        assert err <= 1e-2, (w.name, mode, name, err)


@pytest.mark.slow
@pytest.mark.parametrize("mode", [GRM, RESIDUAL, MEAN])
def test_full_size_backward_identities(mode):
    _identities(LONG_GRM, mode)
