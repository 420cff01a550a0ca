"""Parity of the forward over given segment boundaries (mc_forward_segments) with the
oracle, including the logarithmic segmentation of Log-Linear++ ([MC-sum §4.2]; the
variants appendix of "メモリキャッシング：メモリ容量が増大する RNN"): y and the cached
states element by element, every aggregation, fp32 and bf16.  Tolerances as the
forward: 1e-4 * max|ref| (fp32), 1e-2 * max|ref| (bf16)."""
import zlib

import numpy as np
import pytest
import torch

import memory_caching_linear_gb300 as mcl
import oracle
from mc_inputs import GRM, MEAN, RESIDUAL, SOUP, SSC, make_inputs
from ssc_valid import check_y_over_valid_sets

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from memory_caching_linear_gb300 import build
    build.build()
    mcl.load_library()


def rel_err(got, ref):
    scale = np.abs(ref).max()
    return float(np.abs(np.asarray(got, np.float64) - ref).max() / (scale if scale > 0 else 1.0))


CASES = [
    # (name, B, H, L, d, dtype, boundaries or None for the logarithmic segmentation)
    ("log-1000-f32", 1, 2, 1000, 32, "f32", None),
    ("log-777-bf16", 1, 1, 777, 128, "bf16", None),
    ("log-4095-d64", 1, 1, 4095, 64, "bf16", None),
    ("custom-f32", 2, 1, 300, 16, "f32", [0, 7, 8, 100, 260, 300]),
    ("one-seg", 1, 1, 256, 64, "f32", [0, 256]),
    # segments longer than the scan's 512-token pieces: ragged last pieces, a one-token segment between
    ("pieces-ragged-f32", 1, 2, 2600, 32, "f32", [0, 1300, 1301, 2600]),
    ("pieces-d128-bf16", 1, 1, 2048, 128, "bf16", [0, 1536, 2048]),
]


@pytest.mark.parametrize("mode,topk", [(GRM, 0), (RESIDUAL, 0), (SOUP, 0), (SSC, 2), (MEAN, 0)])
@pytest.mark.parametrize("name,B,H,L,d,dtype,off", CASES, ids=[c[0] for c in CASES])
def test_segments_parity(name, B, H, L, d, dtype, off, mode, topk):
    # the library's and the oracle's logarithmic segmentations are computed separately
    off_gpu = mcl.log_segments(L) if off is None else off
    off = oracle.log_segments(L) if off is None else off
    q, k, v, u = make_inputs(B, H, L, d, seed=zlib.crc32(name.encode()) % 1000, dtype=dtype)
    ref = oracle.forward(q, k, v, u, None, mode, topk, seg_off=off)
    dev = torch.device("cuda")
    y, st = mcl.mc_forward_segments(*(t.to(dev) for t in (q, k, v, u)), off_gpu, mode, topk)
    assert mcl.mc_check_device() == mcl.MC_OK
    y, st = y.float().cpu().numpy(), st.cpu().numpy()
    yref = ref["y"]
    if mode == SSC and 0 < topk < len(off) - 2:
        # fp32 near-ties may rank either way: each such token must match the oracle on
        # one of its valid top-k selections
        check_y_over_valid_sets(
            y, q, k, v, u, off, topk, ref,
            lambda sel: oracle.forward(q, k, v, u, None, SSC, topk, seg_off=off, given_sel=sel)["y"], TOL[dtype])
    else:
        assert rel_err(y, yref) <= TOL[dtype], (name, mode, rel_err(y, yref))
    assert rel_err(st, ref["states"]) <= TOL[dtype]


def test_constant_boundaries_match_mc_forward():
    q, k, v, u = (t.cuda() for t in make_inputs(1, 2, 640, 32, 3, "f32"))
    y0, s0 = mcl.forward(q, k, v, u, 128, GRM)
    y1, s1 = mcl.mc_forward_segments(q, k, v, u, list(range(0, 641, 128)), GRM)
    torch.testing.assert_close(y1, y0, rtol=0, atol=0)
    torch.testing.assert_close(s1, s0, rtol=0, atol=0)


# Given boundaries whose leading segments are whole 128-token chunks and whose other
# segments lie in the last L % 128 tokens run the tensor-core kernels for the former
# and the CUDA-core scan and readout for the tail.
TC_CASES = [
    # (name, B, H, L, d, boundaries or None for the logarithmic segmentation)
    ("tc-log-777", 1, 2, 777, 128, None),         # 512, 256 | 8, 1
    ("tc-log-4095-d64", 1, 1, 4095, 64, None),     # 2048 .. 128 | 64 .. 1
    ("tc-no-tail", 2, 1, 2048, 128, [0, 1536, 2048]),
    ("tc-mixed", 1, 2, 1380, 128, [0, 384, 1152, 1280, 1300, 1301, 1380]),  # 384, 768, 128 | 20, 1, 79
    # segments longer than the state walk's 16-chunk pieces: 32 chunks (two pieces), 48 chunks (three)
    ("tc-log-5000", 1, 1, 5000, 128, None),  # 4096, 512, 256, 128 | 8
    ("tc-pieces-d64", 1, 2, 6500, 64, [0, 6144, 6400, 6500]),  # 6144 (three pieces), 256 | 100
]


@pytest.mark.parametrize("mode,topk", [(GRM, 0), (RESIDUAL, 0), (SOUP, 0), (SSC, 2), (MEAN, 0)])
@pytest.mark.parametrize("name,B,H,L,d,off", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_segments_tensor_core_parity(name, B, H, L, d, off, mode, topk):
    off_gpu = mcl.log_segments(L) if off is None else off
    off = oracle.log_segments(L) if off is None else off
    q, k, v, u = make_inputs(B, H, L, d, seed=zlib.crc32(name.encode()) % 1000, dtype="bf16")
    ref = oracle.forward(q, k, v, u, None, mode, topk, seg_off=off)
    dev = torch.device("cuda")
    args = [t.to(dev) for t in (q, k, v, u)]
    with mcl.KernelProfile() as prof:
        y, st = mcl.mc_forward_segments(*args, off_gpu, mode, topk)
    torch.cuda.synchronize()
    assert mcl.mc_check_device() == mcl.MC_OK
    assert "seg_state_tc" in prof.stages and "readout_tc" in prof.stages, prof.stages
    tail = L % 128 != 0
    assert ("tail_readout_simt" in prof.stages) == tail, prof.stages
    y, st = y.float().cpu().numpy(), st.cpu().numpy()
    if mode == SSC and 0 < topk < len(off) - 2:
        check_y_over_valid_sets(
            y, q, k, v, u, off, topk, ref,
            lambda sel: oracle.forward(q, k, v, u, None, SSC, topk, seg_off=off, given_sel=sel)["y"], TOL["bf16"])
    else:
        assert rel_err(y, ref["y"]) <= TOL["bf16"], (name, mode, rel_err(y, ref["y"]))
    assert rel_err(st, ref["states"]) <= TOL["bf16"]


@pytest.mark.parametrize("mode,topk", [(GRM, 0), (RESIDUAL, 0), (SSC, 2)])
def test_constant_boundaries_match_mc_forward_tensor_cores(mode, topk):
    # the same segments through both tensor-core paths: the same arithmetic per tile
    q, k, v, u = (t.cuda() for t in make_inputs(1, 2, 2048, 128, 4, "bf16"))
    y0, s0 = mcl.forward(q, k, v, u, 256, mode, topk)
    y1, s1 = mcl.mc_forward_segments(q, k, v, u, list(range(0, 2049, 256)), mode, topk)
    torch.testing.assert_close(s1, s0, rtol=0, atol=0)
    torch.testing.assert_close(y1, y0, rtol=0, atol=0)


def test_piece_split_state_walk_matches_mc_forward():
    # 4096-token segments are two 16-chunk pieces for mc_forward_segments and one walk for mc_forward:
    # the same states up to the order of the fp32 sums
    q, k, v, u = (t.cuda() for t in make_inputs(1, 2, 8192, 128, 6, "bf16"))
    y0, s0 = mcl.forward(q, k, v, u, 4096, GRM)
    y1, s1 = mcl.mc_forward_segments(q, k, v, u, [0, 4096, 8192], GRM)
    torch.testing.assert_close(s1, s0, rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(y1.float(), y0.float(), rtol=2e-2, atol=2e-2)
