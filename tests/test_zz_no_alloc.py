"""mc_forward_noalloc, the forward for callers that cannot allocate device
memory while they run (engine plugins whose framework owns all device memory,
serving loops that must not hit the allocator mid-request).

Called through the C ABI and compared, on two calls in a row, with mc_forward
on the same inputs at the bf16 tolerance of the parity tests.  This file runs
last (its name sorts last) so a failure here leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import memory_caching_linear_gb300 as mcl
from mc_inputs import GRM, SSC, make_inputs

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2


@pytest.fixture(scope="module")
def lib():
    from memory_caching_linear_gb300 import build
    build.build()
    return mcl.load_library()


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def _noalloc(lib, q, k, v, u, C, mode, topk, y, states):
    B, H, L, d = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.mc_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), u.data_ptr(), B, H, L, d, C, mode,
                                  topk, y.data_ptr(), states.data_ptr() if states is not None else None, stream)


def test_noalloc_matches_mc_forward_on_two_calls(lib):
    dev = torch.device("cuda")
    # call 1: GRM, states written to a caller buffer
    q1, k1, v1, u1 = (t.to(dev) for t in make_inputs(1, 2, 1024, 128, 21, "bf16"))
    # call 2: other inputs, SSC, states kept inside the static scratch (states = NULL)
    q2, k2, v2, u2 = (t.to(dev) for t in make_inputs(2, 2, 768, 64, 22, "bf16"))
    y1 = torch.empty_like(q1)
    st1 = torch.empty(1, 2, 4, 128, 128, device=dev)
    y2 = torch.empty_like(q2)
    ref1, rst1 = mcl.mc_forward(q1, k1, v1, u1, 256, GRM)
    ref2, _ = mcl.mc_forward(q2, k2, v2, u2, 64, SSC, 3)
    torch.cuda.synchronize()

    assert _noalloc(lib, q1, k1, v1, u1, 256, GRM, 0, y1, st1) == mcl.MC_OK
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    assert _noalloc(lib, q2, k2, v2, u2, 64, SSC, 3, y2, None) == mcl.MC_OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()

    assert _rel(y1, ref1) <= TOL_BF16
    assert _rel(st1, rst1) <= TOL_BF16
    assert _rel(y2, ref2) <= TOL_BF16
    assert free_after == free_before  # the second call took no device memory


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    dev = torch.device("cuda")
    x = torch.zeros(16, dtype=torch.bfloat16, device=dev)  # never read: the size check comes first
    p = x.data_ptr()
    # O_on alone: 8 * 16 * 4096 * 128 * 4 bytes = 256 MiB > 64 MiB
    st = lib.mc_forward_noalloc(p, p, p, p, 8, 16, 4096, 128, 256, GRM, 0, p, None,
                                torch.cuda.current_stream().cuda_stream)
    assert st == mcl.MC_ERR_SCRATCH
    assert "64 MiB" in mcl.mc_status_string(st)
