"""The tensor-core building blocks, each against a plain matrix product, and the
bounded device wait (through the diagnostic entry points in include/mc_selftest.h)."""
import ctypes

import pytest
import torch

import memory_caching_linear_gb300 as mcl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from memory_caching_linear_gb300 import build
    build.build()
    lib = mcl.load_library()
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.mc_selftest_umma.argtypes = [vp, vp, vp, i, vp]
    lib.mc_selftest_umma.restype = i
    lib.mc_selftest_wait_timeout.argtypes = [i, vp]
    lib.mc_selftest_wait_timeout.restype = i
    return lib


def _expected(X, W, form):
    Xf, Wf = X.float(), W.float()
    return {0: Xf @ Wf.T, 1: Xf @ Wf.T, 2: Xf @ Wf, 3: Xf.T @ Wf, 4: Xf @ Wf[:64].T, 5: Xf @ Wf}[form]


@pytest.mark.parametrize("form", [0, 1, 2, 3, 4, 5])
def test_umma_forms(lib, form):
    g = torch.Generator(device="cpu").manual_seed(100 + form)
    X = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    W = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    D = torch.full((128, 128), float("nan"), device="cuda")
    st = lib.mc_selftest_umma(X.data_ptr(), W.data_ptr(), D.data_ptr(), form, torch.cuda.current_stream().cuda_stream)
    assert st == mcl.MC_OK, mcl.mc_status_string(st)
    ref = _expected(X, W, form)
    got = D[:, :64] if form == 4 else D
    err = (got - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, (form, err)


def test_bounded_wait_gives_up_and_reports(lib):
    st = lib.mc_selftest_wait_timeout(50, torch.cuda.current_stream().cuda_stream)
    assert st == mcl.MC_ERR_DEVICE_TIMEOUT
    # the context is still usable afterwards
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0
