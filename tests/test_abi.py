"""The C-ABI library: it builds, loads, exports every entry point mc.h declares,
and rejects bad arguments before touching a device (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import memory_caching_linear_gb300 as mcl
from memory_caching_linear_gb300 import build as mcbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mc.h")

FAKE = 1 << 20  # an aligned, never-dereferenced address: every call below fails validation first


@pytest.fixture(scope="module")
def lib():
    mcbuild.build()
    return mcl.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mc_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(mcl.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", mcl.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_header_compiles_as_c():
    res = subprocess.run(["gcc", "-std=c99", "-fsyntax-only", "-x", "c", "-I", os.path.dirname(HEADER), "-"],
                         input='#include "mc.h"\nint main(void){return mc_forward==0;}\n', text=True,
                         capture_output=True)
    assert res.returncode == 0, res.stderr


def test_status_strings(lib):
    for code in range(-10, 1):
        s = mcl.mc_status_string(code)
        assert s and s != "unknown status", code
    assert mcl.mc_status_string(-100) == "unknown status"


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, u=FAKE, B=1, H=1, L=64, d=16, seg=16, mode=1, topk=0, y=FAKE,
             states=None)
    a.update(kw)
    return lib.mc_forward(a["q"], a["k"], a["v"], a["u"], a["B"], a["H"], a["L"], a["d"], a["seg"], a["mode"],
                          a["topk"], a["y"], a["states"], None)


def test_argument_errors_never_reach_the_device(lib):
    assert _fwd(lib, q=None) == mcl.MC_ERR_NULL
    assert _fwd(lib, y=None) == mcl.MC_ERR_NULL
    assert _fwd(lib, u=None, mode=mcl.MC_GRM) == mcl.MC_ERR_NULL
    for mode in (mcl.MC_RESIDUAL, mcl.MC_MEAN):  # no router input needed: the null check passes (and the
        assert _fwd(lib, u=None, mode=mode, q=FAKE + 8) == mcl.MC_ERR_ALIGN  # alignment check stops the call)
    assert _fwd(lib, mode=7) == mcl.MC_ERR_MODE
    assert _fwd(lib, mode=-1) == mcl.MC_ERR_MODE
    for bad in (dict(d=17), dict(d=256), dict(L=0), dict(B=0), dict(H=-1), dict(seg=0)):
        assert _fwd(lib, **bad) == mcl.MC_ERR_SHAPE, bad
    assert _fwd(lib, mode=mcl.MC_SSC, topk=-1) == mcl.MC_ERR_TOPK
    assert _fwd(lib, mode=mcl.MC_SSC, topk=65, L=4096, seg=16) == mcl.MC_ERR_TOPK
    assert _fwd(lib, q=FAKE + 8) == mcl.MC_ERR_ALIGN
    assert _fwd(lib, states=FAKE + 4) == mcl.MC_ERR_ALIGN
    st = lib.mc_ssc_select(FAKE, FAKE, 1, 1, 64, 16, 16, 0, FAKE, 1, None)
    assert st == mcl.MC_ERR_TOPK
    st = lib.mc_ssc_select(FAKE, FAKE, 1, 1, 64, 16, 16, 65, FAKE, 1, None)
    assert st == mcl.MC_ERR_TOPK
    st = lib.mc_forward_host(None, FAKE, FAKE, FAKE, 1, 1, 64, 16, 16, 1, 0, FAKE, None, 1, None)
    assert st == mcl.MC_ERR_NULL
    dec = lambda **kw: lib.mc_decode_step(*[kw.get(n, FAKE) for n in ("q", "k", "v", "u")], 1, 1, kw.get("d", 16), 16,
                                          kw.get("mode", 1), 0, kw.get("t", 0), FAKE, FAKE, FAKE, FAKE,
                                          kw.get("n_max", 4), FAKE, 1, None)
    assert dec(t=-1) == mcl.MC_ERR_SHAPE
    assert dec(t=64) == mcl.MC_ERR_SHAPE  # segment 4 needs a fifth cache slot
    assert dec(n_max=65) == mcl.MC_ERR_SHAPE
    assert dec(d=24) == mcl.MC_ERR_SHAPE
    assert dec(mode=9) == mcl.MC_ERR_MODE
    assert dec(q=None) == mcl.MC_ERR_NULL
    assert dec(u=None) == mcl.MC_ERR_NULL
    assert dec(u=None, mode=mcl.MC_MEAN, q=FAKE + 4) == mcl.MC_ERR_ALIGN  # past the null check, stopped after
    assert dec(q=FAKE + 4) == mcl.MC_ERR_ALIGN


def test_backward_argument_errors_never_reach_the_device(lib):
    def bwd(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, u=FAKE, dy=FAKE, B=1, H=1, L=64, d=16, seg=16, mode=mcl.MC_GRM, topk=0,
                 dq=FAKE, dk=FAKE, dv=FAKE, du=FAKE)
        a.update(kw)
        return lib.mc_backward(a["q"], a["k"], a["v"], a["u"], a["dy"], a["B"], a["H"], a["L"], a["d"], a["seg"],
                               a["mode"], a["topk"], a["dq"], a["dk"], a["dv"], a["du"], None)
    for name in ("q", "k", "v", "dy", "dq", "dk", "dv"):
        assert bwd(**{name: None}) == mcl.MC_ERR_NULL, name
    assert bwd(u=None) == mcl.MC_ERR_NULL and bwd(du=None) == mcl.MC_ERR_NULL  # the router's input and gradient
    for mode in (mcl.MC_RESIDUAL, mcl.MC_MEAN):  # no router: u and du may be absent (past the null check,
        assert bwd(u=None, du=None, mode=mode, dq=FAKE + 8) == mcl.MC_ERR_ALIGN  # stopped by the alignment one)
    assert bwd(mode=7) == mcl.MC_ERR_MODE
    for bad in (dict(d=17), dict(L=0), dict(seg=0), dict(B=0)):
        assert bwd(**bad) == mcl.MC_ERR_SHAPE, bad
    assert bwd(mode=mcl.MC_SSC, topk=-1) == mcl.MC_ERR_TOPK
    assert bwd(dq=FAKE + 8) == mcl.MC_ERR_ALIGN
    assert bwd(du=FAKE + 4) == mcl.MC_ERR_ALIGN


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device answer")
def test_valid_call_without_a_device_fails_cleanly(lib):
    st = _fwd(lib)
    assert st in (mcl.MC_ERR_CUDA, mcl.MC_ERR_DEVICE)


def test_binding_fails_loudly_without_cuda_tensors(lib):
    x = torch.zeros(1, 1, 8, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mcl.mc_forward(x, x, x, x, 4, mcl.MC_GRM)


def test_build_flags_target_sm103a():
    flags = " ".join(mcbuild.compile_flags())
    assert "arch=compute_103a,code=sm_103a" in flags


def test_log_segments_on_the_host(lib):
    """mc_log_segments needs no device: the pages' worked example (37 -> 32, 4, 1) and the
    oracle's own logarithmic segmentation for other lengths; errors for bad arguments."""
    import oracle
    assert mcl.log_segments(37) == [0, 32, 36, 37]
    for L in (1, 2, 3, 64, 1000, 65535, 1 << 20):
        assert mcl.log_segments(L) == oracle.log_segments(L)
    buf = (ctypes.c_int32 * 2)()
    assert lib.mc_log_segments(0, buf, 2) == mcl.MC_ERR_SHAPE
    assert lib.mc_log_segments(3, buf, 2) == mcl.MC_ERR_SHAPE  # needs three boundaries
    assert lib.mc_log_segments(3, None, 8) == mcl.MC_ERR_NULL
    off = (ctypes.c_int32 * 3)(0, 5, 4)  # not rising
    st = lib.mc_forward_segments(FAKE, FAKE, FAKE, FAKE, 1, 1, 4, 16, off, 2, 1, 0, FAKE, None, 1, None)
    assert st == mcl.MC_ERR_SHAPE
