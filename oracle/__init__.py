"""fp64 CPU oracle for the Memory Caching forward over linear memory.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference leg may import this package.  The
product library never loads it, and it shares no code with the CUDA path: the
arithmetic lives in ``mc_oracle.c`` (plain C, double precision, one token at a
time), compiled here with gcc and called through ctypes.

Functions
---------
forward(q, k, v, u, seg_len, mode, topk=0, ...)
    State form, literal: cached segment states, online state after the token's
    update, key mean-pool gates, Residual / GRM / Soup / SSC / Mean aggregation.
bruteforce(q, k, v, u, seg_len, mode, topk=0)
    Token-level twin that never forms a memory matrix (tiny inputs only).
backward(q, k, v, u, dy, seg_len, mode, topk=0)
    Gradients dq, dk, dv, du of <y, dy> (plain linear memory), by the chain rule
    through the forward's steps.

Both take optional ``swla=(alpha, beta, lam)`` (arrays [B, H, L]): the sliding-
window linear attention update with c = 2, M_t = alpha_t M_{t-1} + beta_t v_{t-1}
k_{t-1}^T + lambda_t v_t k_t^T, under the same caching and aggregation.

Inputs are arrays of shape [B, H, L, d] in any real dtype; they are widened
exactly to float64 (bf16 and fp32 values are exactly representable).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

RESIDUAL, GRM, SOUP, SSC, MEAN = 0, 1, 2, 3, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mc_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile mc_oracle.c into oracle/_build/liboracle.so (IEEE semantics, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            u8 = ctypes.POINTER(ctypes.c_uint8)
            i = ctypes.c_int
            lib.mc_oracle_forward.argtypes = [dp, dp, dp, dp, i, i, i, i, i, i,
                                              u8, ip, dp, dp, ip, dp, i]
            lib.mc_oracle_forward.restype = i
            lib.mc_oracle_bruteforce.argtypes = [dp, dp, dp, dp, i, i, i, i, i, i, dp, i]
            lib.mc_oracle_bruteforce.restype = i
            lib.mc_oracle_forward_swla.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i,
                                                   u8, ip, dp, dp, ip, dp, i]
            lib.mc_oracle_forward_swla.restype = i
            lib.mc_oracle_bruteforce_swla.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, dp, i]
            lib.mc_oracle_bruteforce_swla.restype = i
            lib.mc_oracle_backward.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, ip, dp, dp, dp, dp, i]
            lib.mc_oracle_backward.restype = i
            lib.mc_oracle_forward_segments.argtypes = [dp, dp, dp, dp, i, i, i, ip, i, i, i, ip, dp, dp, ip, dp, i]
            lib.mc_oracle_forward_segments.restype = i
            lib.mc_oracle_bruteforce_segments.argtypes = [dp, dp, dp, dp, i, i, i, ip, i, i, i, dp, i]
            lib.mc_oracle_bruteforce_segments.restype = i
            _lib = lib
    return _lib


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: widen through float32 (exact for bf16)
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype)) if a is not None else None


def num_segments(L: int, seg_len: int) -> int:
    return (L + seg_len - 1) // seg_len


def _swla_args(swla, B, H, L):
    alpha, beta, lam = (_as_f64(a) for a in swla)
    for a in (alpha, beta, lam):
        if a.shape != (B, H, L):
            raise ValueError("alpha, beta, lam must be [B, H, L]")
    return alpha, beta, lam


def log_segments(L: int) -> list:
    """Logarithmic segmentation ([MC-sum §4.2]; the Log-Linear++ variant of [MC-ja]'s
    variants appendix): L written in binary, one segment per set bit with that power of
    two as its length, the longest first.  Returns the boundaries [0, ..., L]."""
    off = [0]
    for bit in reversed(range(L.bit_length())):
        if (L >> bit) & 1:
            off.append(off[-1] + (1 << bit))
    return off


def _seg_array(seg_off, L):
    a = np.ascontiguousarray(np.asarray(seg_off, dtype=np.int32))
    if a.ndim != 1 or len(a) < 2 or a[0] != 0 or a[-1] != L or np.any(np.diff(a) <= 0):
        raise ValueError("seg_off must rise strictly from 0 to L")
    return a


def forward(q, k, v, u, seg_len: int, mode: int, topk: int = 0, *,
            seg_mask=None, given_sel=None, nthreads: int = 0, swla=None, seg_off=None) -> dict:
    """Run the state-form oracle.

    Returns a dict with ``y`` [B,H,L,d] and ``states`` [B,H,N,d,d] (float64); for
    SSC also ``sel`` [B,H,L,topk] int32 (rank order, -1 padded) and ``gap``
    [B,H,L] (fp64 distance between the last selected and the best unselected
    score; inf where nothing was left out).  ``seg_mask`` (length N, bool)
    restricts which segments' outputs are computed; ``given_sel`` replaces the
    router's choice for SSC.  ``seg_off`` (boundaries [0, ..., L]) replaces the
    constant segment length ``seg_len`` by given segments.
    """
    lib = _load()
    q, k, v, u = (_as_f64(a) for a in (q, k, v, u))
    if u.size == 0 and mode in (RESIDUAL, MEAN):
        u = np.zeros_like(q)
    B, H, L, d = q.shape
    for a in (k, v, u):
        if a.shape != q.shape:
            raise ValueError("q, k, v, u must share the shape [B, H, L, d]")
    so = _seg_array(seg_off, L) if seg_off is not None else None
    N = len(so) - 1 if so is not None else num_segments(L, seg_len)
    y = np.zeros((B, H, L, d), np.float64)
    states = np.zeros((B, H, N, d, d), np.float64)
    sel = gap = None
    kk = max(topk, 0)
    if mode == SSC:
        sel = np.full((B, H, L, max(kk, 1)), -1, np.int32)
        gap = np.full((B, H, L), np.inf, np.float64)
    gs = None
    if given_sel is not None:
        gs = np.ascontiguousarray(np.asarray(given_sel, dtype=np.int32))
        if gs.shape != (B, H, L, kk):
            raise ValueError("given_sel must be [B,H,L,topk]")
    sm = None
    if seg_mask is not None:
        sm = np.ascontiguousarray(np.asarray(seg_mask, dtype=np.uint8))
        if sm.shape != (N,):
            raise ValueError("seg_mask must have one entry per segment")
    common = [_ptr(sm, ctypes.c_uint8), _ptr(gs, ctypes.c_int32),
              _ptr(y, ctypes.c_double), _ptr(states, ctypes.c_double),
              _ptr(sel, ctypes.c_int32) if sel is not None else None,
              _ptr(gap, ctypes.c_double) if gap is not None else None, nthreads]
    qkvu = [_ptr(a, ctypes.c_double) for a in (q, k, v, u)]
    if so is not None:
        if swla is not None or sm is not None:
            raise ValueError("seg_off does not combine with swla or seg_mask")
        st = lib.mc_oracle_forward_segments(*qkvu, B * H, L, d, _ptr(so, ctypes.c_int32), N, mode, kk,
                                            *common[1:])
    elif swla is None:
        st = lib.mc_oracle_forward(*qkvu, B * H, L, d, seg_len, mode, kk, *common)
    else:
        abl = _swla_args(swla, B, H, L)
        st = lib.mc_oracle_forward_swla(*qkvu, *[_ptr(a, ctypes.c_double) for a in abl],
                                        B * H, L, d, seg_len, mode, kk, *common)
    if st != 0:
        raise RuntimeError(f"mc_oracle_forward failed with status {st}")
    out = {"y": y, "states": states}
    if mode == SSC:
        out["sel"] = sel[..., :kk]
        out["gap"] = gap
    return out


def bruteforce(q, k, v, u, seg_len: int, mode: int, topk: int = 0, *, nthreads: int = 0,
               swla=None, seg_off=None) -> np.ndarray:
    """Token-level twin: y [B,H,L,d] without forming any memory matrix (O(L^2 d))."""
    lib = _load()
    q, k, v, u = (_as_f64(a) for a in (q, k, v, u))
    B, H, L, d = q.shape
    y = np.zeros((B, H, L, d), np.float64)
    qkvu = [_ptr(a, ctypes.c_double) for a in (q, k, v, u)]
    if seg_off is not None:
        so = _seg_array(seg_off, L)
        st = lib.mc_oracle_bruteforce_segments(*qkvu, B * H, L, d, _ptr(so, ctypes.c_int32), len(so) - 1, mode,
                                               max(topk, 0), _ptr(y, ctypes.c_double), nthreads)
    elif swla is None:
        st = lib.mc_oracle_bruteforce(*qkvu, B * H, L, d, seg_len, mode, max(topk, 0),
                                      _ptr(y, ctypes.c_double), nthreads)
    else:
        abl = _swla_args(swla, B, H, L)
        st = lib.mc_oracle_bruteforce_swla(*qkvu, *[_ptr(a, ctypes.c_double) for a in abl],
                                           B * H, L, d, seg_len, mode, max(topk, 0),
                                           _ptr(y, ctypes.c_double), nthreads)
    if st != 0:
        raise RuntimeError(f"mc_oracle_bruteforce failed with status {st}")
    return y


def backward(q, k, v, u, dy, seg_len: int, mode: int, topk: int = 0, *, given_sel=None,
             nthreads: int = 0) -> dict:
    """Gradients of the forward for the upstream gradient ``dy`` of y (plain linear
    memory): a dict with ``dq``, ``dk``, ``dv``, ``du`` [B,H,L,d] float64 (``du`` is
    zero for Residual and Mean, which read no u).  ``given_sel`` [B,H,L,topk] replaces
    the SSC router's choice, as in :func:`forward`."""
    lib = _load()
    q, k, v, u, dy = (_as_f64(a) for a in (q, k, v, u, dy))
    if u.size == 0 and mode in (RESIDUAL, MEAN):
        u = np.zeros_like(q)
    B, H, L, d = q.shape
    for a in (k, v, u, dy):
        if a.shape != q.shape:
            raise ValueError("q, k, v, u, dy must share the shape [B, H, L, d]")
    out = {n: np.zeros((B, H, L, d), np.float64) for n in ("dq", "dk", "dv", "du")}
    gs = None
    if given_sel is not None:
        gs = np.ascontiguousarray(np.asarray(given_sel, dtype=np.int32))
        if gs.shape != (B, H, L, max(topk, 0)):
            raise ValueError("given_sel must be [B,H,L,topk]")
    st = lib.mc_oracle_backward(*[_ptr(a, ctypes.c_double) for a in (q, k, v, u, dy)], B * H, L, d, seg_len,
                                mode, max(topk, 0), _ptr(gs, ctypes.c_int32),
                                *[_ptr(out[n], ctypes.c_double) for n in ("dq", "dk", "dv", "du")], nthreads)
    if st != 0:
        raise RuntimeError(f"mc_oracle_backward failed with status {st}")
    return out
