"""Memory Caching (MC) forward over a linear matrix-valued memory, for one GB300.

Thin ctypes binding over the C ABI in ``include/mc.h`` (``libmc.so``, built
in-tree by :mod:`memory_caching_linear_gb300.build`).  The functions below only
check and marshal arguments; every step of the forward runs in the library's
CUDA kernels.  There is no CPU fallback: if the library is not built, or the
device is not an sm_103a GPU, calls raise.

    y, states = mc_forward(q, k, v, u, seg_len, MC_GRM)

q, k, v, u are CUDA tensors [B, H, L, d] (bf16 -> ``mc_forward``; fp32 ->
``mc_forward_f32``).  Aggregations: MC_RESIDUAL, MC_GRM, MC_SOUP, MC_SSC, MC_MEAN.
"""
from __future__ import annotations

import ctypes
import os

import torch

MC_RESIDUAL, MC_GRM, MC_SOUP, MC_SSC, MC_MEAN = 0, 1, 2, 3, 4
MC_OK = 0
MC_ERR_NULL, MC_ERR_SHAPE, MC_ERR_MODE, MC_ERR_TOPK = -1, -2, -3, -4
MC_ERR_ALLOC, MC_ERR_CUDA, MC_ERR_DEVICE_TIMEOUT, MC_ERR_ALIGN, MC_ERR_DEVICE = -5, -6, -7, -8, -9
MC_ERR_SCRATCH = -10

EXPORTED = ("mc_forward", "mc_forward_f32", "mc_forward_swla", "mc_forward_segments", "mc_log_segments", "mc_backward", "mc_backward_f32", "mc_decode_step", "mc_ssc_select", "mc_forward_host", "mc_forward_noalloc",
            "mc_check_device", "mc_trim_scratch", "mc_set_readout_form", "mc_profile_begin", "mc_profile_end",
            "mc_profile_stage", "mc_status_string")
MC_READOUT_AUTO, MC_READOUT_FACTORISED = 0, 1

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmc.so")
_lib = None


class MCError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {mc_status_string(status)} (status {status})")
        self.status = status


def load_library():
    """Load libmc.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m memory_caching_linear_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.mc_forward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp]
    lib.mc_forward.restype = i
    lib.mc_forward_f32.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp]
    lib.mc_forward_f32.restype = i
    lib.mc_forward_swla.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp]
    lib.mc_forward_swla.restype = i
    lib.mc_forward_segments.argtypes = [vp, vp, vp, vp, i, i, i, i, vp, i, i, i, vp, vp, i, vp]
    lib.mc_forward_segments.restype = i
    lib.mc_log_segments.argtypes = [i, vp, i]
    lib.mc_log_segments.restype = i
    lib.mc_backward.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp, vp, vp]
    lib.mc_backward.restype = i
    lib.mc_backward_f32.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp, vp, vp]
    lib.mc_backward_f32.restype = i
    lib.mc_decode_step.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp, vp, i, vp, i, vp]
    lib.mc_decode_step.restype = i
    lib.mc_ssc_select.argtypes = [vp, vp, i, i, i, i, i, i, vp, i, vp]
    lib.mc_ssc_select.restype = i
    lib.mc_forward_host.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, i, vp]
    lib.mc_forward_host.restype = i
    lib.mc_forward_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp]
    lib.mc_forward_noalloc.restype = i
    lib.mc_trim_scratch.argtypes = []
    lib.mc_trim_scratch.restype = i
    lib.mc_set_readout_form.argtypes = [i]
    lib.mc_set_readout_form.restype = i
    lib.mc_check_device.argtypes = [vp]
    lib.mc_check_device.restype = i
    lib.mc_profile_begin.argtypes = [vp, i]
    lib.mc_profile_begin.restype = i
    lib.mc_profile_end.argtypes = []
    lib.mc_profile_end.restype = i
    lib.mc_profile_stage.argtypes = [i]
    lib.mc_profile_stage.restype = ctypes.c_char_p
    lib.mc_status_string.argtypes = [i]
    lib.mc_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def mc_status_string(status: int) -> str:
    return load_library().mc_status_string(int(status)).decode()


def num_segments(L: int, seg_len: int) -> int:
    return (L + seg_len - 1) // seg_len


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(t, name, dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}")


def _forward(fn_name, q, k, v, u, seg_len, agg_mode, topk, y, states, want_states, stream, swla=None):
    lib = load_library()
    dtype = q.dtype
    if q.dim() != 4:
        raise ValueError("q must be [B, H, L, d]")
    B, H, L, d = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors (use mc_forward_host for host buffers)")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, dtype, (B, H, L, d), dev)
    if u is not None:
        _check(u, "u", dtype, (B, H, L, d), dev)
    N = num_segments(L, seg_len)
    if y is None:
        y = torch.empty((B, H, L, d), dtype=dtype, device=dev)
    _check(y, "y", dtype, (B, H, L, d), dev)
    if states is None and want_states:
        states = torch.empty((B, H, N, d, d), dtype=torch.float32, device=dev)
    if states is not None:
        _check(states, "states", torch.float32, (B, H, N, d, d), dev)
    head = [q.data_ptr(), k.data_ptr(), v.data_ptr(), u.data_ptr() if u is not None else None]
    if swla is not None:
        for t, n in zip(swla, ("alpha", "beta", "lam")):
            _check(t, n, torch.float32, (B, H, L), dev)
        head += [t.data_ptr() for t in swla]
    st = getattr(lib, fn_name)(*head, B, H, L, d, int(seg_len), int(agg_mode), int(topk), y.data_ptr(),
                               states.data_ptr() if states is not None else None, _stream_handle(stream, dev))
    if st != MC_OK:
        raise MCError(st, fn_name)
    return y, states


def mc_forward(q, k, v, u, seg_len: int, agg_mode: int, topk: int = 0, *, y=None, states=None,
               want_states: bool = True, stream=None):
    """bf16 MC forward (``mc_forward`` in mc.h).  Returns (y, states); states is None
    when ``want_states`` is False and none was given."""
    return _forward("mc_forward", q, k, v, u, seg_len, agg_mode, topk, y, states, want_states, stream)


def mc_forward_swla(q, k, v, u, alpha, beta, lam, seg_len: int, agg_mode: int, topk: int = 0, *, y=None,
                    states=None, want_states: bool = True, stream=None):
    """bf16 MC forward over sliding-window linear attention, c = 2 (``mc_forward_swla`` in
    mc.h); alpha, beta, lam are fp32 [B, H, L] on the device.  Returns (y, states)."""
    return _forward("mc_forward_swla", q, k, v, u, seg_len, agg_mode, topk, y, states, want_states, stream,
                    swla=(alpha, beta, lam))


class DecodeCache:
    """Device caches for recurrent decoding with ``mc_decode_step``: cached segment
    states [B,H,n_max,d,d] and key means [B,H,n_max,d], the online memory
    [B,H,d,d] and key sum [B,H,d] (fp32), plus the next position ``t``."""

    def __init__(self, B: int, H: int, d: int, seg_len: int, n_max: int, device="cuda"):
        self.seg_len, self.n_max, self.t = int(seg_len), int(n_max), 0
        f32 = dict(dtype=torch.float32, device=device)
        self.states = torch.zeros((B, H, n_max, d, d), **f32)
        self.kbar = torch.zeros((B, H, n_max, d), **f32)
        self.online = torch.zeros((B, H, d, d), **f32)
        self.ksum = torch.zeros((B, H, d), **f32)


def mc_decode_step(cache: DecodeCache, q, k, v, u, agg_mode: int, topk: int = 0, *, y=None, stream=None):
    """One decoding step (``mc_decode_step`` in mc.h) for tokens q, k, v, u of shape
    [B, H, d] at position ``cache.t``; advances ``cache.t`` and returns y [B, H, d]."""
    lib = load_library()
    if q.dim() != 3:
        raise ValueError("q must be [B, H, d]")
    B, H, d = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    for t_, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t_, n, q.dtype, (B, H, d), dev)
    if u is not None:
        _check(u, "u", q.dtype, (B, H, d), dev)
    if y is None:
        y = torch.empty((B, H, d), dtype=q.dtype, device=dev)
    _check(y, "y", q.dtype, (B, H, d), dev)
    for t_, n, shp in ((cache.states, "states", (B, H, cache.n_max, d, d)), (cache.kbar, "kbar", (B, H, cache.n_max, d)),
                       (cache.online, "online", (B, H, d, d)), (cache.ksum, "ksum", (B, H, d))):
        _check(t_, n, torch.float32, shp, dev)
    st = lib.mc_decode_step(q.data_ptr(), k.data_ptr(), v.data_ptr(), u.data_ptr() if u is not None else None,
                            B, H, d, cache.seg_len, int(agg_mode), int(topk), cache.t,
                            cache.states.data_ptr(), cache.kbar.data_ptr(), cache.online.data_ptr(),
                            cache.ksum.data_ptr(), cache.n_max, y.data_ptr(), int(q.dtype == torch.bfloat16),
                            _stream_handle(stream, dev))
    if st != MC_OK:
        raise MCError(st, "mc_decode_step")
    cache.t += 1
    return y


def mc_forward_f32(q, k, v, u, seg_len: int, agg_mode: int, topk: int = 0, *, y=None, states=None,
                   want_states: bool = True, stream=None):
    """fp32 MC forward (``mc_forward_f32`` in mc.h)."""
    return _forward("mc_forward_f32", q, k, v, u, seg_len, agg_mode, topk, y, states, want_states, stream)


def forward(q, k, v, u, seg_len: int, agg_mode: int, topk: int = 0, **kw):
    """Dispatch on the input dtype: bf16 -> mc_forward, fp32 -> mc_forward_f32."""
    if q.dtype == torch.bfloat16:
        return mc_forward(q, k, v, u, seg_len, agg_mode, topk, **kw)
    if q.dtype == torch.float32:
        return mc_forward_f32(q, k, v, u, seg_len, agg_mode, topk, **kw)
    raise TypeError("inputs must be bf16 or fp32")


def log_segments(L: int) -> list:
    """The logarithmic segmentation of length L (``mc_log_segments``): boundaries [0, ..., L]."""
    buf = (ctypes.c_int32 * 33)()
    n = load_library().mc_log_segments(int(L), buf, 33)
    if n < 0:
        raise MCError(n, "mc_log_segments")
    return list(buf[:n + 1])


def mc_forward_segments(q, k, v, u, seg_off, agg_mode: int, topk: int = 0, *, y=None, states=None,
                        want_states: bool = True, stream=None):
    """Forward over given segment boundaries (``mc_forward_segments``); bf16 or fp32 inputs.
    ``seg_off`` is a sequence [0, ..., L]; with :func:`log_segments` and MC_GRM this is
    the Log-Linear++ variant.  Returns (y, states)."""
    lib = load_library()
    if q.dim() != 4:
        raise ValueError("q must be [B, H, L, d]")
    B, H, L, d = q.shape
    dev, dtype = q.device, q.dtype
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("inputs must be bf16 or fp32")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, dtype, (B, H, L, d), dev)
    if u is not None:
        _check(u, "u", dtype, (B, H, L, d), dev)
    off = (ctypes.c_int32 * len(seg_off))(*[int(x) for x in seg_off])
    nseg = len(seg_off) - 1
    if y is None:
        y = torch.empty((B, H, L, d), dtype=dtype, device=dev)
    _check(y, "y", dtype, (B, H, L, d), dev)
    if states is None and want_states:
        states = torch.empty((B, H, nseg, d, d), dtype=torch.float32, device=dev)
    if states is not None:
        _check(states, "states", torch.float32, (B, H, nseg, d, d), dev)
    st = lib.mc_forward_segments(q.data_ptr(), k.data_ptr(), v.data_ptr(), u.data_ptr() if u is not None else None,
                                 B, H, L, d, off, nseg, int(agg_mode), int(topk), y.data_ptr(),
                                 states.data_ptr() if states is not None else None,
                                 1 if dtype == torch.bfloat16 else 0, _stream_handle(stream, dev))
    if st != MC_OK:
        raise MCError(st, "mc_forward_segments")
    return y, states


def mc_backward(q, k, v, u, dy, seg_len: int, agg_mode: int, topk: int = 0, *, dq=None, dk=None, dv=None,
                du=None, stream=None):
    """Gradients (dq, dk, dv, du) of <y, dy> for the forward on the same inputs
    (``mc_backward`` / ``mc_backward_f32`` in mc.h, chosen by the dtype).  du is None
    for Residual and Mean unless a buffer is given (then it is zeroed)."""
    lib = load_library()
    if q.dim() != 4:
        raise ValueError("q must be [B, H, L, d]")
    B, H, L, d = q.shape
    dev, dtype = q.device, q.dtype
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("inputs must be bf16 or fp32")
    shape = (B, H, L, d)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dy, "dy")):
        _check(t, n, dtype, shape, dev)
    if u is not None:
        _check(u, "u", dtype, shape, dev)
    uses_u = agg_mode in (MC_GRM, MC_SOUP, MC_SSC)
    out = []
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        t = torch.empty(shape, dtype=dtype, device=dev) if t is None else t
        _check(t, n, dtype, shape, dev)
        out.append(t)
    if du is None and uses_u:
        du = torch.empty(shape, dtype=dtype, device=dev)
    if du is not None:
        _check(du, "du", dtype, shape, dev)
    fn = lib.mc_backward if dtype == torch.bfloat16 else lib.mc_backward_f32
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), u.data_ptr() if u is not None else None, dy.data_ptr(),
            B, H, L, d, int(seg_len), int(agg_mode), int(topk), *[t.data_ptr() for t in out],
            du.data_ptr() if du is not None else None, _stream_handle(stream, dev))
    if st != MC_OK:
        raise MCError(st, "mc_backward")
    return (*out, du)


class MemoryCaching(torch.autograd.Function):
    """Autograd wrapper: y = MemoryCaching.apply(q, k, v, u, seg_len, agg_mode, topk)
    runs the library's forward and, on backward, ``mc_backward`` (u may be None for
    Residual and Mean)."""

    @staticmethod
    def forward(ctx, q, k, v, u, seg_len: int, agg_mode: int, topk: int = 0):
        y, _ = forward(q, k, v, u, seg_len, agg_mode, topk, want_states=False)
        ctx.save_for_backward(q, k, v, u if u is not None else torch.empty(0, device=q.device))
        ctx.cfg = (seg_len, agg_mode, topk, u is not None)
        return y

    @staticmethod
    def backward(ctx, dy):
        q, k, v, u = ctx.saved_tensors
        seg_len, agg_mode, topk, has_u = ctx.cfg
        dq, dk, dv, du = mc_backward(q, k, v, u if has_u else None, dy.contiguous(), seg_len, agg_mode, topk)
        return dq, dk, dv, (du if has_u else None), None, None, None


def mc_check_device(stream=None) -> int:
    """Synchronise the stream and return MC_OK or MC_ERR_DEVICE_TIMEOUT (a kernel gave up
    on a bounded wait since the last check)."""
    return load_library().mc_check_device(_stream_handle(stream, torch.device("cuda")))


def mc_set_readout_form(form: int) -> int:
    """MC_READOUT_AUTO (the default) or MC_READOUT_FACTORISED for later forward calls;
    returns the previous setting."""
    st = load_library().mc_set_readout_form(int(form))
    if st < 0:
        raise MCError(st, "mc_set_readout_form")
    return st


def mc_trim_scratch() -> int:
    """Return the library's cached scratch memory on the current device to the driver."""
    return load_library().mc_trim_scratch()


def mc_ssc_select(k, u, seg_len: int, topk: int, *, idx=None, stream=None):
    """SSC router alone (``mc_ssc_select``): int32 [B,H,L,topk], rank order, -1 padded."""
    lib = load_library()
    B, H, L, d = k.shape
    dev = k.device
    _check(k, "k", k.dtype, (B, H, L, d), dev)
    _check(u, "u", k.dtype, (B, H, L, d), dev)
    if idx is None:
        idx = torch.empty((B, H, L, topk), dtype=torch.int32, device=dev)
    _check(idx, "idx", torch.int32, (B, H, L, topk), dev)
    st = lib.mc_ssc_select(k.data_ptr(), u.data_ptr(), B, H, L, d, int(seg_len), int(topk), idx.data_ptr(),
                           1 if k.dtype == torch.bfloat16 else 0, _stream_handle(stream, dev))
    if st != MC_OK:
        raise MCError(st, "mc_ssc_select")
    return idx


class KernelProfile:
    """Record CUDA events at every kernel boundary of the forward calls made inside
    the ``with`` block (``mc_profile_begin`` / ``mc_profile_end``).  After the block
    and a device synchronise, :meth:`per_kernel_ms` gives {kernel: [ms, ...]}."""

    def __init__(self, capacity: int = 1024):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        self._handles = None
        self.count = 0
        self.stages = []

    def __enter__(self):
        for e in self.events:
            e.record()  # materialise the lazily created events
        torch.cuda.synchronize()
        self._handles = (ctypes.c_void_p * len(self.events))(*[e.cuda_event for e in self.events])
        st = load_library().mc_profile_begin(self._handles, len(self.events))
        if st != MC_OK:
            raise MCError(st, "mc_profile_begin")
        return self

    def __exit__(self, *exc):
        lib = load_library()
        self.count = lib.mc_profile_end()
        self.stages = [lib.mc_profile_stage(j) for j in range(max(self.count - 1, 0))]
        self.stages = [s.decode() if s else None for s in self.stages]
        return False

    def per_kernel_ms(self) -> dict:
        out = {}
        for j, name in enumerate(self.stages):
            if name is None:
                continue
            out.setdefault(name, []).append(self.events[j].elapsed_time(self.events[j + 1]))
        return out

    def kernel_count(self) -> int:
        return sum(1 for s in self.stages if s is not None)


def mc_forward_host(q, k, v, u, seg_len: int, agg_mode: int, topk: int = 0, *, y=None, states=None,
                    stream=None):
    """End-to-end forward on HOST tensors (``mc_forward_host``): the library copies the
    inputs to the device, runs, copies y (and states, if given) back and synchronises."""
    lib = load_library()
    B, H, L, d = q.shape
    dtype = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, dtype, (B, H, L, d), torch.device("cpu"))
    if u is not None:
        _check(u, "u", dtype, (B, H, L, d), torch.device("cpu"))
    if y is None:
        y = torch.empty((B, H, L, d), dtype=dtype)
    _check(y, "y", dtype, (B, H, L, d), torch.device("cpu"))
    if states is not None:
        _check(states, "states", torch.float32, (B, H, num_segments(L, seg_len), d, d), torch.device("cpu"))
    st = lib.mc_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), u.data_ptr() if u is not None else None,
                             B, H, L, d, int(seg_len), int(agg_mode), int(topk), y.data_ptr(),
                             states.data_ptr() if states is not None else None,
                             1 if dtype == torch.bfloat16 else 0, _stream_handle(stream, torch.device("cuda")))
    if st != MC_OK:
        raise MCError(st, "mc_forward_host")
    return y, states
