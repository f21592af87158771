"""Thin Python binding of libgdn (the GB300 gated delta rule forward library).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libgdn.so``.  PyTorch supplies device memory and the current
stream.  If the library has not been built, importing works but every call
raises -- there is no CPU fallback.

    o, hT = gdn_fwd(q, k, v, log_alpha, beta, h0=None)
    o, hT = gdn_fwd_varlen(q, k, v, log_alpha, beta, cu_seqlens, h0=None)
    dq, dk, dv, dlog_alpha, dbeta, dh0 = gdn_bwd(q, k, v, log_alpha, beta, h0, dout, dhT)

Layouts follow ``include/gdn.h``: dense q, k [B,H,T,d_k], v [B,H,T,d_v]; packed
q, k [H,T_total,d_k], v [H,T_total,d_v]; gates fp32; h0 / hT [.., H, d_v, d_k]
fp32; q, k, v share one dtype (bf16 or fp32), which is also the dtype of o.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_ALIGNMENT = 3
GDN_ERR_CUDA = 4
GDN_ERR_DEVICE_TIMEOUT = 5
GDN_ERR_TOO_LARGE = 6
GDN_ERR_BOUNDS = 7
GDN_F32 = 0
GDN_BF16 = 1
GDN_OPT_IMPL = 0
GDN_OPT_SEGMENTS = 1
GDN_OPT_WAIT_LIMIT = 2
GDN_OPT_POISON_SCRATCH = 3
GDN_OPT_HOST_SLICE = 4
GDN_OPT_PREP_LEAD = 5
GDN_OPT_WIDE_CHAIN = 6
GDN_IMPL_AUTO = 0
GDN_IMPL_SIMT = 1
GDN_IMPL_TC = 2
GDN_IMPL_TC_FUSED = 3

CHUNK = 64

_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int

# (name, restype, argtypes) of every symbol include/gdn.h declares.
ABI = [
    ("gdn_fwd", _i, [_vp] * 8 + [_i] * 7 + [_vp]),
    ("gdn_fwd_varlen", _i, [_vp] * 9 + [_i] * 7 + [_vp]),
    ("gdn_fwd_noalloc", _i, [_vp] * 8 + [_i] * 7 + [_vp]),
    ("gdn_decode", _i, [_vp] * 7 + [_i] + [_vp] + [_i] * 5 + [_vp]),
    ("gdn_fwd_host", _i, [_vp] * 8 + [_i] * 7 + [_vp]),
    ("gdn_fwd_ex", _i, [_vp] * 8 + [_i] * 7 + [ctypes.c_uint, _vp]),
    ("gdn_fwd_varlen_ex", _i, [_vp] * 9 + [_i] * 7 + [ctypes.c_uint, _vp]),
    ("gdn_bwd", _i, [_vp] * 14 + [_i] * 7 + [ctypes.c_uint, _vp]),
    ("gdn_bwd_varlen", _i, [_vp] * 15 + [_i] * 7 + [ctypes.c_uint, _vp]),
    ("gdn_status_string", ctypes.c_char_p, [_i]),
    ("gdn_sync_check", _i, [_vp]),
    ("gdn_set_option", _i, [_i, ctypes.c_longlong]),
    ("gdn_get_option", ctypes.c_longlong, [_i]),
    ("gdn_kernel_timer", _i, [_i]),
    ("gdn_kernel_timer_read", _i, [ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_longlong),
                                   ctypes.POINTER(ctypes.c_char_p)]),
    ("gdn_kernel_launches", ctypes.c_uint64, []),
    ("gdn_scratch_stats", _i, [ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64), _i]),
    ("gdn_bounds_violation", _i, [_i]),
    ("gdn_last_impl", _i, []),
    ("gdn_release_scratch", _i, []),
    ("gdn_selftest_wait", _i, [_i, ctypes.c_longlong, ctypes.POINTER(_i), _vp]),
]


class GdnError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s%s" % (what + ": " if what else "", status_string(status)))


def load(path: str | None = None):
    """Load libgdn.so (built by ``_build.build()``) and declare its ABI."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError("libgdn.so is not built (%s); run __graft_entry__.build()" % p)
    lib = ctypes.CDLL(p)
    for name, res, args in ABI:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().gdn_status_string(int(status)).decode()
    except ImportError:
        return "status %d" % status


def _check(rc, what):
    if rc != GDN_OK:
        raise GdnError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


_DT = {torch.bfloat16: GDN_BF16, torch.float32: GDN_F32}


def _prep_io(q, k, v, log_alpha, beta, h0):
    for name, t in (("q", q), ("k", k), ("v", v), ("log_alpha", log_alpha), ("beta", beta)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, bf16 or fp32")
    if log_alpha.dtype != torch.float32 or beta.dtype != torch.float32:
        raise ValueError("log_alpha and beta must be fp32")
    if h0 is not None and (h0.dtype != torch.float32 or not h0.is_contiguous() or not h0.is_cuda):
        raise ValueError("h0 must be a contiguous fp32 CUDA tensor")


GDN_FLAG_NO_ERASE = 1
GDN_FLAG_VECTOR_GATE = 2


def gdn_fwd(q, k, v, log_alpha, beta, h0=None, *, chunk=CHUNK, out=None, final_state=True,
            check=False, erase=True):
    """Dense forward: returns (o [B,H,T,d_v], hT [B,H,d_v,d_k] or None).
    erase=False: gated linear attention (no delta-rule erase term).
    A log_alpha of shape [B,H,T,d_k] is a gate per key dimension."""
    lib = load()
    _prep_io(q, k, v, log_alpha, beta, h0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    vector_gate = log_alpha.dim() == 4
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or beta.shape != (B, H, T) \
            or log_alpha.shape != ((B, H, T, dk) if vector_gate else (B, H, T)):
        raise ValueError("shape mismatch")
    if h0 is not None and h0.shape != (B, H, dv, dk):
        raise ValueError("h0 must be [B,H,d_v,d_k]")
    o = out if out is not None else torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    hT = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device) if final_state else None
    with torch.cuda.device(q.device):
        args = (_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(h0),
                _ptr(o), _ptr(hT), B, H, T, dk, dv, chunk, _DT[q.dtype])
        flags = (0 if erase else GDN_FLAG_NO_ERASE) | (GDN_FLAG_VECTOR_GATE if vector_gate else 0)
        rc = (lib.gdn_fwd_ex(*args, flags, _stream(q.device)) if flags else
              lib.gdn_fwd(*args, _stream(q.device)))
        _check(rc, "gdn_fwd")
        if check:
            _check(lib.gdn_sync_check(_stream(q.device)), "gdn_fwd (device)")
    return o, hT


def gdn_fwd_varlen(q, k, v, log_alpha, beta, cu_seqlens, h0=None, *, chunk=CHUNK, out=None,
                   final_state=True, check=False, erase=True):
    """Packed forward: returns (o [H,T_total,d_v], hT [N,H,d_v,d_k] or None).
    erase=False: gated linear attention (no delta-rule erase term).
    A log_alpha of shape [H,T_total,d_k] is a gate per key dimension."""
    lib = load()
    _prep_io(q, k, v, log_alpha, beta, h0)
    H, TT, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    N = cu_seqlens.shape[0] - 1
    vector_gate = log_alpha.dim() == 3
    if k.shape != q.shape or v.shape[:2] != (H, TT) or beta.shape != (H, TT) \
            or log_alpha.shape != ((H, TT, dk) if vector_gate else (H, TT)):
        raise ValueError("shape mismatch")
    if h0 is not None and h0.shape != (N, H, dv, dk):
        raise ValueError("h0 must be [N,H,d_v,d_k]")
    o = out if out is not None else torch.empty((H, TT, dv), dtype=q.dtype, device=q.device)
    hT = torch.empty((N, H, dv, dk), dtype=torch.float32, device=q.device) if final_state else None
    with torch.cuda.device(q.device):
        args = (_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(h0), _ptr(o),
                _ptr(hT), _ptr(cu_seqlens.contiguous()), N, H, TT, dk, dv, chunk,
                _DT[q.dtype])
        flags = (0 if erase else GDN_FLAG_NO_ERASE) | (GDN_FLAG_VECTOR_GATE if vector_gate else 0)
        rc = (lib.gdn_fwd_varlen_ex(*args, flags, _stream(q.device)) if flags else
              lib.gdn_fwd_varlen(*args, _stream(q.device)))
        _check(rc, "gdn_fwd_varlen")
        if check:
            _check(lib.gdn_sync_check(_stream(q.device)), "gdn_fwd_varlen (device)")
    return o, hT


def _bwd_common(q, k, v, log_alpha, beta, h0, dout, dhT, n_states, dv_shape):
    _prep_io(q, k, v, log_alpha, beta, h0)
    if not isinstance(dout, torch.Tensor) or not dout.is_cuda or not dout.is_contiguous() \
            or dout.dtype != q.dtype or dout.shape != dv_shape:
        raise ValueError("dout must be a contiguous CUDA tensor shaped and typed like o")
    dk, dv = q.shape[-1], v.shape[-1]
    if dhT is not None and (dhT.dtype != torch.float32 or not dhT.is_contiguous()
                            or not dhT.is_cuda or dhT.shape != (*n_states, dv, dk)):
        raise ValueError("dhT must be a contiguous fp32 CUDA tensor shaped like hT")
    if log_alpha.shape != beta.shape:
        raise ValueError("vector gates have no backward pass")
    return (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
            torch.empty_like(log_alpha), torch.empty_like(beta),
            torch.empty((*n_states, dv, dk), dtype=torch.float32, device=q.device))


def gdn_bwd(q, k, v, log_alpha, beta, h0, dout, dhT=None, *, chunk=CHUNK, erase=True,
            check=False):
    """Dense backward pass: the gradient of sum(dout * o) + sum(dhT * hT) for
    the forward gdn_fwd(q, k, v, log_alpha, beta, h0, erase=erase).  Returns
    (dq, dk, dv, dlog_alpha, dbeta, dh0); dh0 [B,H,d_v,d_k] is the gradient
    at the zero state when h0 is None."""
    lib = load()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or log_alpha.shape != (B, H, T) \
            or beta.shape != (B, H, T):
        raise ValueError("shape mismatch")
    if h0 is not None and h0.shape != (B, H, dv, dk):
        raise ValueError("h0 must be [B,H,d_v,d_k]")
    g = _bwd_common(q, k, v, log_alpha, beta, h0, dout, dhT, (B, H), (B, H, T, dv))
    with torch.cuda.device(q.device):
        rc = lib.gdn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(h0),
                         _ptr(dout), _ptr(dhT), *(_ptr(t) for t in g), B, H, T, dk, dv, chunk,
                         _DT[q.dtype], 0 if erase else GDN_FLAG_NO_ERASE, _stream(q.device))
        _check(rc, "gdn_bwd")
        if check:
            _check(lib.gdn_sync_check(_stream(q.device)), "gdn_bwd (device)")
    return g


def gdn_bwd_varlen(q, k, v, log_alpha, beta, cu_seqlens, h0, dout, dhT=None, *, chunk=CHUNK,
                   erase=True, check=False):
    """Packed backward pass (layouts as gdn_fwd_varlen).  Returns
    (dq, dk, dv, dlog_alpha, dbeta, dh0 [N,H,d_v,d_k])."""
    lib = load()
    H, TT, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    N = cu_seqlens.shape[0] - 1
    if k.shape != q.shape or v.shape[:2] != (H, TT) or log_alpha.shape != (H, TT) \
            or beta.shape != (H, TT):
        raise ValueError("shape mismatch")
    if h0 is not None and h0.shape != (N, H, dv, dk):
        raise ValueError("h0 must be [N,H,d_v,d_k]")
    g = _bwd_common(q, k, v, log_alpha, beta, h0, dout, dhT, (N, H), (H, TT, dv))
    with torch.cuda.device(q.device):
        rc = lib.gdn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                _ptr(h0), _ptr(dout), _ptr(dhT), *(_ptr(t) for t in g),
                                _ptr(cu_seqlens.contiguous()), N, H, TT, dk, dv, chunk,
                                _DT[q.dtype], 0 if erase else GDN_FLAG_NO_ERASE,
                                _stream(q.device))
        _check(rc, "gdn_bwd_varlen")
        if check:
            _check(lib.gdn_sync_check(_stream(q.device)), "gdn_bwd_varlen (device)")
    return g


def gdn_fwd_noalloc(q, k, v, log_alpha, beta, h0=None, *, chunk=CHUNK, out=None,
                    final_state=None, check=False):
    """Dense forward through the allocation-free entry point: the library
    allocates nothing (its scratch is a fixed 32 MiB device array); the
    caller passes the outputs (`out`, `final_state`) or they are created here
    with torch.  Returns (o, hT)."""
    lib = load()
    _prep_io(q, k, v, log_alpha, beta, h0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = out if out is not None else torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    hT = final_state if final_state is not None else torch.empty(
        (B, H, dv, dk), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.gdn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                 _ptr(h0), _ptr(o), _ptr(hT), B, H, T, dk, dv, chunk,
                                 _DT[q.dtype], _stream(q.device))
        _check(rc, "gdn_fwd_noalloc")
        if check:
            _check(lib.gdn_sync_check(_stream(q.device)), "gdn_fwd_noalloc (device)")
    return o, hT


def gdn_fwd_host(q, k, v, log_alpha, beta, h0=None, *, chunk=CHUNK, out=None, final_state=True,
                 final_out=None, sync=True, device=None):
    """Dense forward on HOST tensors (page-locked for overlapped copies): the
    library uploads, computes and downloads in a pipeline over time slices.
    Returns host (o, hT); `out` / `final_out` receive them when given.  With
    sync=False the caller synchronises the current stream of `device` before
    reading the results."""
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("log_alpha", log_alpha), ("beta", beta)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous host tensor" % name)
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, bf16 or fp32")
    if log_alpha.dtype != torch.float32 or beta.dtype != torch.float32:
        raise ValueError("log_alpha and beta must be fp32")
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or log_alpha.shape != (B, H, T) \
            or beta.shape != (B, H, T):
        raise ValueError("shape mismatch")
    if h0 is not None and (h0.is_cuda or h0.dtype != torch.float32 or not h0.is_contiguous()
                           or h0.shape != (B, H, dv, dk)):
        raise ValueError("h0 must be a contiguous fp32 host tensor [B,H,d_v,d_k]")
    o = out if out is not None else torch.empty((B, H, T, dv), dtype=q.dtype).pin_memory()
    hT = final_out if final_out is not None else (
        torch.empty((B, H, dv, dk), dtype=torch.float32).pin_memory() if final_state else None)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        rc = lib.gdn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(h0),
                              _ptr(o), _ptr(hT), B, H, T, dk, dv, chunk, _DT[q.dtype],
                              _stream(dev))
        _check(rc, "gdn_fwd_host")
        if sync:
            _check(lib.gdn_sync_check(_stream(dev)), "gdn_fwd_host (device)")
    return o, hT


def gdn_decode(q, k, v, log_alpha, beta, state, *, slots=None, out=None, check=False):
    """One decode step for every (sequence, head), the state updated in place.

    q, k [B,H,d_k] and v [B,H,d_v] (bf16 or fp32, one dtype); log_alpha, beta
    [B,H] fp32; state fp32 [B,H,d_v,d_k], or a pool [P,H,d_v,d_k] indexed by
    `slots` (int32 [B] on the device, distinct).  Returns o [B,H,d_v]."""
    lib = load()
    _prep_io(q, k, v, log_alpha, beta, None)
    if state.dtype != torch.float32 or not state.is_contiguous() or not state.is_cuda:
        raise ValueError("state must be a contiguous fp32 CUDA tensor")
    B, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:2] != (B, H) or log_alpha.shape != (B, H) \
            or beta.shape != (B, H):
        raise ValueError("shape mismatch")
    if slots is not None:
        if slots.dtype != torch.int32 or not slots.is_cuda or slots.shape != (B,):
            raise ValueError("slots must be an int32 CUDA tensor of shape [B]")
        slots = slots.contiguous()
        n_slots = state.shape[0]
    else:
        n_slots = B
    if state.shape[1:] != (H, dv, dk) or state.shape[0] != n_slots:
        raise ValueError("state must be [B or P, H, d_v, d_k]")
    o = out if out is not None else torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.gdn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                            _ptr(state), _ptr(slots), n_slots, _ptr(o), B, H, dk, dv,
                            _DT[q.dtype], _stream(q.device))
        _check(rc, "gdn_decode")
        if check:
            _check(lib.gdn_sync_check(_stream(q.device)), "gdn_decode (device)")
    return o


def sync_check(device=None):
    """Synchronise the current stream and raise if a kernel recorded an error."""
    _check(load().gdn_sync_check(_stream(device)), "device")


def set_option(key: int, value: int):
    _check(load().gdn_set_option(int(key), int(value)), "gdn_set_option")


def get_option(key: int) -> int:
    return int(load().gdn_get_option(int(key)))


def kernel_launches() -> int:
    return int(load().gdn_kernel_launches())


def scratch_stats(reset_high: bool = False):
    """(bytes in use, high-water mark) of the current device's scratch pool;
    reset_high restarts the high-water mark from the current use afterwards."""
    cur = ctypes.c_uint64(0)
    high = ctypes.c_uint64(0)
    _check(load().gdn_scratch_stats(ctypes.byref(cur), ctypes.byref(high), 1 if reset_high else 0),
           "gdn_scratch_stats")
    return int(cur.value), int(high.value)


def kernel_timer(enable: bool):
    _check(load().gdn_kernel_timer(1 if enable else 0), "gdn_kernel_timer")


def kernel_timer_read():
    """(total_ms, launches, kernel_name) of the dominant kernel since the last read."""
    ms = ctypes.c_double(0.0)
    n = ctypes.c_longlong(0)
    name = ctypes.c_char_p()
    _check(load().gdn_kernel_timer_read(ctypes.byref(ms), ctypes.byref(n), ctypes.byref(name)),
           "gdn_kernel_timer_read")
    return ms.value, n.value, (name.value or b"").decode()


def last_impl() -> int:
    return int(load().gdn_last_impl())


def release_scratch(device=None) -> None:
    """Hand the scratch memory the library's pool keeps on `device` (default:
    the current one) back to the CUDA driver."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _check(load().gdn_release_scratch(), "gdn_release_scratch")


def selftest_wait(complete: bool, limit: int, device=None):
    """Device self-test of the bounded waits (include/gdn_selftest.h): one CTA
    waits on an mbarrier phase and a counter that it completes itself
    (complete=True) or that nothing completes (the mbarrier wait then gives
    up after `limit` suspending polls, the counter wait after 4 * limit loads,
    and a timeout is recorded that the next sync_check reports).
    Returns (mbarrier wait succeeded, counter wait succeeded)."""
    ok = (_i * 2)()
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _check(load().gdn_selftest_wait(1 if complete else 0, int(limit), ok, _stream(device)),
               "gdn_selftest_wait")
    return bool(ok[0]), bool(ok[1])


class use_impl:
    """Context manager forcing GDN_IMPL_SIMT / GDN_IMPL_TC / GDN_IMPL_TC_FUSED / GDN_IMPL_AUTO."""

    def __init__(self, impl: int, segments: int | None = None):
        self.impl, self.segments = impl, segments

    def __enter__(self):
        self.prev = (get_option(GDN_OPT_IMPL), get_option(GDN_OPT_SEGMENTS))
        set_option(GDN_OPT_IMPL, self.impl)
        if self.segments is not None:
            set_option(GDN_OPT_SEGMENTS, self.segments)
        return self

    def __exit__(self, *exc):
        set_option(GDN_OPT_IMPL, self.prev[0])
        set_option(GDN_OPT_SEGMENTS, self.prev[1])
        return False
