"""fp64 CPU oracle for the gated delta rule forward pass.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference arm of ``bench.py`` are the only callers.  The
product package never imports this module, and this module never imports the
product package.

The arithmetic lives in ``gdn_oracle.c`` (plain single-threaded fp64 C, the
per-token loop of "Gated DeltaNet GPU并行实现" section 1.3 with the update of
sections 2.1-2.2).  This file only compiles it with gcc and marshals numpy
arrays.  ``threads > 1`` runs independent (sequence, head) problems on several
host threads; each problem is still the same single-threaded loop.

``gdn_bwd`` / ``gdn_bwd_varlen`` return the gradient of
L = sum(dO * o) + sum(dhT * hT) with respect to every input (reverse-mode
differentiation of the same loop, the forward states kept).

Parity status: pinned by closed forms and invariants in
tests/test_oracle_pins.py (beta = 0 decay, exact recall S k = v for
alpha = beta = 1, affine-map bracketing, the T = 1 closed form, reduction to
(gated) linear attention, linearity, continuation, varlen splitting; for the
gradient: central finite differences of the forward loop, the exact adjoint
identities of its linear arguments), by examples worked by hand
(tests/golden/, checked in tests/test_golden.py), and by planted-mistake
checks that each of those pins catches.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)


def compile_source(src: str, out: str) -> str:
    """Compile one oracle C source into a shared library with plain gcc -O2."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", src, "-o", tmp, "-lm"],
                   check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build libgdn_oracle.so next to this file (idempotent)."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    lib = ctypes.CDLL(path)
    lib.gdn_oracle_fwd.restype = ctypes.c_int
    lib.gdn_oracle_fwd.argtypes = [_dp] * 8 + [ctypes.c_long] * 5
    lib.gdn_oracle_fwd_varlen.restype = ctypes.c_int
    lib.gdn_oracle_fwd_varlen.argtypes = [_dp] * 8 + [_lp] + [ctypes.c_long] * 5
    lib.gdn_oracle_gla_fwd.restype = ctypes.c_int
    lib.gdn_oracle_gla_fwd.argtypes = [_dp] * 8 + [ctypes.c_long] * 5
    lib.gdn_oracle_gla_fwd_varlen.restype = ctypes.c_int
    lib.gdn_oracle_gla_fwd_varlen.argtypes = [_dp] * 8 + [_lp] + [ctypes.c_long] * 5
    lib.gdn_oracle_vg_fwd.restype = ctypes.c_int
    lib.gdn_oracle_vg_fwd.argtypes = [_dp] * 8 + [ctypes.c_long] * 6
    lib.gdn_oracle_vg_fwd_varlen.restype = ctypes.c_int
    lib.gdn_oracle_vg_fwd_varlen.argtypes = [_dp] * 8 + [_lp] + [ctypes.c_long] * 6
    lib.gdn_oracle_bwd.restype = ctypes.c_int
    lib.gdn_oracle_bwd.argtypes = [_dp] * 14 + [ctypes.c_long] * 6
    lib.gdn_oracle_bwd_varlen.restype = ctypes.c_int
    lib.gdn_oracle_bwd_varlen.argtypes = [_dp] * 14 + [_lp] + [ctypes.c_long] * 6
    return lib


def _get():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def gdn_fwd(q, k, v, log_alpha, beta, h0=None, *, threads: int = 1, lib=None, erase=True,
            vector_gate=False):
    """Dense oracle.  q,k [B,H,T,dk]; v [B,H,T,dv]; log_alpha, beta [B,H,T];
    h0 [B,H,dv,dk] or None.  Returns (o [B,H,T,dv], hT [B,H,dv,dk]) in fp64.
    erase=False runs gated linear attention (the recurrence without the
    delta rule's erase term); vector_gate=True takes log_alpha [B,H,T,dk], a
    gate per key dimension."""
    lib = lib or _get()
    if vector_gate:
        def fwd(*a):
            return lib.gdn_oracle_vg_fwd(*a, 1 if erase else 0)
    else:
        fwd = lib.gdn_oracle_fwd if erase else lib.gdn_oracle_gla_fwd
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, be = _f64(log_alpha), _f64(beta)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape == (B, H, T, dv)
    assert la.shape == ((B, H, T, dk) if vector_gate else (B, H, T)) and be.shape == (B, H, T)
    if h0 is not None:
        h0 = _f64(h0)
        assert h0.shape == (B, H, dv, dk)
    o = np.zeros((B, H, T, dv), dtype=np.float64)
    hT = np.zeros((B, H, dv, dk), dtype=np.float64)

    def run(b, h):
        rc = fwd(_ptr(q[b, h]), _ptr(k[b, h]), _ptr(v[b, h]),
                                _ptr(la[b, h]), _ptr(be[b, h]),
                                None if h0 is None else _ptr(h0[b, h]),
                                _ptr(o[b, h]), _ptr(hT[b, h]), 1, 1, T, dk, dv)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")

    jobs = [(b, h) for b in range(B) for h in range(H)]
    if threads <= 1 or len(jobs) <= 1:
        for j in jobs:
            run(*j)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda j: run(*j), jobs))
    return o, hT


def gdn_fwd_varlen(q, k, v, log_alpha, beta, cu_seqlens, h0=None, *, threads: int = 1,
                   lib=None, erase=True, vector_gate=False):
    """Packed oracle.  q,k [H,T_total,dk]; v [H,T_total,dv]; log_alpha, beta
    [H,T_total] (log_alpha [H,T_total,dk] with vector_gate); cu_seqlens [N+1];
    h0 [N,H,dv,dk] or None.  Returns (o [H,T_total,dv], hT [N,H,dv,dk]) in
    fp64.  erase=False runs gated linear attention."""
    lib = lib or _get()
    if vector_gate:
        def fwd(*a):
            return lib.gdn_oracle_vg_fwd(*a, 1 if erase else 0)

        def fwd_varlen(*a):
            return lib.gdn_oracle_vg_fwd_varlen(*a, 1 if erase else 0)
    else:
        fwd = lib.gdn_oracle_fwd if erase else lib.gdn_oracle_gla_fwd
        fwd_varlen = lib.gdn_oracle_fwd_varlen if erase else lib.gdn_oracle_gla_fwd_varlen
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, be = _f64(log_alpha), _f64(beta)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    H, TT, dk = q.shape
    dv = v.shape[-1]
    N = cu.shape[0] - 1
    if h0 is not None:
        h0 = _f64(h0)
        assert h0.shape == (N, H, dv, dk)
    o = np.zeros((H, TT, dv), dtype=np.float64)
    hT = np.zeros((N, H, dv, dk), dtype=np.float64)
    if threads <= 1 or N * H <= 1:
        rc = fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(be),
                                       _ptr(h0), _ptr(o), _ptr(hT),
                                       cu.ctypes.data_as(_lp), N, H, TT, dk, dv)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return o, hT

    # Independent (sequence, head) problems on several threads: each job is the
    # dense single-head loop on that sequence's contiguous token range.
    def run(n, h):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        ob = np.zeros((t1 - t0, dv), dtype=np.float64)
        hb = np.zeros((dv, dk), dtype=np.float64)
        rc = fwd(_ptr(np.ascontiguousarray(q[h, t0:t1])),
                                _ptr(np.ascontiguousarray(k[h, t0:t1])),
                                _ptr(np.ascontiguousarray(v[h, t0:t1])),
                                _ptr(np.ascontiguousarray(la[h, t0:t1])),
                                _ptr(np.ascontiguousarray(be[h, t0:t1])),
                                None if h0 is None else _ptr(np.ascontiguousarray(h0[n, h])),
                                _ptr(ob), _ptr(hb), 1, 1, t1 - t0, dk, dv)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        o[h, t0:t1] = ob
        hT[n, h] = hb

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda j: run(*j), [(n, h) for n in range(N) for h in range(H)]))
    return o, hT


def gdn_bwd(q, k, v, log_alpha, beta, h0, dout, dhT=None, *, threads: int = 1, lib=None,
            erase=True):
    """Dense gradient oracle.  Inputs as gdn_fwd; dout [B,H,T,dv]; dhT
    [B,H,dv,dk] or None (zero).  Returns (dq, dk, dv, dlog_alpha, dbeta, dh0)
    in fp64, each in its input's layout (dh0 [B,H,dv,dk] even when h0 is None:
    the gradient at the zero state)."""
    lib = lib or _get()
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, be, do = _f64(log_alpha), _f64(beta), _f64(dout)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape == (B, H, T, dv) and do.shape == v.shape
    assert la.shape == (B, H, T) and be.shape == (B, H, T)
    h0 = None if h0 is None else _f64(h0)
    dhT = None if dhT is None else _f64(dhT)
    for t in (h0, dhT):
        assert t is None or t.shape == (B, H, dv, dk)
    out = [np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape), np.zeros(la.shape),
           np.zeros(be.shape), np.zeros((B, H, dv, dk))]

    def run(b, h):
        def sl(a):
            return None if a is None else _ptr(a[b, h])
        rc = lib.gdn_oracle_bwd(sl(q), sl(k), sl(v), sl(la), sl(be), sl(h0), sl(do), sl(dhT),
                                *(sl(x) for x in out), 1, 1, T, dk, dv, 1 if erase else 0)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")

    jobs = [(b, h) for b in range(B) for h in range(H)]
    if threads <= 1 or len(jobs) <= 1:
        for j in jobs:
            run(*j)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda j: run(*j), jobs))
    return tuple(out)


def gdn_bwd_varlen(q, k, v, log_alpha, beta, cu_seqlens, h0, dout, dhT=None, *, lib=None,
                   erase=True):
    """Packed gradient oracle.  Inputs as gdn_fwd_varlen; dout [H,T_total,dv];
    dhT [N,H,dv,dk] or None.  Returns (dq, dk, dv, dlog_alpha, dbeta, dh0)."""
    lib = lib or _get()
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, be, do = _f64(log_alpha), _f64(beta), _f64(dout)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    H, TT, dk = q.shape
    dv = v.shape[-1]
    N = cu.shape[0] - 1
    h0 = None if h0 is None else _f64(h0)
    dhT = None if dhT is None else _f64(dhT)
    out = [np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape), np.zeros(la.shape),
           np.zeros(be.shape), np.zeros((N, H, dv, dk))]
    rc = lib.gdn_oracle_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(be), _ptr(h0),
                                   _ptr(do), _ptr(dhT), *(_ptr(x) for x in out),
                                   cu.ctypes.data_as(_lp), N, H, TT, dk, dv,
                                   1 if erase else 0)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return tuple(out)
