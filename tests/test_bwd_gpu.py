"""Backward pass (gdn_bwd / gdn_bwd_varlen) against the fp64 gradient oracle
on the same seeded inputs and output weights (GPU)."""
import numpy as np
import pytest
import torch

import gated_deltanet_recurrence_gdn_gb300 as gdn
import oracle
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dh0")
# max|delta| / max|reference| per gradient.  fp32 I/O: fp32 arithmetic
# throughout; bf16 I/O: dq, dk, dv are rounded to bf16 once (2^-9 relative)
# on top of the same fp32 arithmetic.
BWD_TOL = {"f32": 1e-4, "bf16": 1e-2}


def _weights(x, seed, dhT=True, packed=False):
    g = torch.Generator(device="cuda").manual_seed(seed)
    dout = torch.randn(x.v.shape, generator=g, device="cuda").to(x.q.dtype)
    if not dhT:
        return dout, None
    n_states = (x.meta["N"], x.meta["H"]) if packed else (x.meta["B"], x.meta["H"])
    dk, dv = x.q.shape[-1], x.v.shape[-1]
    return dout, torch.randn((*n_states, dv, dk), generator=g, device="cuda")


def _compare(got, ref, io, skip=()):
    errs = {}
    for name, a, b in zip(NAMES, got, ref):
        if name in skip:
            continue
        a = U.f64(a)
        assert np.isfinite(a).all(), name
        errs[name] = U.rel(a, b)
    assert max(errs.values()) <= BWD_TOL[io], errs
    return errs


def _expected_impl(io, dk, dv, impl):
    """The state adjoint the backward takes: the tcgen05 kernel for bf16 I/O
    with d_k 64 or 128 and d_v a multiple of 64, unless mma.sync is forced."""
    tc_fits = io == "bf16" and dk in (64, 128) and dv % 64 == 0
    return gdn.GDN_IMPL_TC if (tc_fits and impl != gdn.GDN_IMPL_SIMT) else gdn.GDN_IMPL_SIMT


@pytest.mark.parametrize("impl", [gdn.GDN_IMPL_AUTO, gdn.GDN_IMPL_SIMT], ids=["auto", "simt"])
@pytest.mark.parametrize("erase", [True, False])
@pytest.mark.parametrize("B,H,T,dk,dv,io", [(1, 2, 130, 64, 64, "f32"),
                                            (2, 2, 257, 64, 64, "bf16"),
                                            (2, 2, 300, 128, 128, "bf16"),
                                            (1, 3, 200, 64, 128, "bf16"),
                                            (2, 1, 150, 32, 48, "f32"),
                                            (1, 1, 64, 128, 256, "bf16")])
def test_bwd_matches_oracle(impl, erase, B, H, T, dk, dv, io):
    x = synth.make_dense(B, H, T, dk, dv, io=io, h0_std=0.1, seed=T + 61, device="cuda")
    dout, dhT = _weights(x, T + 62)
    with gdn.use_impl(impl):
        got = gdn.gdn_bwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, dout, dhT, erase=erase,
                          check=True)
        U.sync()
    assert gdn.last_impl() == _expected_impl(io, dk, dv, impl)
    ref = oracle.gdn_bwd(U.f64(x.q), U.f64(x.k), U.f64(x.v), U.f64(x.log_alpha),
                         U.f64(x.beta), U.f64(x.h0), U.f64(dout), U.f64(dhT),
                         threads=U.ORACLE_THREADS, erase=erase)
    _compare(got, ref, io)


@pytest.mark.parametrize("impl", [gdn.GDN_IMPL_AUTO, gdn.GDN_IMPL_SIMT], ids=["auto", "simt"])
@pytest.mark.parametrize("erase", [True, False])
def test_bwd_varlen_matches_oracle(impl, erase):
    y = synth.make_varlen([1, 63, 64, 65, 200, 0, 129], 2, 128, 128, io="bf16", h0_std=0.1,
                          seed=71, device="cuda")
    dout, dhT = _weights(y, 72, packed=True)
    with gdn.use_impl(impl):
        got = gdn.gdn_bwd_varlen(y.q, y.k, y.v, y.log_alpha, y.beta, y.cu_seqlens, y.h0, dout,
                                 dhT, erase=erase, check=True)
        U.sync()
    assert gdn.last_impl() == _expected_impl("bf16", 128, 128, impl)
    ref = oracle.gdn_bwd_varlen(U.f64(y.q), U.f64(y.k), U.f64(y.v), U.f64(y.log_alpha),
                                U.f64(y.beta), y.cu_seqlens.cpu().numpy(), U.f64(y.h0),
                                U.f64(dout), U.f64(dhT), erase=erase)
    _compare(got, ref, "bf16")


def test_bwd_without_h0_or_dhT():
    x = synth.make_dense(1, 2, 190, 64, 64, io="f32", seed=73, device="cuda")
    dout, _ = _weights(x, 74, dhT=False)
    got = gdn.gdn_bwd(x.q, x.k, x.v, x.log_alpha, x.beta, None, dout, None, check=True)
    U.sync()
    ref = oracle.gdn_bwd(U.f64(x.q), U.f64(x.k), U.f64(x.v), U.f64(x.log_alpha),
                         U.f64(x.beta), None, U.f64(dout), None)
    _compare(got, ref, "f32")


def test_bwd_empty_sequence_passes_dhT_through():
    x = synth.make_dense(2, 2, 0, 64, 64, io="bf16", h0_std=0.1, seed=75, device="cuda")
    dout, dhT = _weights(x, 76)
    got = gdn.gdn_bwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, dout, dhT, check=True)
    U.sync()
    assert torch.equal(got[5], dhT)
    assert got[0].numel() == 0


def test_bwd_adjoint_identity_full_size():
    # At B4 H16 T4096 d128 bf16: L = <dO, O> + <dhT, hT> is linear in (h0, V),
    # so L = <dV, V> + <dh0, h0>, and <dO, O> = <dq, q>; both hold for the exact
    # gradient at any size.  The forward here is the tensor-core gdn_fwd.
    x = synth.make_workload("gdn_fwd_b4_h16_t4096_d128_bf16", device="cuda")
    h0 = torch.randn((4, 16, 128, 128), device="cuda") * 0.05
    dout, dhT = _weights(x, 77)
    o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, h0)
    dq, _, dv, _, _, dh0 = gdn.gdn_bwd(x.q, x.k, x.v, x.log_alpha, x.beta, h0, dout, dhT,
                                       check=True)
    U.sync()
    f = lambda a, b: float((a.double() * b.double()).sum())
    L_o, L_h = f(dout, o), f(dhT, hT)
    lin = f(dv, x.v) + f(dh0, h0)
    assert abs(L_o + L_h - lin) <= 2e-2 * (abs(L_o) + abs(L_h))
    assert abs(L_o - f(dq, x.q)) <= 2e-2 * abs(L_o)


def test_bwd_full_size_sampled_heads():
    # The same workload, two (batch, head) pairs against the oracle gradient.
    x = synth.make_workload("gdn_fwd_b4_h16_t4096_d128_bf16", device="cuda")
    dout, dhT = _weights(x, 78)
    got = gdn.gdn_bwd(x.q, x.k, x.v, x.log_alpha, x.beta, None, dout, dhT, check=True)
    U.sync()
    for b, h in ((0, 0), (3, 15)):
        sl = lambda t: U.f64(t[b:b + 1, h:h + 1])
        ref = oracle.gdn_bwd(sl(x.q), sl(x.k), sl(x.v), sl(x.log_alpha), sl(x.beta), None,
                             sl(dout), sl(dhT))
        _compare([t[b:b + 1, h:h + 1] for t in got], ref, "bf16")


def test_bwd_vector_gate_and_forced_tc_outside_its_shapes_are_unsupported():
    x = synth.make_dense(1, 1, 64, 64, 64, io="bf16", seed=79, device="cuda")
    dout, dhT = _weights(x, 80)
    lib = gdn.load()
    g = [torch.empty_like(t) for t in (x.q, x.k, x.v, x.log_alpha, x.beta)]
    ptr = gdn._ptr
    stream = gdn._stream(x.q.device)
    rc = lib.gdn_bwd(ptr(x.q), ptr(x.k), ptr(x.v), ptr(x.log_alpha), ptr(x.beta), None,
                     ptr(dout), ptr(dhT), *(ptr(t) for t in g), None, 1, 1, 64, 64, 64, 64,
                     gdn.GDN_BF16, gdn.GDN_FLAG_VECTOR_GATE, stream)
    assert rc == gdn.GDN_ERR_UNSUPPORTED
    # the tcgen05 state adjoint takes bf16 I/O only: forced on fp32 I/O it refuses
    xf = synth.make_dense(1, 1, 64, 64, 64, io="f32", seed=79, device="cuda")
    doutf, dhTf = _weights(xf, 80)
    with gdn.use_impl(gdn.GDN_IMPL_TC):
        with pytest.raises(gdn.GdnError) as e:
            gdn.gdn_bwd(xf.q, xf.k, xf.v, xf.log_alpha, xf.beta, None, doutf, dhTf)
        assert e.value.status == gdn.GDN_ERR_UNSUPPORTED
        # and runs where it fits
        gdn.gdn_bwd(x.q, x.k, x.v, x.log_alpha, x.beta, None, dout, dhT, check=True)
        U.sync()
    assert gdn.last_impl() == gdn.GDN_IMPL_TC


@pytest.mark.parametrize("impl", [gdn.GDN_IMPL_AUTO, gdn.GDN_IMPL_SIMT], ids=["auto", "simt"])
@pytest.mark.parametrize("steep", [(1, 3), (1, 2, 3)], ids=["apart", "consecutive"])
def test_bwd_steep_decay_matches_oracle(impl, steep):
    # log gates of -3 per step in some chunks: their total log decay is below
    # -80, where exp(-g_s) would overflow, so those chunks take the
    # unscaled-dO branch of the tensor-core state adjoint (and the wide-span
    # branch of the state pass); the others the gamma dO one
    x = synth.make_dense(1, 2, 256, 128, 128, io="bf16", h0_std=0.1, seed=83, device="cuda")
    la = x.log_alpha.clone()
    for c in steep:
        la[..., 64 * c:64 * (c + 1)] = -3.0
    dout, dhT = _weights(x, 84)
    with gdn.use_impl(impl):
        got = gdn.gdn_bwd(x.q, x.k, x.v, la, x.beta, x.h0, dout, dhT, check=True)
        U.sync()
    assert gdn.last_impl() == _expected_impl("bf16", 128, 128, impl)
    ref = oracle.gdn_bwd(U.f64(x.q), U.f64(x.k), U.f64(x.v), U.f64(la), U.f64(x.beta),
                         U.f64(x.h0), U.f64(dout), U.f64(dhT))
    _compare(got, ref, "bf16")


def test_bwd_long_sequence_adjoint_identity():
    # 256 chunks per head: the state adjoint crosses many chunk boundaries.
    # <dO, O> + <dhT, hT> = <dV, V> + <dh0, h0> and <dO, O> = <dq, q> hold for
    # the exact gradient at any length (the fp64 oracle, which keeps every
    # state, would need 17 GB per head here).
    x = synth.make_dense(1, 2, 16384, 128, 128, io="bf16", decay="slow", h0_std=0.05, seed=81,
                         device="cuda")
    dout, dhT = _weights(x, 82)
    o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0)
    dq, _, dv, _, _, dh0 = gdn.gdn_bwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, dout, dhT,
                                       check=True)
    U.sync()
    f = lambda a, b: float((a.double() * b.double()).sum())
    L_o, L_h = f(dout, o), f(dhT, hT)
    assert abs(L_o + L_h - f(dv, x.v) - f(dh0, x.h0)) <= 2e-2 * (abs(L_o) + abs(L_h))
    assert abs(L_o - f(dq, x.q)) <= 2e-2 * abs(L_o)


def test_bwd_varlen_without_h0_or_dhT_fp32():
    y = synth.make_varlen([5, 64, 0, 150], 3, 64, 32, io="f32", seed=83, device="cuda")
    dout = torch.randn(y.v.shape, generator=torch.Generator(device="cuda").manual_seed(84),
                       device="cuda")
    got = gdn.gdn_bwd_varlen(y.q, y.k, y.v, y.log_alpha, y.beta, y.cu_seqlens, None, dout,
                             None, check=True)
    U.sync()
    ref = oracle.gdn_bwd_varlen(U.f64(y.q), U.f64(y.k), U.f64(y.v), U.f64(y.log_alpha),
                                U.f64(y.beta), y.cu_seqlens.cpu().numpy(), None, U.f64(dout))
    _compare(got, ref, "f32")
