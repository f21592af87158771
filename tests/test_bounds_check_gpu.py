"""The debug bounds-check build (-DGDN_BOUNDS_CHECK, csrc/gdn_check.cuh).

Builds the library with every shared-memory, tensor-memory and global index
of the tcgen05 and chunk-prep kernels checked, runs small parity cases
through it (dense and packed, ragged tails, both d_k, the fused variant and
one backward pass) and requires that no check failed: gdn_sync_check returns
GDN_OK and gdn_bounds_violation reports no line.  The outputs must still match
the fp64 oracle.
"""
import ctypes

import pytest
import torch

import gated_deltanet_recurrence_gdn_gb300 as gdn
from gated_deltanet_recurrence_gdn_gb300 import _build
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked_lib():
    lib = gdn.load(_build.build_variant("check"))
    prev = gdn._lib
    gdn._lib = lib   # the binding's calls go through the checked library
    try:
        assert lib.gdn_bounds_violation(1) == 0   # a checked build, nothing recorded yet
        yield lib
    finally:
        gdn._lib = prev


def _assert_clean(lib):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.gdn_sync_check(stream) == gdn.GDN_OK
    line = lib.gdn_bounds_violation(1)
    assert line == 0, "bounds check failed at source line %d" % line


@pytest.mark.parametrize("impl", [gdn.GDN_IMPL_TC, gdn.GDN_IMPL_TC_FUSED], ids=["tc", "fused"])
@pytest.mark.parametrize("case", [(2, 2, 3 * 64 + 17, 128, 128), (1, 2, 5 * 64 + 3, 64, 64),
                                  (1, 2, 2 * 64 + 40, 128, 256)],
                         ids=["t209_k128", "t323_k64", "t168_v256"])
def test_dense_parity_under_bounds_checks(checked_lib, impl, case):
    B, H, T, dk, dv = case
    x = synth.make_dense(B, H, T, dk, dv, io="bf16", h0_std=0.02, seed=400 + T, device="cuda")
    with gdn.use_impl(impl):
        o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0)
    _assert_clean(checked_lib)
    o_ref, h_ref = U.oracle_dense(x)
    to, th = U.TOL["bf16"]
    assert U.rel(U.f64(o), o_ref.reshape(o.shape)) <= to
    assert U.rel(U.f64(hT), h_ref.reshape(hT.shape)) <= th


@pytest.mark.parametrize("impl", [gdn.GDN_IMPL_TC, gdn.GDN_IMPL_TC_FUSED], ids=["tc", "fused"])
def test_packed_parity_under_bounds_checks(checked_lib, impl):
    import oracle
    y = synth.make_varlen([1, 63, 64, 65, 200, 0], 3, 128, 128, io="bf16", h0_std=0.02,
                          seed=431, device="cuda")
    with gdn.use_impl(impl):
        o, hT = gdn.gdn_fwd_varlen(y.q, y.k, y.v, y.log_alpha, y.beta, y.cu_seqlens, y.h0)
    _assert_clean(checked_lib)
    o_ref, h_ref = oracle.gdn_fwd_varlen(U.f64(y.q), U.f64(y.k), U.f64(y.v), U.f64(y.log_alpha),
                                         U.f64(y.beta), y.cu_seqlens.cpu().numpy(),
                                         U.f64(y.h0))
    to, th = U.TOL["bf16"]
    assert U.rel(U.f64(o), o_ref) <= to
    assert U.rel(U.f64(hT), h_ref) <= th


def test_segment_scan_and_backward_under_bounds_checks(checked_lib):
    x = synth.make_dense(1, 2, 8 * 64 + 5, 128, 128, io="bf16", h0_std=0.02, seed=433,
                         device="cuda")
    with gdn.use_impl(gdn.GDN_IMPL_TC, 3):   # three sequence segments
        gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0)
    _assert_clean(checked_lib)
    dout = torch.randn_like(x.v)
    grads = gdn.gdn_bwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, dout)
    _assert_clean(checked_lib)
    assert all(torch.isfinite(g.float()).all() for g in grads)
