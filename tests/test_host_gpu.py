"""gdn_fwd_host: the forward pass on host buffers, pipelined over time slices.

The slices are chunk-aligned and the fp32 state passes between them through
device memory, so the result must equal the device entry point's on the same
inputs bit for bit (when the device call does not split the sequence for its
segment scan), and match the fp64 oracle within the stated tolerances."""
from __future__ import annotations

import pytest
import torch

import gated_deltanet_recurrence_gdn_gb300 as gdn
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def host_inputs(x, pin=True):
    f = (lambda t: None if t is None else t.cpu().pin_memory()) if pin else \
        (lambda t: None if t is None else t.cpu())
    return [f(t) for t in (x.q, x.k, x.v, x.log_alpha, x.beta, x.h0)]


@pytest.mark.parametrize("io,B,H,T,dk,dv", [("bf16", 2, 3, 1500, 128, 128),
                                            ("bf16", 1, 2, 2048, 64, 64),
                                            ("bf16", 1, 1, 700, 128, 256),
                                            ("f32", 2, 2, 1100, 64, 64)])
def test_host_equals_device_call(io, B, H, T, dk, dv):
    x = synth.make_dense(B, H, T, dk, dv, io=io, h0_std=0.02, seed=T + dk, device="cuda")
    with gdn.use_impl(gdn.GDN_IMPL_AUTO, 1):
        o_d, h_d = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
        o_h, h_h = gdn.gdn_fwd_host(*host_inputs(x))
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(h_h, h_d.cpu())


def test_host_matches_oracle():
    x = synth.make_dense(2, 2, 1300, 128, 128, io="bf16", h0_std=0.02, seed=12, device="cuda")
    o, hT = gdn.gdn_fwd_host(*host_inputs(x))
    o_ref, h_ref = U.oracle_dense(x)
    assert U.rel(U.f64(o), o_ref.reshape(o.shape)) <= 1e-2
    assert U.rel(U.f64(hT), h_ref.reshape(hT.shape)) <= 2e-2


def test_host_pageable_and_options():
    x = synth.make_dense(1, 2, 600, 64, 64, io="bf16", h0_std=0.02, seed=13, device="cuda")
    o_p, h_p = gdn.gdn_fwd_host(*host_inputs(x, pin=False))
    o_q, h_q = gdn.gdn_fwd_host(*host_inputs(x))
    assert torch.equal(o_p, o_q) and torch.equal(h_p, h_q)
    o_n, h_n = gdn.gdn_fwd_host(*host_inputs(x), final_state=False)
    assert h_n is None and torch.equal(o_n, o_q)
    # no initial state: the same as a zero one
    q, k, v, la, be, h0 = host_inputs(x)
    o_z, h_z = gdn.gdn_fwd_host(q, k, v, la, be, None)
    o_0, h_0 = gdn.gdn_fwd_host(q, k, v, la, be, torch.zeros_like(h0).pin_memory())
    assert torch.equal(o_z, o_0) and torch.equal(h_z, h_0)


def test_host_empty_sequence_gives_h0():
    x = synth.make_dense(2, 3, 0, 64, 64, io="bf16", h0_std=0.3, seed=1, device="cuda")
    o, hT = gdn.gdn_fwd_host(*host_inputs(x))
    assert o.numel() == 0 and torch.equal(hT, x.h0.cpu())


@pytest.mark.parametrize("slice_tokens", [64, 100, 320, 4096])
def test_host_slice_lengths_equal_device_call(slice_tokens):
    # GDN_OPT_HOST_SLICE changes only how the pipeline cuts T (rounded up to a
    # chunk multiple; at most 32 slices): the result stays bit-identical
    x = synth.make_dense(2, 2, 1000, 128, 128, io="bf16", h0_std=0.02, seed=21, device="cuda")
    prev = gdn.get_option(gdn.GDN_OPT_HOST_SLICE)
    try:
        with gdn.use_impl(gdn.GDN_IMPL_AUTO, 1):
            o_d, h_d = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
            gdn.set_option(gdn.GDN_OPT_HOST_SLICE, slice_tokens)
            o_h, h_h = gdn.gdn_fwd_host(*host_inputs(x))
    finally:
        gdn.set_option(gdn.GDN_OPT_HOST_SLICE, prev)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(h_h, h_d.cpu())
