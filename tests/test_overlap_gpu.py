"""The tensor-core forward with the chunk prep overlapped on the chain's spare
SMs (k_gdn_tc_ov), against the fp64 oracle and against the same call without
the overlap.

The prep units are computed by the same pipeline code in either launch and
the chain's arithmetic does not depend on which CTA prepared a chunk, so the
overlapped result must equal the plain one bit for bit; a missing or early
ready flag would hand the chain stale T_u / W rows (the scratch is poisoned
with NaN in these tests) and show up in both comparisons.  The lead (chunks
prepared before the chain starts) is swept from 1 (almost every chunk
prepared beside the chain, the chain waiting on its flags) to the chunk
count minus one.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gated_deltanet_recurrence_gdn_gb300 as gdn
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


class prep_lead:
    def __init__(self, lead, wide=0):
        self.lead, self.wide = lead, wide

    def __enter__(self):
        self.prev = (gdn.get_option(gdn.GDN_OPT_PREP_LEAD), gdn.get_option(gdn.GDN_OPT_WIDE_CHAIN))
        gdn.set_option(gdn.GDN_OPT_PREP_LEAD, self.lead)
        gdn.set_option(gdn.GDN_OPT_WIDE_CHAIN, self.wide)

    def __exit__(self, *exc):
        gdn.set_option(gdn.GDN_OPT_PREP_LEAD, self.prev[0])
        gdn.set_option(gdn.GDN_OPT_WIDE_CHAIN, self.prev[1])


def _run(x, lead, wide=0):
    with gdn.use_impl(gdn.GDN_IMPL_TC, 1), prep_lead(lead, wide):
        o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
        assert gdn.last_impl() == gdn.GDN_IMPL_TC
    U.sync()
    return o, hT


def _steep(la, starts):
    la = la.clone()
    for s0, val in starts:
        la[..., s0:s0 + 64] = val
    return la


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (128, 256)])
@pytest.mark.parametrize("lead", [1, 4, 10])
def test_overlap_matches_oracle_and_plain(dk, dv, lead):
    # 11 chunks (the last one ragged); steep chunks take the chain's wide-span branch
    x = synth.make_dense(2, 3, 10 * 64 + 17, dk, dv, io="bf16", h0_std=0.1, seed=601 + dk + dv,
                         device="cuda")
    x = dataclasses.replace(x, log_alpha=_steep(x.log_alpha, [(128, -3.0), (448, -1.3)]))
    o, hT = _run(x, lead)
    o_ref, h_ref = U.oracle_dense(x)
    to, th = U.TOL["bf16"]
    eo = U.rel(U.f64(o), o_ref.reshape(o.shape))
    eh = U.rel(U.f64(hT), h_ref.reshape(hT.shape))
    assert eo <= to and eh <= th, (eo, eh)
    assert np.isfinite(U.f64(o)).all()
    o1, h1 = _run(x, -1)
    assert torch.equal(o, o1) and torch.equal(hT, h1)


@pytest.mark.parametrize("B,H,T,dk,dv", [(3, 5, 2000, 128, 128), (1, 2, 700, 64, 192)])
def test_overlap_automatic_lead_small(B, H, T, dk, dv):
    # the automatic lead on batches whose chain CTAs leave most SMs to the
    # prep (ragged last chunk, h0), against the oracle and the plain path
    x = synth.make_dense(B, H, T, dk, dv, io="bf16", h0_std=0.1, seed=621 + T, device="cuda")
    o, hT = _run(x, 0)
    o_ref, h_ref = U.oracle_dense(x)
    to, th = U.TOL["bf16"]
    assert U.rel(U.f64(o), o_ref.reshape(o.shape)) <= to
    assert U.rel(U.f64(hT), h_ref.reshape(hT.shape)) <= th
    o1, h1 = _run(x, -1)
    assert torch.equal(o, o1) and torch.equal(hT, h1)


def test_overlap_repeatable():
    # the chain waits on flags for 15 of 16 chunks; calls with a cold L2 or
    # another launch in between must all give the same bits
    x = synth.make_dense(4, 4, 16 * 64, 128, 128, io="bf16", h0_std=0.1, seed=611,
                         device="cuda")
    o0, h0 = _run(x, 1)
    for i in range(5):
        if i % 2:
            torch.empty(256 << 20, dtype=torch.uint8, device="cuda").zero_()
        else:
            torch.randn(1 << 20, device="cuda").sum()
        o, h = _run(x, 1)
        assert torch.equal(o, o0) and torch.equal(h, h0), "call %d differs" % (i + 1)
    o1, h1 = _run(x, -1)
    assert torch.equal(o0, o1) and torch.equal(h0, h1)


def test_overlap_automatic_lead_workload():
    # B8 H8 T8192 d64 with h0 (64 chain CTAs, 88 SMs for the prep) and the
    # automatic lead: every output equals the plain path's, two heads the
    # oracle's
    x = synth.make_workload("gdn_fwd_b8_h8_t8192_d64_bf16_h0", device="cuda")
    o, hT = _run(x, 0)
    o1, h1 = _run(x, -1)
    assert torch.equal(o, o1) and torch.equal(hT, h1)
    heads = [(0, 0), (7, 7)]
    o_ref, h_ref = U.oracle_dense_heads_gpu(x, heads)
    for i, (b, h) in enumerate(heads):
        assert U.rel(U.f64(o[b, h]), o_ref[i]) <= U.TOL["bf16"][0]
        assert U.rel(U.f64(hT[b, h]), h_ref[i]) <= U.TOL["bf16"][1]


# The chunk loop with both d_v halves in one CTA (GDN_OPT_WIDE_CHAIN): the
# same products as N = 128 MMAs, the same register arithmetic.
@pytest.mark.parametrize("dk", [128, 64])
@pytest.mark.parametrize("lead", [1, 4, 10, 0])
def test_wide_chain_matches_oracle(dk, lead):
    x = synth.make_dense(2, 3, 10 * 64 + 17, dk, 128, io="bf16", h0_std=0.1, seed=631 + dk,
                         device="cuda")
    x = dataclasses.replace(x, log_alpha=_steep(x.log_alpha, [(128, -3.0), (448, -1.3)]))
    o, hT = _run(x, lead, wide=1)
    o_ref, h_ref = U.oracle_dense(x)
    to, th = U.TOL["bf16"]
    eo = U.rel(U.f64(o), o_ref.reshape(o.shape))
    eh = U.rel(U.f64(hT), h_ref.reshape(hT.shape))
    assert eo <= to and eh <= th, (eo, eh)
    assert np.isfinite(U.f64(o)).all()
    # the plain path's products are N = 64 MMAs over the same operands
    o1, h1 = _run(x, -1)
    assert U.rel(U.f64(o), U.f64(o1)) <= 1e-3 and U.rel(U.f64(hT), U.f64(h1)) <= 1e-3


def test_wide_chain_repeatable_and_workload():
    # B4 H16 T4096 d128 (64 chain CTAs, 88 prep SMs): repeated calls with a
    # cold L2 or another launch between them give the same bits; two heads
    # against the oracle
    x = synth.make_workload("gdn_fwd_b4_h16_t4096_d128_bf16", device="cuda")
    o0, h0 = _run(x, 0, wide=1)
    for i in range(4):
        if i % 2:
            torch.empty(256 << 20, dtype=torch.uint8, device="cuda").zero_()
        else:
            torch.randn(1 << 20, device="cuda").sum()
        o, h = _run(x, 0, wide=1)
        assert torch.equal(o, o0) and torch.equal(h, h0), "call %d differs" % (i + 1)
    heads = [(0, 0), (3, 15)]
    o_ref, h_ref = U.oracle_dense_heads_gpu(x, heads)
    for i, (b, h) in enumerate(heads):
        assert U.rel(U.f64(o0[b, h]), o_ref[i]) <= U.TOL["bf16"][0]
        assert U.rel(U.f64(h0[b, h]), h_ref[i]) <= U.TOL["bf16"][1]


@pytest.mark.parametrize("B,H,T,dk,wide", [(8, 20, 200, 128, 0), (8, 20, 200, 64, 1),
                                           (5, 16, 700, 128, 0)])
def test_wide_chain_plain_and_automatic(B, H, T, dk, wide):
    # the wide loop as a launch of its own (B H >= the SMs of a GB300, or forced)
    # and where the automatic choice takes it (more two-CTA chains than SMs):
    # the oracle's result, and the 64-column loop's bits
    x = synth.make_dense(B, H, T, dk, 128, io="bf16", h0_std=0.1, seed=641 + B * H + T,
                         device="cuda")
    o, hT = _run(x, 0, wide=wide)
    o_ref, h_ref = U.oracle_dense(x)
    to, th = U.TOL["bf16"]
    assert U.rel(U.f64(o), o_ref.reshape(o.shape)) <= to
    assert U.rel(U.f64(hT), h_ref.reshape(hT.shape)) <= th
    o1, h1 = _run(x, -1, wide=-1)
    assert U.rel(U.f64(o), U.f64(o1)) <= 1e-3 and U.rel(U.f64(hT), U.f64(h1)) <= 1e-3


@pytest.mark.parametrize("lengths", [[300, 1, 64, 200, 0, 129, 700],
                                     [129, 64, 129, 0, 64, 700, 0, 1]])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 256)])
def test_wide_chain_packed_batch(dk, dv, lengths):
    # packed sequences (chunk tails that the next sequence's rows would fill,
    # empty ones, h0; the wide loop runs them longest first, the second list
    # with ties in length): the wide loop forced, against the oracle and the
    # 64-column loop
    y = synth.make_varlen(lengths, 3, dk, dv, io="bf16", h0_std=0.1,
                          seed=651 + dk + dv + len(lengths), device="cuda")
    y = dataclasses.replace(y, log_alpha=_steep(y.log_alpha, [(64, -3.0), (365, -1.3)]))

    def run(wide):
        with gdn.use_impl(gdn.GDN_IMPL_TC, 1), prep_lead(0, wide):
            o, hT = gdn.gdn_fwd_varlen(y.q, y.k, y.v, y.log_alpha, y.beta, y.cu_seqlens, y.h0,
                                       check=True)
        U.sync()
        return o, hT

    o, hT = run(1)
    import oracle
    o_ref, h_ref = oracle.gdn_fwd_varlen(U.f64(y.q), U.f64(y.k), U.f64(y.v),
                                         U.f64(y.log_alpha), U.f64(y.beta),
                                         y.cu_seqlens.cpu().numpy(), U.f64(y.h0))
    to, th = U.TOL["bf16"]
    assert U.rel(U.f64(o), o_ref) <= to
    assert U.rel(U.f64(hT), h_ref) <= th
    o1, h1 = run(-1)
    assert U.rel(U.f64(o), U.f64(o1)) <= 1e-3 and U.rel(U.f64(hT), U.f64(h1)) <= 1e-3


def test_wide_chain_dv256_dense():
    x = synth.make_dense(2, 3, 5 * 64 + 9, 128, 256, io="bf16", h0_std=0.1, seed=661,
                         device="cuda")
    o, hT = _run(x, 0, wide=1)
    o_ref, h_ref = U.oracle_dense(x)
    to, th = U.TOL["bf16"]
    assert U.rel(U.f64(o), o_ref.reshape(o.shape)) <= to
    assert U.rel(U.f64(hT), h_ref.reshape(hT.shape)) <= th
    o1, h1 = _run(x, -1, wide=-1)
    assert U.rel(U.f64(o), U.f64(o1)) <= 1e-3 and U.rel(U.f64(hT), U.f64(h1)) <= 1e-3


@pytest.mark.parametrize("B,H,T,dk,dv,kernel", [
    (4, 16, 4096, 128, 128, "k_gdn_tc"),       # 128 two-CTA chains, 24 spare SMs: no overlap
    (8, 8, 8192, 64, 64, "k_gdn_tc_ov"),       # 64 chains, prep beside them on 88 SMs
    (8, 16, 4096, 128, 128, "k_gdn_tcw_ov"),   # 256 two-CTA chains > SMs: 128 wide ones + prep
    (8, 20, 256, 128, 128, "k_gdn_tcw"),       # 160 wide chains >= SMs: the wide loop alone
])
def test_automatic_path_on_gb300(B, H, T, dk, dv, kernel):
    # the forward's automatic choice of chunk loop, read from the kernel the
    # library times for the call; the thresholds follow the SM count, so the
    # cases are set for GB300's 152
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("cases set for a 152-SM GB300")
    x = synth.make_dense(B, H, T, dk, dv, io="bf16", seed=671, device="cuda")
    gdn.kernel_timer(True)
    gdn.kernel_timer_read()
    try:
        _run(x, 0)
        _, n, name = gdn.kernel_timer_read()
    finally:
        gdn.kernel_timer(False)
    assert n == 1 and name == kernel, (n, name)


@pytest.mark.parametrize("segments", [2, 3, 5])
@pytest.mark.parametrize("dv", [128, 256])
def test_wide_segment_scan(segments, dv):
    # the segment scan with the wide chunk loop (maps from zero and from the
    # identity, one CTA each, then every segment from its folded state):
    # against the oracle and the scan with the 64-column loop
    x = synth.make_dense(2, 2, 9 * 64 + 13, 128, dv, io="bf16", h0_std=0.05,
                         seed=681 + segments + dv, device="cuda")
    x = dataclasses.replace(x, log_alpha=_steep(x.log_alpha, [(192, -3.0), (320, -1.3)]))

    def run(wide):
        with gdn.use_impl(gdn.GDN_IMPL_TC, segments), prep_lead(0, wide):
            o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
        U.sync()
        return o, hT

    o, hT = run(1)
    o_ref, h_ref = U.oracle_dense(x)
    to, th = U.TOL["bf16"]
    assert U.rel(U.f64(o), o_ref.reshape(o.shape)) <= to
    assert U.rel(U.f64(hT), h_ref.reshape(hT.shape)) <= th
    o1, h1 = run(0)
    assert U.rel(U.f64(o), U.f64(o1)) <= 1e-3 and U.rel(U.f64(hT), U.f64(h1)) <= 1e-3


@pytest.mark.parametrize("segments", [0, 10])
def test_wide_segment_scan_first_segment_in_full(segments):
    # 16 heads x 257 chunks (the last ragged): on a 152-SM device the plan
    # runs segment 0 in full (from h0, with outputs) beside the maps of
    # segments 1 .. S - 2, then segments 1 .. S - 1 from their folded states;
    # against the oracle on three heads and the unsegmented wide loop on all
    x = synth.make_dense(1, 16, 256 * 64 + 29, 128, 128, io="bf16", h0_std=0.05,
                         seed=697 + segments, device="cuda")
    x = dataclasses.replace(x, log_alpha=_steep(x.log_alpha, [(1024, -3.0), (9000, -1.3)]))
    with gdn.use_impl(gdn.GDN_IMPL_TC, segments), prep_lead(0, 1 if segments else 0):
        o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
    U.sync()
    heads = [(0, 0), (0, 7), (0, 15)]
    o_ref, h_ref = U.oracle_dense_heads_gpu(x, heads)
    to, th = U.TOL["bf16"]
    for i, (b, h) in enumerate(heads):
        assert U.rel(U.f64(o[b, h]), o_ref[i]) <= to
        assert U.rel(U.f64(hT[b, h]), h_ref[i]) <= th
    with gdn.use_impl(gdn.GDN_IMPL_TC, 1), prep_lead(0, 1):
        o1, h1 = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
    U.sync()
    assert U.rel(U.f64(o), U.f64(o1)) <= 1e-3 and U.rel(U.f64(hT), U.f64(h1)) <= 1e-3
