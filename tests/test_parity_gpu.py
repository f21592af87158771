"""CUDA path vs the fp64 oracle, element by element, on the same seeded inputs.

Small cases span several 64-token chunks and a ragged tail; the workload
cases run at full size in the launch configuration the benchmark times and
compare either every output (when the oracle finishes in seconds) or a
sampled subset of heads / sequences / a causal prefix.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gated_deltanet_recurrence_gdn_gb300 as gdn
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

IMPLS = {"simt": gdn.GDN_IMPL_SIMT, "tc": gdn.GDN_IMPL_TC, "fused": gdn.GDN_IMPL_TC_FUSED,
         "auto": gdn.GDN_IMPL_AUTO}


def run_dense(x, impl, **kw):
    with gdn.use_impl(IMPLS[impl], kw.pop("segments", None)):
        try:
            o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True, **kw)
        except gdn.GdnError as e:
            if e.status == gdn.GDN_ERR_UNSUPPORTED and impl in ("tc", "fused"):
                pytest.skip("shape not covered by the tensor-core path")
            raise
        used = gdn.last_impl()
    if impl != "auto":
        assert used == IMPLS[impl]
    U.sync()
    return o, hT


def run_varlen(y, impl, **kw):
    with gdn.use_impl(IMPLS[impl], kw.pop("segments", None)):
        try:
            o, hT = gdn.gdn_fwd_varlen(y.q, y.k, y.v, y.log_alpha, y.beta, y.cu_seqlens, y.h0,
                                       check=True, **kw)
        except gdn.GdnError as e:
            if e.status == gdn.GDN_ERR_UNSUPPORTED and impl in ("tc", "fused"):
                pytest.skip("shape not covered by the tensor-core path")
            raise
    U.sync()
    return o, hT


def check(o, hT, o_ref, h_ref, io):
    to, th = U.TOL[io]
    eo, eh = U.rel(U.f64(o), o_ref), U.rel(U.f64(hT), h_ref)
    assert eo <= to and eh <= th, (eo, eh)
    assert np.isfinite(U.f64(o)).all()
    return eo, eh


DENSE_CASES = [
    # B, H, T, dk, dv, io, h0_std, decay
    (1, 1, 1, 64, 64, "f32", 0.02, "fast"),
    (2, 3, 63, 64, 64, "bf16", 0.02, "fast"),
    (2, 2, 64, 128, 128, "bf16", 0.0, "fast"),
    (1, 3, 65, 128, 128, "bf16", 0.5, "slow"),
    (2, 2, 3 * 64 + 17, 128, 128, "bf16", 0.02, "fast"),
    (2, 2, 3 * 64 + 17, 128, 128, "f32", 0.02, "fast"),
    (1, 2, 5 * 64 + 3, 64, 64, "bf16", 0.02, "slow"),
    (1, 2, 2 * 64 + 40, 128, 256, "bf16", 0.02, "fast"),
    (1, 2, 2 * 64 + 40, 64, 128, "bf16", 0.0, "fast"),
    (1, 1, 130, 32, 48, "f32", 0.1, "fast"),
    (1, 2, 4 * 64, 128, 64, "bf16", 0.02, "none"),
]


@pytest.mark.parametrize("impl", ["simt", "tc", "fused"])
@pytest.mark.parametrize("case", DENSE_CASES, ids=lambda c: "b%dh%dt%d_k%dv%d_%s_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[7]))
def test_dense_small(impl, case):
    B, H, T, dk, dv, io, h0s, decay = case
    x = synth.make_dense(B, H, T, dk, dv, io=io, h0_std=h0s, decay=decay, seed=100 + T,
                         device="cuda")
    o, hT = run_dense(x, impl)
    o_ref, h_ref = U.oracle_dense(x)
    check(o, hT, o_ref.reshape(o.shape), h_ref.reshape(hT.shape), io)


VARLEN_CASES = [
    ([70, 0, 5, 130, 64], 2, 64, 64, "f32"),
    ([1, 63, 64, 65, 200, 0], 3, 128, 128, "bf16"),
    ([300, 17, 128], 2, 128, 256, "bf16"),
    ([0, 0], 1, 64, 64, "bf16"),
]


@pytest.mark.parametrize("impl", ["simt", "tc", "fused"])
@pytest.mark.parametrize("case", VARLEN_CASES, ids=lambda c: "n%d_k%dv%d_%s" % (
    len(c[0]), c[2], c[3], c[4]))
def test_varlen_small(impl, case):
    lens, H, dk, dv, io = case
    y = synth.make_varlen(lens, H, dk, dv, io=io, h0_std=0.02, seed=200 + len(lens),
                          device="cuda")
    o, hT = run_varlen(y, impl)
    import oracle
    o_ref, h_ref = oracle.gdn_fwd_varlen(U.f64(y.q), U.f64(y.k), U.f64(y.v),
                                         U.f64(y.log_alpha), U.f64(y.beta),
                                         y.cu_seqlens.cpu().numpy(), U.f64(y.h0))
    check(o, hT, o_ref, h_ref, io)


@pytest.mark.parametrize("impl", ["simt", "tc", "fused"])
def test_varlen_equals_dense(impl):
    # equal lengths: the packed call must reproduce the dense call bit for bit
    # up to the different memory layout
    B, H, T, dk, dv = 3, 2, 150, 128, 128
    x = synth.make_dense(B, H, T, dk, dv, io="bf16", h0_std=0.02, seed=5, device="cuda")
    od, hd = run_dense(x, impl)
    pack = lambda t: t.permute(1, 0, 2, 3).reshape(H, B * T, t.shape[-1]).contiguous()  # noqa
    packg = lambda t: t.permute(1, 0, 2).reshape(H, B * T).contiguous()  # noqa
    cu = torch.arange(0, B * T + 1, T, dtype=torch.int32, device="cuda")
    y = synth.Inputs(pack(x.q), pack(x.k), pack(x.v), packg(x.log_alpha), packg(x.beta), x.h0,
                     cu)
    ov, hv = run_varlen(y, impl)
    assert torch.equal(ov, pack(od)) and torch.equal(hv, hd)


@pytest.mark.parametrize("impl", ["simt", "tc", "fused"])
def test_continuation(impl):
    B, H, T1, T2, dk, dv = 1, 4, 192, 137, 128, 128
    x = synth.make_dense(B, H, T1 + T2, dk, dv, io="bf16", h0_std=0.02, seed=9, device="cuda")
    o, hT = run_dense(x, impl)
    s1, s2 = np.s_[:, :, :T1], np.s_[:, :, T1:]
    part = lambda s, h0: synth.Inputs(*(t[s].contiguous() for t in (x.q, x.k, x.v,  # noqa
                                                                  x.log_alpha, x.beta)), h0)
    o1, h1 = run_dense(part(s1, x.h0), impl)
    o2, h2 = run_dense(part(s2, h1), impl)
    o12 = torch.cat([o1, o2], dim=2)
    assert U.rel(U.f64(o12), U.f64(o)) <= 1e-2
    assert U.rel(U.f64(h2), U.f64(hT)) <= 2e-2


@pytest.mark.parametrize("impl", ["simt", "tc"])
def test_empty_sequence_gives_h0(impl):
    x = synth.make_dense(2, 3, 0, 64, 64, io="bf16", h0_std=0.3, seed=1, device="cuda")
    o, hT = run_dense(x, impl)
    assert o.numel() == 0 and torch.equal(hT, x.h0)


@pytest.mark.parametrize("impl", ["simt", "tc", "fused"])
def test_scratch_pool_release_and_reuse(impl):
    # scratch comes from the library's own pool: results do not depend on
    # whether the pool was just emptied or still holds the previous call's
    # blocks
    x = synth.make_dense(2, 2, 333, 128, 128, io="bf16", h0_std=0.02, seed=21, device="cuda")
    o1, h1 = run_dense(x, impl)
    gdn.release_scratch()
    o2, h2 = run_dense(x, impl)
    o3, h3 = run_dense(x, impl)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    assert torch.equal(o1, o3) and torch.equal(h1, h3)


# ------------------------------------------------------------ steep decay
#
# Where a chunk's total log decay g_C is below -80, exp(-g_s) could overflow:
# the chunk-prep kernels then form A with one exponential per entry, and the
# chunk loop scales Q by gamma in place and forms P exactly.  The synthetic
# gates never reach that (about -25 per chunk), so these cases set log gates
# of -3 per step (g_C about -190) and -1.3 (about -83, just past the switch)
# in some chunks and keep the synthetic ones elsewhere.


def _steep(la, T):
    la = la.clone()
    la[..., 64:min(T, 128)] = -3.0
    if T > 128:
        la[..., 128:min(T, 192)] = -1.3
    if T > 192:
        la[..., 192:min(T, 256)] = -3.0
    return la


@pytest.mark.parametrize("impl", ["simt", "tc", "fused"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (128, 256)])
def test_steep_decay_matches_oracle(impl, dk, dv):
    x = synth.make_dense(1, 2, 4 * 64 + 9, dk, dv, io="bf16", h0_std=0.1, seed=91 + dk + dv,
                         device="cuda")
    x = dataclasses.replace(x, log_alpha=_steep(x.log_alpha, x.log_alpha.shape[-1]))
    o, hT = run_dense(x, impl)
    o_ref, h_ref = U.oracle_dense(x)
    check(o, hT, o_ref.reshape(o.shape), h_ref.reshape(hT.shape), "bf16")


def test_steep_decay_fp32_io_matches_oracle():
    # the general path with fp32 I/O (3xTF32 products) through the same chunks
    x = synth.make_dense(1, 2, 4 * 64 + 9, 64, 64, io="f32", h0_std=0.1, seed=95, device="cuda")
    x = dataclasses.replace(x, log_alpha=_steep(x.log_alpha, x.log_alpha.shape[-1]))
    o, hT = run_dense(x, "simt")
    o_ref, h_ref = U.oracle_dense(x)
    check(o, hT, o_ref.reshape(o.shape), h_ref.reshape(hT.shape), "f32")


@pytest.mark.parametrize("impl", ["simt", "tc"])
def test_steep_decay_no_erase_matches_oracle(impl):
    # gated linear attention (no erase term) through the same chunks
    import oracle
    x = synth.make_dense(1, 2, 4 * 64 + 9, 128, 128, io="bf16", h0_std=0.1, seed=96,
                         device="cuda")
    x = dataclasses.replace(x, log_alpha=_steep(x.log_alpha, x.log_alpha.shape[-1]))
    with gdn.use_impl(IMPLS[impl]):
        o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True, erase=False)
    U.sync()
    o_ref, h_ref = oracle.gdn_fwd(U.f64(x.q), U.f64(x.k), U.f64(x.v), U.f64(x.log_alpha),
                                  U.f64(x.beta), U.f64(x.h0), threads=U.ORACLE_THREADS,
                                  erase=False)
    check(o, hT, o_ref, h_ref, "bf16")


@pytest.mark.parametrize("impl", ["simt", "tc", "fused"])
def test_steep_decay_varlen_matches_oracle(impl):
    import oracle
    y = synth.make_varlen([300, 40, 200], 2, 128, 128, io="bf16", h0_std=0.1, seed=97,
                          device="cuda")
    # steep chunks inside the first and the third sequence
    la = y.log_alpha.clone()
    la[..., 64:128] = -3.0
    la[..., 340 + 64:340 + 128] = -1.3
    y = dataclasses.replace(y, log_alpha=la)
    o, hT = run_varlen(y, impl)
    o_ref, h_ref = oracle.gdn_fwd_varlen(U.f64(y.q), U.f64(y.k), U.f64(y.v), U.f64(y.log_alpha),
                                         U.f64(y.beta), y.cu_seqlens.cpu().numpy(),
                                         U.f64(y.h0))
    check(o, hT, o_ref, h_ref, "bf16")


# ------------------------------------------------------------ segment scan


@pytest.mark.parametrize("segments", [2, 3, 7])
@pytest.mark.parametrize("dk,dv,decay", [(128, 128, "slow"), (64, 64, "none"),
                                         (128, 256, "fast")])
def test_segment_scan(segments, dk, dv, decay):
    # the sequence is cut into segments whose affine maps are folded and then
    # rerun from their true initial states; every output and hT must match
    x = synth.make_dense(2, 2, 9 * 64 + 13, dk, dv, io="bf16", h0_std=0.05, decay=decay,
                         seed=300 + segments + dk, device="cuda")
    o, hT = run_dense(x, "tc", segments=segments)
    o_ref, h_ref = U.oracle_dense(x)
    check(o, hT, o_ref.reshape(o.shape), h_ref.reshape(hT.shape), "bf16")


def test_segment_scan_equals_single_pass():
    x = synth.make_dense(1, 3, 20 * 64, 128, 128, io="bf16", h0_std=0.05, decay="none", seed=9,
                         device="cuda")
    o1, h1 = run_dense(x, "tc", segments=1)
    o4, h4 = run_dense(x, "tc", segments=4)
    assert U.rel(U.f64(o4), U.f64(o1)) <= 1e-2
    assert U.rel(U.f64(h4), U.f64(h1)) <= 2e-2


# ----------------------------------------------------------------- workloads


def test_workload_fp32_small_full():
    x = synth.make_workload("gdn_fwd_b1_h1_t256_d64_fp32", device="cuda")
    o, hT = run_dense(x, "auto")
    o_ref, h_ref = U.oracle_dense(x)
    check(o, hT, o_ref.reshape(o.shape), h_ref.reshape(hT.shape), "f32")


@pytest.mark.parametrize("impl", ["auto", "fused", "simt"])
def test_workload_b4_h16_t4096_d128_full(impl):
    x = synth.make_workload("gdn_fwd_b4_h16_t4096_d128_bf16", device="cuda")
    o, hT = run_dense(x, impl)
    o_ref, h_ref = U.oracle_dense(x)           # every head, every token
    check(o, hT, o_ref.reshape(o.shape), h_ref.reshape(hT.shape), "bf16")


def test_fp32_io_b4_h16_t1024_d128_full():
    # the general path with fp32 I/O (three tf32 products per step) at the
    # headline batch's width over 16 chunks per head, every head and token
    x = synth.make_dense(4, 16, 1024, 128, 128, io="f32", h0_std=0.02, seed=29, device="cuda")
    o, hT = run_dense(x, "auto")
    assert gdn.load().gdn_last_impl() == gdn.GDN_IMPL_SIMT
    o_ref, h_ref = U.oracle_dense(x)
    check(o, hT, o_ref.reshape(o.shape), h_ref.reshape(hT.shape), "f32")


def test_workload_b8_h8_t8192_d64_h0_full():
    x = synth.make_workload("gdn_fwd_b8_h8_t8192_d64_bf16_h0", device="cuda")
    o, hT = run_dense(x, "auto")
    o_ref, h_ref = U.oracle_dense(x)
    check(o, hT, o_ref.reshape(o.shape), h_ref.reshape(hT.shape), "bf16")


def test_workload_b8_h16_t4096_d128_sampled():
    # the batch the forward runs with both d_v halves in one CTA (and the chunk
    # prep beside it): every output equals the 64-column loop's, four heads
    # the oracle's
    x = synth.make_workload("gdn_fwd_b8_h16_t4096_d128_bf16", device="cuda")
    o, hT = run_dense(x, "auto")
    prev = gdn.get_option(gdn.GDN_OPT_WIDE_CHAIN)
    gdn.set_option(gdn.GDN_OPT_WIDE_CHAIN, -1)
    try:
        o1, h1 = run_dense(x, "auto")
    finally:
        gdn.set_option(gdn.GDN_OPT_WIDE_CHAIN, prev)
    assert U.rel(U.f64(o), U.f64(o1)) <= 1e-3 and U.rel(U.f64(hT), U.f64(h1)) <= 1e-3
    heads = [(0, 0), (3, 7), (5, 12), (7, 15)]
    o_ref, h_ref = U.oracle_dense_heads_gpu(x, heads)
    for i, (b, h) in enumerate(heads):
        assert U.rel(U.f64(o[b, h]), o_ref[i]) <= U.TOL["bf16"][0]
        assert U.rel(U.f64(hT[b, h]), h_ref[i]) <= U.TOL["bf16"][1]


def test_workload_long_context_sampled():
    name = "gdn_fwd_b1_h16_t131072_d128_bf16"
    x = synth.make_workload(name, device="cuda")
    o, hT = run_dense(x, "auto")
    # causal prefix of every head
    P = 8192
    o_ref, _ = U.oracle_dense_prefix_gpu(x, P)
    assert U.rel(U.f64(o[:, :, :P]), o_ref) <= U.TOL["bf16"][0]
    # full length (every output and hT) of two heads
    heads = [(0, 0), (0, 11)]
    o_ref, h_ref = U.oracle_dense_heads_gpu(x, heads)
    for i, (b, h) in enumerate(heads):
        assert U.rel(U.f64(o[b, h]), o_ref[i]) <= U.TOL["bf16"][0]
        assert U.rel(U.f64(hT[b, h]), h_ref[i]) <= U.TOL["bf16"][1]


def test_workload_varlen_sampled():
    name = "gdn_fwd_varlen_n64_h32_dk128_dv256_bf16"
    y = synth.make_workload(name, device="cuda")
    o, hT = run_varlen(y, "auto")
    cu = y.cu_seqlens.cpu().numpy()
    lens = np.diff(cu)
    order = np.argsort(lens)
    pairs = [(int(order[0]), 0), (int(order[-1]), 31), (int(order[-2]), 7),
             (int(order[len(order) // 2]), 16), (5, 3), (63, 30)]
    ref = U.oracle_varlen_pairs_gpu(y, pairs)
    for (n, h), (o_ref, h_ref) in ref.items():
        a, b = int(cu[n]), int(cu[n + 1])
        assert U.rel(U.f64(o[h, a:b]), o_ref) <= U.TOL["bf16"][0], (n, h)
        assert U.rel(U.f64(hT[n, h]), h_ref) <= U.TOL["bf16"][1], (n, h)


# ------------------------------------------------------------ error handling


def test_argument_errors():
    x = synth.make_dense(1, 2, 70, 64, 64, io="bf16", seed=3, device="cuda")
    lib = gdn.load()
    s = torch.cuda.current_stream().cuda_stream
    p = lambda t: t.data_ptr()  # noqa: E731
    o = torch.empty_like(x.v)
    args = [p(x.q), p(x.k), p(x.v), p(x.log_alpha), p(x.beta), None, p(o), None]
    assert lib.gdn_fwd(*args, 1, 2, 70, 64, 64, 32, 1, s) == gdn.GDN_ERR_UNSUPPORTED
    assert lib.gdn_fwd(*args, 1, 2, 70, 100, 64, 64, 1, s) == gdn.GDN_ERR_UNSUPPORTED
    bad = list(args)
    bad[0] = p(x.q) + 2
    assert lib.gdn_fwd(*bad, 1, 2, 70, 64, 64, 64, 1, s) == gdn.GDN_ERR_ALIGNMENT
    bad = list(args)
    bad[1] = None
    assert lib.gdn_fwd(*bad, 1, 2, 70, 64, 64, 64, 1, s) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_fwd(*args, 1, 2, 70, 64, 64, 64, 7, s) == gdn.GDN_ERR_INVALID_ARG


@pytest.mark.parametrize("impl", ["simt", "tc"])
def test_bad_cu_seqlens_reported(impl):
    # a decreasing / out-of-range offset table is caught by the kernels and
    # reported on the host; nothing is read out of bounds
    y = synth.make_varlen([40, 50], 2, 64, 64, io="bf16", seed=4, device="cuda")
    bad = torch.tensor([0, 95, 90], dtype=torch.int32, device="cuda")
    with gdn.use_impl(IMPLS[impl]):
        try:
            gdn.gdn_fwd_varlen(y.q, y.k, y.v, y.log_alpha, y.beta, bad, None)
        except gdn.GdnError as e:
            if e.status == gdn.GDN_ERR_UNSUPPORTED and impl in ("tc", "fused"):
                pytest.skip("shape not covered by the tensor-core path")
            raise
    lib = gdn.load()
    assert lib.gdn_sync_check(torch.cuda.current_stream().cuda_stream) == gdn.GDN_ERR_INVALID_ARG
    # the error word is cleared by reading it
    assert lib.gdn_sync_check(torch.cuda.current_stream().cuda_stream) == gdn.GDN_OK


# ------------------------------------------------- gated linear attention


@pytest.mark.parametrize("impl", ["simt", "tc"])
@pytest.mark.parametrize("B,H,T,dk,dv,io", [(2, 2, 300, 128, 128, "bf16"),
                                            (1, 3, 200, 64, 64, "bf16"),
                                            (2, 1, 150, 64, 64, "f32")])
def test_no_erase_matches_oracle(impl, B, H, T, dk, dv, io):
    # the recurrence without the erase term (gated linear attention)
    x = synth.make_dense(B, H, T, dk, dv, io=io, h0_std=0.02, seed=T + 3, device="cuda")
    with gdn.use_impl(IMPLS[impl]):
        try:
            o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True, erase=False)
        except gdn.GdnError as e:
            if e.status == gdn.GDN_ERR_UNSUPPORTED and impl in ("tc", "fused"):
                pytest.skip("shape not covered by the tensor-core path")
            raise
    U.sync()
    import oracle
    o_ref, h_ref = oracle.gdn_fwd(U.f64(x.q), U.f64(x.k), U.f64(x.v), U.f64(x.log_alpha),
                                  U.f64(x.beta), U.f64(x.h0), threads=U.ORACLE_THREADS,
                                  erase=False)
    check(o, hT, o_ref, h_ref, io)


@pytest.mark.parametrize("impl", ["simt", "tc"])
def test_no_erase_varlen_matches_oracle(impl):
    y = synth.make_varlen([1, 63, 64, 65, 200, 0, 129], 2, 128, 128, io="bf16", h0_std=0.02,
                          seed=17, device="cuda")
    with gdn.use_impl(IMPLS[impl]):
        o, hT = gdn.gdn_fwd_varlen(y.q, y.k, y.v, y.log_alpha, y.beta, y.cu_seqlens, y.h0,
                                   check=True, erase=False)
    U.sync()
    import oracle
    o_ref, h_ref = oracle.gdn_fwd_varlen(U.f64(y.q), U.f64(y.k), U.f64(y.v),
                                         U.f64(y.log_alpha), U.f64(y.beta),
                                         y.cu_seqlens.cpu().numpy(), U.f64(y.h0),
                                         erase=False)
    check(o, hT, o_ref, h_ref, "bf16")


@pytest.mark.parametrize("impl", ["simt", "tc"])
def test_no_erase_plain_linear_attention(impl):
    # alpha = beta = 1, no initial state: causally masked (Q K^T) V
    B, H, T, d = 1, 2, 192, 64
    x = synth.make_dense(B, H, T, d, d, io="bf16", seed=19, device="cuda")
    la = torch.zeros_like(x.log_alpha)
    be = torch.ones_like(x.beta)
    with gdn.use_impl(IMPLS[impl]):
        o, _ = gdn.gdn_fwd(x.q, x.k, x.v, la, be, None, check=True, erase=False)
    U.sync()
    qf, kf, vf = (t.double() for t in (x.q, x.k, x.v))
    mask = torch.tril(torch.ones(T, T, dtype=torch.float64, device="cuda"))
    ref = ((qf @ kf.transpose(-1, -2)) * mask) @ vf
    assert U.rel(U.f64(o), U.f64(ref)) <= 1e-2


# ------------------------------------------------- a forget gate per key dimension


@pytest.mark.parametrize("erase", [True, False])
@pytest.mark.parametrize("B,H,T,dk,dv,io", [(2, 2, 300, 128, 128, "bf16"),
                                            (1, 3, 200, 64, 64, "bf16"),
                                            (2, 1, 150, 32, 48, "f32")])
def test_vector_gate_matches_oracle(erase, B, H, T, dk, dv, io):
    x = synth.make_dense(B, H, T, dk, dv, io=io, h0_std=0.02, seed=T + 5, device="cuda",
                         vector_gate=True)
    assert x.log_alpha.shape == (B, H, T, dk)
    with gdn.use_impl(gdn.GDN_IMPL_AUTO):
        o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True, erase=erase)
    assert gdn.load().gdn_last_impl() == gdn.GDN_IMPL_SIMT
    U.sync()
    import oracle
    o_ref, h_ref = oracle.gdn_fwd(U.f64(x.q), U.f64(x.k), U.f64(x.v), U.f64(x.log_alpha),
                                  U.f64(x.beta), U.f64(x.h0), threads=U.ORACLE_THREADS,
                                  erase=erase, vector_gate=True)
    check(o, hT, o_ref, h_ref, io)


@pytest.mark.parametrize("erase", [True, False])
def test_vector_gate_varlen_matches_oracle(erase):
    y = synth.make_varlen([1, 63, 64, 65, 200, 0, 129], 2, 128, 128, io="bf16", h0_std=0.02,
                          seed=23, device="cuda", vector_gate=True)
    o, hT = gdn.gdn_fwd_varlen(y.q, y.k, y.v, y.log_alpha, y.beta, y.cu_seqlens, y.h0,
                               check=True, erase=erase)
    U.sync()
    import oracle
    o_ref, h_ref = oracle.gdn_fwd_varlen(U.f64(y.q), U.f64(y.k), U.f64(y.v),
                                         U.f64(y.log_alpha), U.f64(y.beta),
                                         y.cu_seqlens.cpu().numpy(), U.f64(y.h0),
                                         erase=erase, vector_gate=True)
    check(o, hT, o_ref, h_ref, "bf16")


def test_vector_gate_uniform_rows_equal_scalar_gate():
    # a per-dimension gate whose d_k entries are all equal is the scalar gate:
    # the vector-gate kernels must agree with the tensor-core scalar path
    x = synth.make_dense(2, 2, 300, 128, 128, io="bf16", h0_std=0.02, seed=41, device="cuda")
    la_vec = x.log_alpha[..., None].expand(-1, -1, -1, 128).contiguous()
    with gdn.use_impl(gdn.GDN_IMPL_TC):
        o_s, h_s = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
    o_v, h_v = gdn.gdn_fwd(x.q, x.k, x.v, la_vec, x.beta, x.h0, check=True)
    U.sync()
    assert U.rel(U.f64(o_v), U.f64(o_s)) <= 1e-2
    assert U.rel(U.f64(h_v), U.f64(h_s)) <= 2e-2


def test_vector_gate_not_on_tensor_core_path():
    x = synth.make_dense(1, 1, 128, 128, 128, io="bf16", seed=43, device="cuda",
                         vector_gate=True)
    with gdn.use_impl(gdn.GDN_IMPL_TC):
        with pytest.raises(gdn.GdnError) as e:
            gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, None)
    assert e.value.status == gdn.GDN_ERR_UNSUPPORTED


@pytest.mark.parametrize("B,H,T,dk,dv,io,decay", [(1, 2, 200, 128, 256, "bf16", "fast"),
                                                  (2, 2, 150, 64, 64, "f32", "slow"),
                                                  (1, 3, 130, 128, 128, "f32", "fast")])
def test_vector_gate_wide_and_fp32(B, H, T, dk, dv, io, decay):
    # the widest tiles (d_v = 256) and fp32 I/O (three tf32 products per step)
    x = synth.make_dense(B, H, T, dk, dv, io=io, decay=decay, h0_std=0.05, seed=T + 7,
                         device="cuda", vector_gate=True)
    o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
    U.sync()
    import oracle
    o_ref, h_ref = oracle.gdn_fwd(U.f64(x.q), U.f64(x.k), U.f64(x.v), U.f64(x.log_alpha),
                                  U.f64(x.beta), U.f64(x.h0), threads=U.ORACLE_THREADS,
                                  vector_gate=True)
    check(o, hT, o_ref, h_ref, io)


def test_vector_gate_steep_decay_stays_finite():
    # log gates of -20 per step in some dimensions: exp(G_r - G_s) spans far
    # below fp32's range inside one chunk; the factored products must neither
    # overflow nor lose the near-diagonal terms
    x = synth.make_dense(1, 2, 192, 64, 64, io="f32", seed=37, device="cuda", vector_gate=True)
    la = x.log_alpha.clone()
    la[..., ::3] = -20.0
    o, hT = gdn.gdn_fwd(x.q, x.k, x.v, la, x.beta, None, check=True)
    U.sync()
    assert torch.isfinite(o).all() and torch.isfinite(hT).all()
    import oracle
    o_ref, h_ref = oracle.gdn_fwd(U.f64(x.q), U.f64(x.k), U.f64(x.v), U.f64(la), U.f64(x.beta),
                                  None, vector_gate=True)
    check(o, hT, o_ref, h_ref, "f32")
