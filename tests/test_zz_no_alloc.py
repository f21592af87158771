"""gdn_fwd_noalloc: the forward pass for callers that cannot allocate.

Some users cannot let a library allocate device memory while they run: a
serving process that gives all of the GPU's memory to its own pool at start-up
and forbids other allocations, or a latency-critical loop in which an
allocation that stalls or fails is not acceptable.  gdn_fwd_noalloc keeps its
scratch in a fixed 32 MiB device array instead.  This test calls it through
the C ABI and checks it against gdn_fwd, the allocating entry point, on two
calls in a row (the second call finds the first call's data in the shared
scratch and must not be affected by it).  It lives in its own file, collected
last, and passes both alone in a fresh process and after the other tests.
"""
import ctypes

import pytest
import torch

import gated_deltanet_recurrence_gdn_gb300 as gdn
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, x, o, hT):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    B, H, T, dk = x.q.shape
    dv = x.v.shape[-1]
    dt = gdn.GDN_BF16 if x.q.dtype == torch.bfloat16 else gdn.GDN_F32
    return lib.gdn_fwd_noalloc(p(x.q), p(x.k), p(x.v), p(x.log_alpha), p(x.beta), p(x.h0),
                               p(o), p(hT), B, H, T, dk, dv, 64, dt,
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_gdn_fwd_on_two_calls():
    lib = gdn.load()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(2, 3, 200, 128, 128, 0.02, 31), (1, 4, 3 * 64 + 5, 64, 64, 0.0, 32)]
    for B, H, T, dk, dv, h0s, seed in cases:
        x = synth.make_dense(B, H, T, dk, dv, io="bf16", h0_std=h0s, seed=seed, device="cuda")
        o_ref, h_ref = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
        o = torch.full_like(o_ref, float("nan"))
        hT = torch.full_like(h_ref, float("nan"))
        assert _call_noalloc(lib, x, o, hT) == gdn.GDN_OK
        assert lib.gdn_sync_check(stream) == gdn.GDN_OK
        torch.cuda.synchronize()
        eo = U.rel(U.f64(o), U.f64(o_ref))
        eh = U.rel(U.f64(hT), U.f64(h_ref))
        assert eo <= U.TOL["bf16"][0] and eh <= U.TOL["bf16"][1], (eo, eh)


def test_noalloc_rejects_calls_beyond_its_scratch():
    lib = gdn.load()
    # 1 x 16 x 4096 tokens at d_k = d_v = 128 needs ~67 MB of scratch > 32 MiB
    x = synth.make_dense(1, 16, 4096, 128, 128, io="bf16", seed=3, device="cuda")
    o = torch.empty_like(x.v)
    hT = torch.empty((1, 16, 128, 128), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, x, o, hT) == gdn.GDN_ERR_TOO_LARGE
    assert b"32 MiB" in lib.gdn_status_string(gdn.GDN_ERR_TOO_LARGE)
