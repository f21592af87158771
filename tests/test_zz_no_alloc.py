"""gdn_fwd_noalloc: the forward pass for callers that cannot allocate.

Some users cannot let a library allocate device memory while they run: a
serving process that gives all of the GPU's memory to its own pool at start-up
and forbids other allocations, or a latency-critical loop in which an
allocation that stalls or fails is not acceptable.  gdn_fwd_noalloc keeps its
scratch in a fixed 32 MiB device array instead.

These tests call it through the C ABI and compare every output element with
the fp64 oracle, for bf16 and fp32 I/O, on two calls in a row: the first call
on a device maps the array (the driver loads the library's device code
lazily), and the second call must succeed, find the first call's data in the
shared scratch without being affected by it, and take nothing from the
library's scratch pool.  The file is collected last and passes both alone in
a fresh process and after the other tests.
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


def _run_and_check(lib, x, io):
    B, H, T, dk = x.q.shape
    dv = x.v.shape[-1]
    o = torch.full_like(x.v, float("nan"))
    hT = torch.full((B, H, dv, dk), float("nan"), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, x, o, hT) == gdn.GDN_OK
    assert lib.gdn_sync_check(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == gdn.GDN_OK
    torch.cuda.synchronize()
    o_ref, h_ref = U.oracle_dense(x)
    to, th = U.TOL[io]
    eo = U.rel(U.f64(o), o_ref.reshape(o.shape))
    eh = U.rel(U.f64(hT), h_ref.reshape(hT.shape))
    assert eo <= to and eh <= th, (io, eo, eh)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_noalloc_two_calls_match_oracle(io):
    lib = gdn.load()
    first = synth.make_dense(2, 3, 200, 128, 128, io=io, h0_std=0.02, seed=31, device="cuda")
    second = synth.make_dense(1, 4, 3 * 64 + 5, 64, 64, io=io, h0_std=0.0, seed=32,
                              device="cuda")
    # first call on this device: maps the fixed array if nothing has yet
    _run_and_check(lib, first, io)
    # second call: must succeed and draw nothing from the scratch pool
    torch.cuda.synchronize()
    cur0, _ = gdn.scratch_stats(reset_high=True)
    _run_and_check(lib, second, io)
    cur1, high1 = gdn.scratch_stats()
    assert high1 <= cur0 and cur1 <= cur0, (cur0, cur1, high1)


def test_noalloc_rejects_calls_beyond_its_scratch():
    lib = gdn.load()
    # 1 x 16 x 4096 tokens at d_k = d_v = 128 needs ~67 MB of scratch > 32 MiB
    x = synth.make_dense(1, 16, 4096, 128, 128, io="bf16", seed=3, device="cuda")
    o = torch.empty_like(x.v)
    hT = torch.empty((1, 16, 128, 128), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, x, o, hT) == gdn.GDN_ERR_TOO_LARGE
    assert b"32 MiB" in lib.gdn_status_string(gdn.GDN_ERR_TOO_LARGE)
