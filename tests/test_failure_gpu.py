"""Failure detection on the device without a fault: the bounded waits that
the pipelined kernels hand work through give up after their poll limit,
record a timeout that the host reads (GDN_ERR_DEVICE_TIMEOUT), and leave the
context usable.  The failure is an mbarrier phase and a counter that nothing
completes; no kernel traps, faults or spins without a bound."""
import pytest

import gated_deltanet_recurrence_gdn_gb300 as gdn
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _status():
    return gdn.load().gdn_sync_check(gdn._stream(None))


def test_completed_waits_succeed_without_error():
    _status()                                     # clear anything left over
    assert gdn.selftest_wait(True, 1000) == (True, True)
    assert _status() == gdn.GDN_OK


def test_wait_nothing_completes_times_out_and_context_survives():
    _status()
    assert gdn.selftest_wait(False, 64) == (False, False)
    assert _status() == gdn.GDN_ERR_DEVICE_TIMEOUT
    assert _status() == gdn.GDN_OK                # the word is cleared once read
    # the context still works: a forward pass right after matches the oracle
    x = synth.make_dense(1, 2, 130, 64, 64, io="bf16", h0_std=0.02, seed=5, device="cuda")
    o, hT = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
    U.sync()
    o_ref, h_ref = U.oracle_dense(x)
    assert U.rel(U.f64(o), o_ref) <= 1e-2
    assert U.rel(U.f64(hT), h_ref) <= 2e-2
