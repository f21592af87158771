"""Parity of the decode step (gdn_decode) with the fp64 oracle.

One decode step is the recurrence for a single token
("Gated DeltaNet GPU并行实现", sections 2.1-2.2), so the oracle is its
token-by-token loop run with T = 1 and h0 = the state."""
from __future__ import annotations

import pytest
import torch

import gated_deltanet_recurrence_gdn_gb300 as gdn
import oracle
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def oracle_step(x, state):
    q, k, v, la, be = (U.f64(t)[:, :, None] for t in (x.q, x.k, x.v, x.log_alpha, x.beta))
    o, hT = oracle.gdn_fwd(q, k, v, la, be, state, threads=U.ORACLE_THREADS)
    return o[:, :, 0], hT


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,dk,dv", [(3, 5, 128, 128), (7, 2, 64, 256), (2, 3, 32, 40),
                                       (1, 1, 128, 1), (33, 4, 64, 64)])
def test_decode_matches_oracle(io, B, H, dk, dv):
    x = synth.make_decode(B, H, dk, dv, io=io, state_std=0.05, seed=7 * B + dk, device="cuda")
    s0 = U.f64(x.h0)
    o = gdn.gdn_decode(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
    U.sync()
    o_ref, s_ref = oracle_step(x, s0)
    # o is rounded once to the I/O dtype; the state stays fp32 arithmetic on
    # exactly representable inputs whatever the I/O dtype
    assert U.rel(U.f64(o), o_ref) <= (1e-4 if io == "f32" else 1e-2)
    assert U.rel(U.f64(x.h0), s_ref) <= 1e-4


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32)])
def test_decode_steps_equal_forward(dk, dv):
    # T decode steps from h0 give the chunked forward pass's outputs and state
    B, H, T = 2, 3, 70
    x = synth.make_dense(B, H, T, dk, dv, io="f32", h0_std=0.05, seed=31, device="cuda")
    o_f, h_f = gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
    state = x.h0.clone()
    outs = []
    for t in range(T):
        step = [a[:, :, t].contiguous() for a in (x.q, x.k, x.v, x.log_alpha, x.beta)]
        outs.append(gdn.gdn_decode(*step, state, check=True))
    o_d = torch.stack(outs, dim=2)
    U.sync()
    assert U.rel(U.f64(o_d), U.f64(o_f)) <= 1e-4
    assert U.rel(U.f64(state), U.f64(h_f)) <= 1e-4


def test_decode_slots():
    # a pool of states indexed by slot: the same result as the dense call on
    # the gathered states, and the slots nobody uses stay as they were
    P, B, H, dk, dv = 9, 4, 2, 64, 96
    x = synth.make_decode(B, H, dk, dv, io="bf16", state_std=0.05, n_slots=P, seed=3,
                          device="cuda")
    pool0 = x.h0.clone()
    idx = x.slots.long()
    sub = pool0[idx].clone()
    o = gdn.gdn_decode(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, slots=x.slots, check=True)
    o_ref = gdn.gdn_decode(x.q, x.k, x.v, x.log_alpha, x.beta, sub, check=True)
    U.sync()
    assert torch.equal(o, o_ref)
    assert torch.equal(x.h0[idx], sub)
    used = set(x.slots.tolist())
    rest = torch.tensor([i for i in range(P) if i not in used], device="cuda")
    assert torch.equal(x.h0[rest], pool0[rest])


def test_decode_bad_slot_reported():
    x = synth.make_decode(2, 2, 64, 64, io="bf16", state_std=0.05, n_slots=3, seed=4,
                          device="cuda")
    pool0 = x.h0.clone()
    slots = torch.tensor([1, 5], dtype=torch.int32, device="cuda")   # 5 is out of range
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_decode(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, slots=slots, check=True)
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG
    assert not torch.equal(x.h0[1], pool0[1])          # sequence 0 was stepped
    assert torch.equal(x.h0[0], pool0[0]) and torch.equal(x.h0[2], pool0[2])
    gdn.sync_check()                                   # the error was consumed


def test_decode_workload_sampled():
    # the timed workload (256 sequences x 32 heads, d = 128, bf16): the oracle
    # on a sample of (sequence, head) pairs
    x = synth.make_workload("gdn_decode_b256_h32_d128_bf16", device="cuda")
    pick = [(0, 0), (17, 5), (255, 31), (128, 16)]
    s0 = {p: U.f64(x.h0[p]) for p in pick}
    o = gdn.gdn_decode(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, check=True)
    U.sync()
    for b, h in pick:
        sel = lambda t: U.f64(t[b, h])[None, None, None]   # noqa: E731
        o_ref, s_ref = oracle.gdn_fwd(sel(x.q), sel(x.k), sel(x.v),
                                      U.f64(x.log_alpha[b, h]).reshape(1, 1, 1),
                                      U.f64(x.beta[b, h]).reshape(1, 1, 1),
                                      s0[(b, h)][None, None])
        assert U.rel(U.f64(o[b, h]), o_ref[0, 0, 0]) <= 1e-2
        assert U.rel(U.f64(x.h0[b, h]), s_ref[0, 0]) <= 1e-4
