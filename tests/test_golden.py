"""Hand-worked examples (tests/golden/) against the oracle (CPU) and against
the CUDA path (GPU, through zero padding to widths the kernels take)."""
from __future__ import annotations

import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
from tests import golden_fixtures as G

# the examples are dyadic, so fp64 reproduces them exactly; the bound only
# leaves room for exp(log(alpha)) rounding
ORACLE_TOL = 1e-12


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library(oracle.build())


@pytest.mark.parametrize("name", G.FORWARD)
def test_oracle_matches_hand_worked_forward(lib, name):
    errs = G.oracle_forward_errors(lib, name)
    assert max(errs.values()) <= ORACLE_TOL, errs


def test_oracle_matches_hand_worked_gradient(lib):
    errs = G.oracle_gradient_errors(lib)
    assert max(errs.values()) <= ORACLE_TOL, errs


def test_oracle_matches_hand_worked_gradient_packed(lib):
    errs = G.oracle_packed_gradient_errors(lib)
    assert max(errs.values()) <= ORACLE_TOL, errs


def test_fixture_derivations_are_consistent():
    # what the derivations lean on: recall at beta = 1 (S_2 k_2 = v_2 for the
    # hand-derived S_2), and the gradient fixture's forward is the first
    # token of the forward fixture
    g = G.load("delta_rule_d2_t3")
    S2 = np.array([[1.25, -2.0], [2.0, 2.0]])
    assert np.array_equal(S2 @ g["k"][1], g["v"][1])
    assert np.array_equal(S2 @ g["q"][1], g["o"][1])
    d = G.load(G.GRADIENT)
    assert np.array_equal(d["h0"], g["h0"])
    for key in ("q", "k", "v", "alpha", "beta"):
        assert np.array_equal(d[key][0], g[key][0]), key


def _planted():
    from tests.test_oracle_pins import MUTANTS
    return sorted(MUTANTS)


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="gdn_golden_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", _planted())
def test_hand_worked_values_catch_planted_mistake(mutant_dir, name):
    from tests.test_oracle_pins import MUTANTS
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")).read()
    old, new = MUTANTS[name]
    path = os.path.join(mutant_dir, name + ".c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    mlib = oracle.load_library(oracle.compile_source(path, os.path.join(mutant_dir, name + ".so")))
    errs = {}
    for fx in G.FORWARD:
        errs.update({fx + ":" + k: v for k, v in G.oracle_forward_errors(mlib, fx).items()})
    errs.update(G.oracle_gradient_errors(mlib))
    errs.update({"packed:" + k: v for k, v in G.oracle_packed_gradient_errors(mlib).items()})
    assert max(errs.values()) > 1e-6, errs


# --------------------------------------------------------------------- GPU

# widths the parity tests already run on each path: fp32 I/O at d = 32 (the
# mma.sync path), bf16 I/O at d = 64 (tensor-core path for scalar gates)
WIDTH = {"f32": 32, "bf16": 64}
# fp32 I/O: 1e-4 on o and hT; bf16 I/O: 1e-2 on o, 2e-2 on hT
TOL = {"f32": (1e-4, 1e-4), "bf16": (1e-2, 2e-2)}


def _dev(a, dtype):
    import torch
    return torch.tensor(np.ascontiguousarray(a), dtype=torch.float32,
                        device="cuda").to(dtype).contiguous()


def _host(t):
    return t.detach().to("cpu").double().numpy()


def _padded_inputs(g, D, io):
    """The fixture as [1,1,T,D] device tensors, zero beyond its 2 x 2 block."""
    import torch
    dt = torch.float32 if io == "f32" else torch.bfloat16
    one = lambda a: a[None, None]  # noqa: E731
    q, k, v = (_dev(one(G.pad(g[n], (D,))), dt) for n in ("q", "k", "v"))
    la = g["log_alpha"]
    la = _dev(one(G.pad(la, (D,)) if g["vector_gate"] else la), torch.float32)
    be = _dev(one(g["beta"]), torch.float32)
    h0 = _dev(one(G.pad(g["h0"], (D, D))), torch.float32)
    return q, k, v, la, be, h0


@pytest.mark.gpu
@pytest.mark.parametrize("impl", ["auto", "simt"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("name", G.FORWARD)
def test_gpu_forward_matches_hand_worked(name, io, impl):
    import torch
    import gated_deltanet_recurrence_gdn_gb300 as gdn
    g = G.load(name)
    D, T = WIDTH[io], g["T"]
    q, k, v, la, be, h0 = _padded_inputs(g, D, io)
    mode = gdn.GDN_IMPL_AUTO if impl == "auto" else gdn.GDN_IMPL_SIMT
    with gdn.use_impl(mode):
        o, hT = gdn.gdn_fwd(q, k, v, la, be, h0, check=True, erase=g["erase"])
        # the same sequence twice in one packed batch, both from h0
        cu = torch.tensor([0, T, 2 * T], dtype=torch.int32, device="cuda")
        cat = lambda t: torch.cat([t[0, 0], t[0, 0]]).unsqueeze(0).contiguous()  # noqa: E731
        op, hp = gdn.gdn_fwd_varlen(cat(q), cat(k), cat(v), cat(la), cat(be), cu,
                                    torch.cat([h0, h0]).contiguous(), check=True,
                                    erase=g["erase"])
    torch.cuda.synchronize()
    to, th = TOL[io]
    o_ref, h_ref = G.pad(g["o"], (D,)), G.pad(g["hT"], (D, D))
    assert G.rel(_host(o)[0, 0], o_ref) <= to
    assert G.rel(_host(hT)[0, 0], h_ref) <= th
    assert G.rel(_host(op)[0], np.concatenate([o_ref, o_ref])) <= to
    assert max(G.rel(_host(hp)[n, 0], h_ref) for n in range(2)) <= th


@pytest.mark.gpu
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_gpu_decode_matches_hand_worked(io):
    # three decode steps from h0 walk the delta-rule example token by token
    import torch
    import gated_deltanet_recurrence_gdn_gb300 as gdn
    g = G.load("delta_rule_d2_t3")
    D = 32
    q, k, v, la, be, state = _padded_inputs(g, D, io)
    for t in range(g["T"]):
        # clone: a [1, 1] slice of the gates counts as contiguous, and the
        # view would start 4 t bytes into the buffer (the library wants 16)
        step = [a[:, :, t].clone() for a in (q, k, v, la, be)]
        o = gdn.gdn_decode(*step, state, check=True)
        torch.cuda.synchronize()
        assert G.rel(_host(o)[0, 0], G.pad(g["o"][t], (D,))) <= TOL[io][0]
    assert G.rel(_host(state)[0, 0], G.pad(g["hT"], (D, D))) <= 1e-4


@pytest.mark.gpu
@pytest.mark.parametrize("impl", ["auto", "simt"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_gpu_gradient_matches_hand_worked(io, impl):
    import torch
    import gated_deltanet_recurrence_gdn_gb300 as gdn
    g = G.load(G.GRADIENT)
    D = WIDTH[io]
    q, k, v, la, be, h0 = _padded_inputs(g, D, io)
    dout = _dev(G.pad(g["dO"], (D,))[None, None], q.dtype)
    dhT = _dev(G.pad(g["dhT"], (D, D))[None, None], torch.float32)
    mode = gdn.GDN_IMPL_AUTO if impl == "auto" else gdn.GDN_IMPL_SIMT
    with gdn.use_impl(mode):
        got = gdn.gdn_bwd(q, k, v, la, be, h0, dout, dhT, check=True)
    torch.cuda.synchronize()
    want = {"dq": G.pad(g["dq"], (D,)), "dk": G.pad(g["dk"], (D,)), "dv": G.pad(g["dv"], (D,)),
            "dlog_alpha": g["dlog_alpha"], "dbeta": g["dbeta"],
            "dh0": G.pad(g["dh0"], (D, D))}
    errs = {n: G.rel(_host(a)[0, 0], want[n]) for n, a in zip(G.GRAD_NAMES, got)}
    assert max(errs.values()) <= (1e-4 if io == "f32" else 1e-2), errs
