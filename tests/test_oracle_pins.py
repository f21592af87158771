"""The oracle against closed forms, invariants and planted mistakes (CPU)."""
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
from tests import oracle_pins as P


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library(oracle.build())


@pytest.mark.parametrize("name", sorted(P.ALL_PINS))
def test_pin(lib, name):
    assert P.ALL_PINS[name](lib) <= P.PIN_TOL


@pytest.mark.parametrize("dk,dv", [(2, 2), (3, 5), (8, 4)])
def test_pins_other_shapes(lib, dk, dv):
    # d = 2 is the tiny case the page recommends checking first
    assert P.pin_bracketing(lib, dk=dk, dv=dv, T=9, seed=11 + dk) <= P.PIN_TOL
    assert P.pin_t1_closed_form(lib, dk=dk, dv=dv, seed=12 + dv) <= P.PIN_TOL
    assert P.pin_beta_zero(lib, dk=dk, dv=dv, seed=13) <= P.PIN_TOL
    assert P.pin_exact_recall(lib, dk=dk, dv=dv, seed=14) <= P.PIN_TOL


def test_reversed_order_is_detected(lib):
    # composing the maps in the wrong order must NOT reproduce the oracle
    assert P.reversed_order_error(lib) > 1e-3


def test_empty_and_degenerate(lib):
    # T = 0: no outputs, hT = h0
    rng = np.random.default_rng(0)
    h0 = rng.standard_normal((1, 2, 3, 4))
    z = np.zeros((1, 2, 0, 4))
    o, hT = oracle.gdn_fwd(z, z, np.zeros((1, 2, 0, 3)), np.zeros((1, 2, 0)),
                           np.zeros((1, 2, 0)), h0, lib=lib)
    assert o.shape == (1, 2, 0, 3)
    assert np.array_equal(hT, h0)
    # k = 0: nothing is erased or written, only decay
    T = 6
    q = rng.standard_normal((1, 1, T, 4))
    la = -rng.uniform(0, 1, (1, 1, T))
    be = rng.uniform(0, 1, (1, 1, T))
    o, hT = oracle.gdn_fwd(q, np.zeros((1, 1, T, 4)), rng.standard_normal((1, 1, T, 3)),
                           la, be, h0[:, :1], lib=lib)
    assert np.allclose(hT[0, 0], np.exp(la.sum()) * h0[0, 0], rtol=1e-13, atol=0)


def test_threads_match_single(lib):
    rng = np.random.default_rng(5)
    q, k, v, la, be = P._rand_inputs(rng, 2, 3, 20, 4, 5)
    o1, h1 = oracle.gdn_fwd(q, k, v, la, be, lib=lib)
    o2, h2 = oracle.gdn_fwd(q, k, v, la, be, threads=4, lib=lib)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)
    cu = np.array([0, 7, 7, 20])
    qv, kv, vv = q[0], k[0], v[0]
    a = oracle.gdn_fwd_varlen(qv, kv, vv, la[0], be[0], cu, lib=lib)
    b = oracle.gdn_fwd_varlen(qv, kv, vv, la[0], be[0], cu, threads=3, lib=lib)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# Each planted mistake is a plausible slip in the oracle's loop.  Every one of
# them must make at least one pin fail; square shapes keep the transposed
# variants in bounds.
MUTANTS = {
    "erase_sign": ("a * (s - b * kS[i] * kt[j])", "a * (s + b * kS[i] * kt[j])"),
    "alpha_dropped": ("a * (s - b * kS[i] * kt[j])", "(s - b * kS[i] * kt[j])"),
    "alpha_on_write": ("+ b * vt[i] * kt[j];", "+ a * b * vt[i] * kt[j];"),
    "beta_dropped_on_write": ("+ b * vt[i] * kt[j];", "+ vt[i] * kt[j];"),
    "erase_left_side": ("acc += S[i * dk + j] * kt[j];", "acc += S[j * dk + i] * kt[j];"),
    "output_transposed": ("acc += S[i * dk + j] * qt[j];", "acc += S[j * dk + i] * qt[j];"),
    "output_uses_key": ("acc += S[i * dk + j] * qt[j];", "acc += S[i * dk + j] * kt[j];"),
    "beta_off_by_one": ("const double b = beta[t];", "const double b = beta[t > 0 ? t - 1 : 0];"),
    "gate_not_exponentiated": ("const double a = exp(la[t]);", "const double a = 1.0 + la[t];"),
    "h0_ignored": ("if (h0)\n        memcpy", "if (0)\n        memcpy"),
    "varlen_offset": ("long row = h * T_total + t0;", "long row = h * T_total + t0 / 2;"),
    # the gated-linear-attention loop
    "gla_alpha_dropped": ("g * S[i * dk + j] + w", "S[i * dk + j] + w"),
    "gla_beta_dropped": ("+ w * vt[i] * kt[j];", "+ vt[i] * kt[j];"),
    "gla_alpha_on_write": ("+ w * vt[i] * kt[j];", "+ g * w * vt[i] * kt[j];"),
    "gla_gate_not_exponentiated": ("const double g = exp(la[t]);", "const double g = 1.0 + la[t];"),
    "gla_output_transposed": ("sum += S[i * dk + j] * qt[j];", "sum += S[j * dk + i] * qt[j];"),
    "gla_h0_ignored": ("if (h0)\n        memcpy(S, h0, sizeof(double) * (size_t)(dv * dk));\n    else\n        memset(S, 0, sizeof(double) * (size_t)(dv * dk));\n    for (t = 0; t < T; ++t) {\n        const double *kt = k + t * dk;\n        const double *vt = v + t * dv;\n        const double *qt = q + t * dk;\n        const double g",
                       "if (0)\n        memcpy(S, h0, sizeof(double) * (size_t)(dv * dk));\n    else\n        memset(S, 0, sizeof(double) * (size_t)(dv * dk));\n    for (t = 0; t < T; ++t) {\n        const double *kt = k + t * dk;\n        const double *vt = v + t * dv;\n        const double *qt = q + t * dk;\n        const double g"),
    "gla_varlen_offset": ("long rw = h * T_total + s0;", "long rw = h * T_total + s0 / 2;"),
    # the per-dimension-gate loop
    "vg_gate_wrong_axis": ("S[i * dk + j] *= exp(lat[j]);", "S[i * dk + j] *= exp(lat[i % dk]);"),
    "vg_gate_not_exponentiated": ("S[i * dk + j] *= exp(lat[j]);", "S[i * dk + j] *= 1.0 + lat[j];"),
    "vg_beta_dropped": ("+= bt * (vt[i] - Sk[i]) * kt[j];", "+= (vt[i] - Sk[i]) * kt[j];"),
    "vg_erase_sign": ("+= bt * (vt[i] - Sk[i]) * kt[j];", "+= bt * (vt[i] + Sk[i]) * kt[j];"),
    "vg_erase_ignored": ("Sk[i] = erase ? dot : 0.0;", "Sk[i] = 0.0;"),
    "vg_output_transposed": ("out += S[i * dk + j] * qt[j];", "out += S[j * dk + i] * qt[j];"),
    "vg_varlen_offset": ("long at = h * T_total + first;", "long at = h * T_total + first / 2;"),
    # gradient loop
    "bwd_output_term_dropped": ("dS[i * dk + j] += dot[i] * qt[j];",
                                "dS[i * dk + j] += 0.0 * dot[i] * qt[j];"),
    "bwd_dq_from_old_state": ("acc += Y[i * dk + j] * dot[i];", "acc += X[i * dk + j] * dot[i];"),
    "bwd_dbeta_sign": ("(erase ? vt[i] - a * Xk[i] : vt[i])", "(erase ? vt[i] + a * Xk[i] : vt[i])"),
    "bwd_dlog_alpha_unscaled": ("dla[t] = a * (erase ? sx - b * cross : sx);",
                                "dla[t] = (erase ? sx - b * cross : sx);"),
    "bwd_dk_cross_term_dropped": ("(X[i * dk + j] * dSk[i] + dS[i * dk + j] * Xk[i])",
                                  "(X[i * dk + j] * dSk[i])"),
    "bwd_adjoint_erase_dropped": ("(erase ? b * dSk[i] * kt[j] : 0.0)", "0.0"),
    "bwd_dv_beta_dropped": ("dv_[t * dv + i] = b * dSk[i];", "dv_[t * dv + i] = dSk[i];"),
    "bwd_varlen_state_offset": ("long st = (n * H + h) * dv * dk;",
                                "long st = (h * N + n) * dv * dk;"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="gdn_oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant_dir, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, "mutation anchor missing: " + old
    path = os.path.join(mutant_dir, name + ".c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    mlib = oracle.load_library(oracle.compile_source(path, os.path.join(mutant_dir, name + ".so")))
    square = dict(dk=5, dv=5)
    errs = {
        "beta_zero": P.pin_beta_zero(mlib, **square),
        "exact_recall": P.pin_exact_recall(mlib, **square),
        "bracketing": P.pin_bracketing(mlib, **square),
        "t1": P.pin_t1_closed_form(mlib, **square),
        "linear_attention": P.pin_linear_attention(mlib, dk=8, dv=8),
        "continuation": P.pin_continuation(mlib, **square),
        "varlen": P.pin_varlen_split(mlib, dk=5, dv=5),
        "gla_closed_form": P.pin_gla_closed_form(mlib, **square),
        "gla_linear_attention": P.pin_gla_linear_attention(mlib, **square),
        "gla_varlen": P.pin_gla_varlen_split(mlib, dk=5, dv=5),
        "vg_scalar": P.pin_vg_scalar_reduction(mlib, **square),
        "vg_bracketing": P.pin_vg_bracketing(mlib, **square),
        "vg_beta_zero": P.pin_vg_beta_zero(mlib, **square),
        "vg_varlen": P.pin_vg_varlen_split(mlib, dk=5, dv=5),
        "bwd_fd": P.pin_bwd_finite_differences(mlib),
        "bwd_fd_no_erase": P.pin_bwd_fd_no_erase(mlib),
        "bwd_adjoint": P.pin_bwd_adjoint(mlib),
        "bwd_varlen": P.pin_bwd_varlen_split(mlib),
    }
    assert max(errs.values()) > 1e-6, errs


def test_bwd_empty_sequence_passes_dhT_through(lib):
    # T = 0: hT = h0, so dh0 = dhT and there are no token gradients
    rng = np.random.default_rng(3)
    h0 = rng.standard_normal((1, 2, 3, 4))
    dhT = rng.standard_normal((1, 2, 3, 4))
    z = np.zeros((1, 2, 0, 4))
    g = oracle.gdn_bwd(z, z, np.zeros((1, 2, 0, 3)), np.zeros((1, 2, 0)), np.zeros((1, 2, 0)),
                       h0, np.zeros((1, 2, 0, 3)), dhT, lib=lib)
    assert g[0].shape == (1, 2, 0, 4) and np.array_equal(g[5], dhT)
