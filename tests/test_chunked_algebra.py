"""The chunked (WY / UT) form the kernels compute, written out in fp64 numpy,
equals the token-by-token oracle (CPU).

"Gated DeltaNet GPU并行实现", section 3.2, splits the sequence into chunks
whose insides are dense matrix products while a state is carried across
chunks; section 2.3 composes the per-chunk affine maps.  Writing the update
as S_t = alpha_t S_{t-1} + u_t k_t^T with u_t = beta_t (v_t - alpha_t S_{t-1} k_t)
and unrolling it inside a chunk that starts from S_0 (g_r = sum of log alpha
up to r, gamma_r = e^{g_r}):

    u_r + sum_{s<r} beta_r e^{g_r - g_s} (k_r . k_s) u_s = beta_r v_r - beta_r gamma_r S_0 k_r

so with A_rs = beta_r e^{g_r - g_s} (k_r . k_s) for s < r and T = (I + A)^{-1},
the rows u_r form V' = U - W S_0^T, where W = T diag(beta gamma) K and
U = T diag(beta) V; then

    O   = (Q * gamma) S_0^T + [mask_{r >= s} (Q K^T) * e^{g_r - g_s}] V'
    S_C = S_0 (gamma_C I - W^T Kt) + U^T Kt,        Kt = K * e^{g_C - g_r},

the second line being the chunk's affine map S -> S A_c + B_c.  Nothing here
is shared with the oracle or the CUDA path; the inverse is a library solve.
"""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as P

TOL = 1e-10


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library(oracle.build())


def chunk_factors(k, v, la, be):
    """g, gamma, W, U and Kt of one chunk (rows = its tokens)."""
    g = np.cumsum(la)
    gam = np.exp(g)
    L = len(la)
    A = np.zeros((L, L))
    for r in range(L):
        for s in range(r):
            A[r, s] = be[r] * np.exp(g[r] - g[s]) * (k[r] @ k[s])
    inv = np.linalg.solve(np.eye(L) + A, np.eye(L))
    W = inv @ ((be * gam)[:, None] * k)
    U = inv @ (be[:, None] * v)
    Kt = k * np.exp(g[-1] - g)[:, None]
    return g, gam, W, U, Kt


def chunked_forward(q, k, v, la, be, h0, C):
    """One (sequence, head): o [T][d_v] and the final state [d_v][d_k]."""
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if h0 is None else h0.copy()
    o = np.zeros((T, dv))
    for t0 in range(0, T, C):
        sl = slice(t0, min(t0 + C, T))
        qc, kc, vc = q[sl], k[sl], v[sl]
        g, gam, W, U, Kt = chunk_factors(kc, vc, la[sl], be[sl])
        Vn = U - W @ S.T
        decay = np.tril(np.exp(g[:, None] - g[None, :]))
        o[sl] = (qc * gam[:, None]) @ S.T + ((qc @ kc.T) * decay) @ Vn
        S = gam[-1] * S + Vn.T @ Kt
    return o, S


def chunk_maps(k, v, la, be, C):
    """The affine map (A_c, B_c) of every chunk: S -> S A_c + B_c."""
    maps = []
    for t0 in range(0, len(la), C):
        sl = slice(t0, min(t0 + C, len(la)))
        g, gam, W, U, Kt = chunk_factors(k[sl], v[sl], la[sl], be[sl])
        maps.append((gam[-1] * np.eye(k.shape[1]) - W.T @ Kt, U.T @ Kt))
    return maps


@pytest.mark.parametrize("T", [1, 15, 16, 17, 64, 65, 130])
@pytest.mark.parametrize("C", [16, 64])
def test_chunked_form_equals_token_loop(lib, T, C):
    rng = np.random.default_rng(100 + T + C)
    q, k, v, la, be = P._rand_inputs(rng, 1, 1, T, 6, 5)
    h0 = rng.standard_normal((1, 1, 5, 6))
    o_ref, h_ref = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib)
    o, S = chunked_forward(q[0, 0], k[0, 0], v[0, 0], la[0, 0], be[0, 0], h0[0, 0], C)
    assert P._rel(o, o_ref[0, 0]) <= TOL
    assert P._rel(S, h_ref[0, 0]) <= TOL


def test_chunk_maps_compose_to_final_state(lib):
    # the per-chunk affine maps folded earlier-first (S -> S A + B), and the
    # same maps grouped into two segments first and the segments composed
    rng = np.random.default_rng(7)
    T, dk, dv = 150, 4, 7
    q, k, v, la, be = P._rand_inputs(rng, 1, 1, T, dk, dv)
    h0 = rng.standard_normal((1, 1, dv, dk))
    _, h_ref = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib)
    maps = chunk_maps(k[0, 0], v[0, 0], la[0, 0], be[0, 0], 32)
    S = h0[0, 0].copy()
    for A, B in maps:
        S = S @ A + B
    assert P._rel(S, h_ref[0, 0]) <= TOL

    def compose(ms):
        A, B = np.eye(dk), np.zeros((dv, dk))
        for A2, B2 in ms:
            A, B = A @ A2, B @ A2 + B2
        return A, B
    (A1, B1), (A2, B2) = compose(maps[:2]), compose(maps[2:])
    S2 = (h0[0, 0] @ A1 + B1) @ A2 + B2
    assert P._rel(S2, h_ref[0, 0]) <= TOL


def test_no_erase_makes_the_inverse_the_identity(lib):
    # without the erase term u_r = beta_r v_r: A = 0, T = I, W = 0 in V'
    rng = np.random.default_rng(9)
    T, dk, dv = 70, 5, 3
    q, k, v, la, be = P._rand_inputs(rng, 1, 1, T, dk, dv)
    o_ref, h_ref = oracle.gdn_fwd(q, k, v, la, be, None, lib=lib, erase=False)
    S = np.zeros((dv, dk))
    o = np.zeros((T, dv))
    qq, kk, vv, ll, bb = q[0, 0], k[0, 0], v[0, 0], la[0, 0], be[0, 0]
    for t0 in range(0, T, 64):
        sl = slice(t0, min(t0 + 64, T))
        g = np.cumsum(ll[sl])
        Vn = bb[sl][:, None] * vv[sl]
        decay = np.tril(np.exp(g[:, None] - g[None, :]))
        o[sl] = (qq[sl] * np.exp(g)[:, None]) @ S.T + ((qq[sl] @ kk[sl].T) * decay) @ Vn
        S = np.exp(g[-1]) * S + Vn.T @ (kk[sl] * np.exp(g[-1] - g)[:, None])
    assert P._rel(o, o_ref[0, 0]) <= TOL
    assert P._rel(S, h_ref[0, 0]) <= TOL
