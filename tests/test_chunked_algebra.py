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


# ------------------------------------------------- a forget gate per key dimension
#
# With alpha_t a d_k-vector ("Gated DeltaNet GPU并行实现", section 2.2, the
# diagonal gate acting on the old state first) the same unrolling gives, with
# G_r the running sum of the log-gate vectors and Gamma_r = e^{G_r}:
#   A_rs = beta_r sum_j k_rj k_sj e^{G_rj - G_sj}       (s < r)
#   W = T diag(beta) (K * Gamma),  U = T diag(beta) V,  V' = U - W S_0^T
#   O = (Q * Gamma) S_0^T + P V',  P_rs = sum_j q_rj k_sj e^{G_rj - G_sj}  (s <= r)
#   S_C = S_0 diag(Gamma_C) + V'^T (K * e^{G_C - G})
# The decay inside A and P is taken block by block (16 rows): for a row block
# after a key block, e^{G_r - G_s} = e^{G_r - G_m} e^{G_m - G_s} with m the key
# block's last row, so both factors are at most 1 and nothing overflows.

BLK = 16


def decayed_products(X, K, G, inclusive):
    """sum_j X_rj K_sj e^{G_rj - G_sj} for s < r (s <= r when inclusive), by
    16-row blocks with every exponent <= 0."""
    L = len(G)
    out = np.zeros((L, L))
    for b0 in range(0, L, BLK):
        rows = slice(b0, min(b0 + BLK, L))
        for c0 in range(0, b0 + 1, BLK):
            cols = slice(c0, min(c0 + BLK, L))
            if c0 < b0:
                m = cols.stop - 1                  # the key block's last row
                fr, fs = G[rows] - G[m], G[m] - G[cols]
                assert fr.max() <= 0 and fs.max() <= 0
                out[rows, cols] = (X[rows] * np.exp(fr)) @ (K[cols] * np.exp(fs)).T
            else:                                  # diagonal block: pairwise
                for r in range(rows.start, rows.stop):
                    last = r + 1 if inclusive else r
                    for s in range(cols.start, last):
                        assert (G[r] - G[s]).max() <= 0
                        out[r, s] = X[r] @ (K[s] * np.exp(G[r] - G[s]))
    return out


def chunked_forward_vg(q, k, v, la, be, h0, C, erase=True):
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if h0 is None else h0.copy()
    o = np.zeros((T, dv))
    for t0 in range(0, T, C):
        sl = slice(t0, min(t0 + C, T))
        qc, kc, vc, bc = q[sl], k[sl], v[sl], be[sl]
        G = np.cumsum(la[sl], axis=0)
        Gam = np.exp(G)
        L = len(bc)
        A = (bc[:, None] * decayed_products(kc, kc, G, inclusive=False) if erase
             else np.zeros((L, L)))
        inv = np.linalg.solve(np.eye(L) + A, np.eye(L))
        W = inv @ (bc[:, None] * kc * Gam) if erase else np.zeros((L, dk))
        U = inv @ (bc[:, None] * vc)
        Vn = U - W @ S.T
        Pm = decayed_products(qc, kc, G, inclusive=True)
        o[sl] = (qc * Gam) @ S.T + Pm @ Vn
        S = S * Gam[-1][None, :] + Vn.T @ (kc * np.exp(G[-1] - G))
    return o, S


@pytest.mark.parametrize("erase", [True, False])
@pytest.mark.parametrize("T,C", [(1, 64), (40, 16), (64, 64), (100, 64), (131, 32)])
def test_vector_gate_chunked_form_equals_token_loop(lib, T, C, erase):
    rng = np.random.default_rng(500 + T + C)
    dk, dv = 6, 5
    q, k, v, _, be = P._rand_inputs(rng, 1, 1, T, dk, dv)
    la = -0.5 * np.log1p(np.exp(rng.standard_normal((1, 1, T, dk))))
    h0 = rng.standard_normal((1, 1, dv, dk))
    o_ref, h_ref = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib, erase=erase, vector_gate=True)
    o, S = chunked_forward_vg(q[0, 0], k[0, 0], v[0, 0], la[0, 0], be[0, 0], h0[0, 0], C,
                              erase=erase)
    assert P._rel(o, o_ref[0, 0]) <= TOL
    assert P._rel(S, h_ref[0, 0]) <= TOL


def test_vector_gate_blocks_survive_steep_decay(lib):
    # decays far beyond fp32's exponent range over one chunk: the blocked
    # factors stay <= 1, so the chunked form still matches the token loop
    rng = np.random.default_rng(77)
    T, dk, dv = 64, 4, 3
    q, k, v, _, be = P._rand_inputs(rng, 1, 1, T, dk, dv)
    la = -rng.uniform(2.0, 6.0, (1, 1, T, dk))
    h0 = rng.standard_normal((1, 1, dv, dk))
    o_ref, h_ref = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib, vector_gate=True)
    o, S = chunked_forward_vg(q[0, 0], k[0, 0], v[0, 0], la[0, 0], be[0, 0], h0[0, 0], 64)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    assert P._rel(o, o_ref[0, 0]) <= TOL
