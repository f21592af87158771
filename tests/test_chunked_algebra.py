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


@pytest.mark.parametrize("T", [1, 15, 16, 17, 64, 65, 130, 300])
@pytest.mark.parametrize("C", [16, 64, 128])
def test_chunked_form_equals_token_loop(lib, T, C):
    # the chunk length is a free parameter of the algebra: 128 gives the same
    # result as 64 and 16 (only the cost differs)
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


# ------------------------------------------------------------- backward pass
#
# The chunked adjoint the backward kernels compute (scalar gates), for
# L = sum dO . o + <dhT, hT>.  Per chunk, with M = strictly_lower(G * K K^T),
# A = diag(beta) M, P = mask * G * Q K^T (mask: s <= r) and dSC the adjoint of
# the chunk's end state, in reverse over the chunks:
#   dV' = P^T dO + diag(e) K dSC^T
#   dS0 = gamma_C dSC + dO^T diag(gamma) Q - dV'^T W
# and then, chunk by chunk with no order:
#   dQ = diag(gamma) dO S0 + dP K,   dP = mask * G * (dO V'^T)
#   dW = -dV' S0,  dV = diag(beta) T^T dV',  dT = dV' (diag(beta) V)^T + dW (diag(beta gamma) K)^T
#   dA = strictly_lower(-T^T dT T^T),  dM = diag(beta) dA
#   dK = dP^T Q + diag(e) V' dSC + diag(beta gamma) T^T dW + (N + N^T) K,  N = dM * G
#   dbeta_r = v_r . (T^T dV')_r + gamma_r k_r . (T^T dW)_r + sum_s dA_rs M_rs
#   dg      = gamma * rowdot(dO S0, Q) + rowsum - colsum of (P * dO V'^T) and of (dM * M)
#             + beta gamma rowdot(T^T dW, K), plus at the chunk's end
#             gamma_C <dSC, S0> + sum_r e_r v'_r . dSC k_r, minus e_r v'_r . dSC k_r at r
#   dlog_alpha = the reverse running sum of dg inside the chunk.


def _chunk_fwd(k, v, la, be, S0, erase):
    g = np.cumsum(la)
    gam = np.exp(g)
    L = len(la)
    diff = g[:, None] - g[None, :]
    G = np.exp(np.tril(diff))                      # e^{g_r - g_s}, 1 above the diagonal
    M = np.tril(G * (k @ k.T), -1) if erase else np.zeros((L, L))
    T = np.linalg.solve(np.eye(L) + be[:, None] * M, np.eye(L))
    W = T @ ((be * gam)[:, None] * k) if erase else np.zeros_like(k)
    U = T @ (be[:, None] * v)
    Vn = U - W @ S0.T
    e = np.exp(g[-1] - g)
    SC = gam[-1] * S0 + Vn.T @ (e[:, None] * k)
    return dict(g=g, gam=gam, G=G, M=M, T=T, W=W, Vn=Vn, e=e, SC=SC)


def chunked_backward(q, k, v, la, be, h0, dO, dhT, C, erase=True):
    """One (sequence, head): (dq, dk, dv, dlog_alpha, dbeta, dh0)."""
    Tn, dk = k.shape
    dv = v.shape[1]
    chunks = [slice(t0, min(t0 + C, Tn)) for t0 in range(0, Tn, C)]
    # forward: every chunk's starting state and factors
    S = np.zeros((dv, dk)) if h0 is None else h0.copy()
    fw = []
    for sl in chunks:
        f = _chunk_fwd(k[sl], v[sl], la[sl], be[sl], S, erase)
        f["S0"] = S
        fw.append(f)
        S = f["SC"]
    # reverse over chunks: the adjoint of each chunk's end state
    dSC = np.zeros((dv, dk)) if dhT is None else dhT.copy()
    for sl, f in zip(reversed(chunks), reversed(fw)):
        f["dSC"] = dSC
        P = np.tril(f["G"] * (q[sl] @ k[sl].T))
        f["P"] = P
        f["dVn"] = P.T @ dO[sl] + (f["e"][:, None] * k[sl]) @ dSC.T
        dSC = (f["gam"][-1] * dSC + dO[sl].T @ (f["gam"][:, None] * q[sl])
               - f["dVn"].T @ f["W"])
    dh0 = dSC
    out = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(la),
           np.zeros_like(be)]
    for sl, f in zip(chunks, fw):
        for i, grad in enumerate(_chunk_grads(q[sl], k[sl], v[sl], be[sl], dO[sl], f, erase)):
            out[i][sl] = grad
    return (*out, dh0)


def _chunk_grads(q, k, v, be, dO, f, erase):
    g, gam, G, M, T, Vn, e = (f[n] for n in ("g", "gam", "G", "M", "T", "Vn", "e"))
    S0, dSC, dVn, P = f["S0"], f["dSC"], f["dVn"], f["P"]
    dOV = dO @ Vn.T
    dP = np.tril(G * dOV)
    TdU = T.T @ dVn
    # W = T diag(beta gamma) K only exists with the erase term
    dW = -dVn @ S0
    TdW = T.T @ dW if erase else np.zeros_like(k)
    dq = gam[:, None] * (dO @ S0) + dP @ k
    dv = be[:, None] * TdU
    dk = dP.T @ q + e[:, None] * (Vn @ dSC) + (be * gam)[:, None] * TdW
    dbeta = np.sum(v * TdU, axis=1) + gam * np.sum(k * TdW, axis=1)
    dg = gam * np.sum((dO @ S0) * q, axis=1) + be * gam * np.sum(TdW * k, axis=1)
    Y = P * dOV
    dg += Y.sum(axis=1) - Y.sum(axis=0)
    if erase:
        dT = dVn @ (be[:, None] * v).T + dW @ ((be * gam)[:, None] * k).T
        dA = np.tril(-T.T @ dT @ T.T, -1)
        dM = be[:, None] * dA
        N = dM * G
        dk += (N + N.T) @ k
        dbeta += np.sum(dA * M, axis=1)
        Z = dM * M
        dg += Z.sum(axis=1) - Z.sum(axis=0)
    # the chunk's end state: gamma_C S0 and e_r = e^{g_C - g_r}
    de = np.einsum("ri,ij,rj->r", Vn, dSC, k)      # v'_r . dSC k_r
    dg[-1] += gam[-1] * np.sum(dSC * S0) + np.sum(e * de)
    dg -= e * de
    dla = np.cumsum(dg[::-1])[::-1]
    return dq, dk, dv, dla, dbeta


BWD_NAMES = ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dh0")


@pytest.mark.parametrize("erase", [True, False])
@pytest.mark.parametrize("T,C", [(1, 64), (17, 16), (64, 64), (100, 64), (130, 32)])
def test_chunked_adjoint_equals_oracle_gradient(lib, T, C, erase):
    rng = np.random.default_rng(900 + T + C)
    dk, dv = 6, 5
    q, k, v, la, be = P._rand_inputs(rng, 1, 1, T, dk, dv)
    h0 = rng.standard_normal((1, 1, dv, dk))
    dO = rng.standard_normal((1, 1, T, dv))
    dhT = rng.standard_normal((1, 1, dv, dk))
    ref = oracle.gdn_bwd(q, k, v, la, be, h0, dO, dhT, lib=lib, erase=erase)
    got = chunked_backward(q[0, 0], k[0, 0], v[0, 0], la[0, 0], be[0, 0], h0[0, 0],
                           dO[0, 0], dhT[0, 0], C, erase=erase)
    errs = {n: P._rel(a, b[0, 0]) for n, a, b in zip(BWD_NAMES, got, ref)}
    assert max(errs.values()) <= TOL, errs


def test_factorised_decay_holds_in_fp32_up_to_the_span_guard():
    # P^T dO with P_rs = e^{g_r - g_s} (q_r . k_s) equals P'^T (gamma * dO),
    # P'_rs = e^{-g_s} (q_r . k_s): the backward's tensor-core adjoint forms the
    # latter while the chunk's total log-decay g_C stays >= -80, where e^{-g_s}
    # is finite in fp32 (its exponent range ends near 88.7); past that bound
    # it forms P directly
    rng = np.random.default_rng(11)
    L, dk, dv = 64, 8, 4
    q = rng.standard_normal((L, dk)).astype(np.float32)
    k = rng.standard_normal((L, dk)).astype(np.float32)
    dO = rng.standard_normal((L, dv)).astype(np.float32)
    mask = np.tril(np.ones((L, L), dtype=np.float32))
    for gC, finite in ((-20.0, True), (-80.0, True), (-95.0, False)):
        g = np.linspace(gC / L, gC, L).astype(np.float32)
        with np.errstate(over="ignore", invalid="ignore"):
            direct = (mask * np.exp(np.tril(g[:, None] - g[None, :])) * (q @ k.T)).T @ dO
            Pp = mask * np.exp(-g)[None, :] * (q @ k.T)
            fact = Pp.T @ (np.exp(g)[:, None] * dO)
        ref = (np.tril(np.exp(np.float64(g)[:, None] - np.float64(g)[None, :]))
               * (q.astype(np.float64) @ k.T.astype(np.float64))).T @ dO
        assert np.isfinite(direct).all()
        assert P._rel(direct, ref) <= 1e-5
        assert np.isfinite(fact).all() == finite
        if finite:
            assert P._rel(fact, ref) <= 1e-5


def test_decode_row_form_equals_one_token(lib):
    # the decode kernel's form of one step: S' = alpha S + d k^T with
    # d = beta (v - alpha S k), and o = alpha S q + d (k . q); each row of the
    # new state needs only the same row of the old one
    rng = np.random.default_rng(13)
    dk, dv = 7, 5
    q, k, v, la, be = P._rand_inputs(rng, 1, 1, 1, dk, dv)
    S = rng.standard_normal((1, 1, dv, dk))
    o_ref, h_ref = oracle.gdn_fwd(q, k, v, la, be, S, lib=lib)
    a, b = np.exp(la[0, 0, 0]), be[0, 0, 0]
    qq, kk, vv, SS = q[0, 0, 0], k[0, 0, 0], v[0, 0, 0], S[0, 0]
    d = b * (vv - a * SS @ kk)
    assert P._rel(a * SS + np.outer(d, kk), h_ref[0, 0]) <= TOL
    assert P._rel(a * SS @ qq + d * (kk @ qq), o_ref[0, 0, 0]) <= TOL


def test_segment_map_from_the_forward_itself(lib):
    # a segment's affine map S -> S A + B read off two forward runs: A is the
    # final state from h0 = I with v = 0 (d_v taken as d_k), B the final
    # state from h0 = 0 with the real v; then any h0 gives h0 A + B
    rng = np.random.default_rng(17)
    T, dk, dv = 90, 5, 3
    q, k, v, la, be = P._rand_inputs(rng, 1, 1, T, dk, dv)
    _, A = oracle.gdn_fwd(q, k, np.zeros((1, 1, T, dk)), la, be, np.eye(dk)[None, None], lib=lib)
    _, B = oracle.gdn_fwd(q, k, v, la, be, None, lib=lib)
    h0 = rng.standard_normal((1, 1, dv, dk))
    _, h_ref = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib)
    assert P._rel(h0[0, 0] @ A[0, 0] + B[0, 0], h_ref[0, 0]) <= TOL
