"""Checks that pin the fp64 oracle to facts other than itself.

Each function takes a loaded oracle library (so the planted-mistake test can
run the same checks against a deliberately broken build) and returns the
worst relative error it saw; the caller compares it with PIN_TOL.

Passages ("Gated DeltaNet GPU并行实现"): the update is the gated delta rule of
sections 2.1-2.2; section 2.3 states that the per-token maps are affine and
compose associatively; section 5.2 (first pitfall) warns that composing them
in the wrong order is the classic bug and recommends checking tiny random
problems (d = 2) against the naive loop.  The reduction to (gated) linear
attention follows the linear-attention recurrence of "线性注意力机制与Gated
DeltaNet的优化实践" sections 2.2-2.3, with the erase term vanishing for
mutually orthogonal keys.  The gated-linear-attention loop (the recurrence
without the erase term, same page sections 2.2-2.3) is pinned to its
unrolled closed form, to plain linear attention, and to the delta rule where
the two coincide.  The per-key-dimension gate loop (section 2.2's diagonal
factor) is pinned to the scalar loops when its entries are equal, to the
explicit affine maps diag(alpha_t)(I - beta_t k k^T), beta_t v k^T composed in
random bracketings (which fixes that the decay acts before the erase), and to
its beta = 0 closed form.

The gradient oracle (no page writes the delta rule's backward pass out; the
page "企业官网建设流程全解析" recomputes the state in the backward pass,
sections 2 and 4.3, and checks gradients numerically, section 5.3) is pinned
to central finite differences of the forward loops (a five-point stencil in
fp64, every input along a random direction), to the exact adjoint identities
of the forward's linear arguments -- L = <dO, O> + <dhT, hT> is linear in
(h0, V) jointly, so L = <dV, V> + <dh0, h0>, and O is linear in q while hT
does not depend on it, so <dO, O> = <dq, q> -- and to per-sequence calls for
packed batches.
"""
from __future__ import annotations

import numpy as np

import oracle

PIN_TOL = 1e-10


def _rel(a, b):
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def _rand_inputs(rng, B, H, T, dk, dv, unit_k=True):
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv))
    la = -np.log1p(np.exp(rng.standard_normal((B, H, T)))) * 0.5
    be = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, T))))
    return q, k, v, la, be


def pin_beta_zero(lib, dk=5, dv=3, T=9, seed=1):
    """beta = 0: the state only decays, S_t = (prod_{i<=t} alpha_i) h0, so
    o_t = (prod alpha) h0 q_t and hT = (prod alpha) h0."""
    rng = np.random.default_rng(seed)
    q, k, v, la, _ = _rand_inputs(rng, 1, 2, T, dk, dv)
    be = np.zeros_like(la)
    h0 = rng.standard_normal((1, 2, dv, dk))
    o, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib)
    cum = np.exp(np.cumsum(la, axis=-1))                      # [1,2,T]
    o_ref = np.einsum("bht,bhij,bhtj->bhti", cum, h0, q)
    hT_ref = cum[..., -1][..., None, None] * h0
    return max(_rel(o, o_ref), _rel(hT, hT_ref))


def pin_exact_recall(lib, dk=6, dv=4, T=11, seed=2):
    """alpha = 1, beta = 1, unit k: after the write S_t k_t = v_t exactly,
    because S (I - k k^T) k = 0 and v k^T k = v.  With q_t = k_t the output
    is therefore o_t = v_t at every step, whatever h0 is."""
    rng = np.random.default_rng(seed)
    _, k, v, _, _ = _rand_inputs(rng, 1, 1, T, dk, dv)
    la = np.zeros((1, 1, T))
    be = np.ones((1, 1, T))
    h0 = rng.standard_normal((1, 1, dv, dk))
    o, hT = oracle.gdn_fwd(k, k, v, la, be, h0, lib=lib)
    err = _rel(o, v)
    err = max(err, _rel(hT[0, 0] @ k[0, 0, -1], v[0, 0, -1]))
    return err


def _affine_maps(k, v, la, be):
    """Per-token maps S -> S A_t + B_t with A_t = alpha_t (I - beta_t k k^T)
    and B_t = beta_t v_t k_t^T (section 2.2's A_t, B_t, for the row-state)."""
    T, dk = k.shape
    A = np.empty((T, dk, dk))
    Bm = np.empty((T, v.shape[1], dk))
    for t in range(T):
        a = np.exp(la[t])
        A[t] = a * (np.eye(dk) - be[t] * np.outer(k[t], k[t]))
        Bm[t] = be[t] * np.outer(v[t], k[t])
    return A, Bm


def _fold(A, Bm, lo, hi, rng, reverse=False):
    """Compose maps lo..hi-1 with a random bracketing.  Earlier map first:
    (A1,B1) then (A2,B2) is (A1 A2, B1 A2 + B2).  reverse=True composes in
    the wrong order (the mistake section 5.2 warns about)."""
    if hi - lo == 1:
        return A[lo], Bm[lo]
    mid = int(rng.integers(lo + 1, hi))
    A1, B1 = _fold(A, Bm, lo, mid, rng, reverse)
    A2, B2 = _fold(A, Bm, mid, hi, rng, reverse)
    if reverse:
        return A2 @ A1, B2 @ A1 + B1
    return A1 @ A2, B1 @ A2 + B2


def pin_bracketing(lib, dk=4, dv=3, T=13, seed=3, trials=6):
    """Section 2.3: any bracketing of the affine composition equals the
    sequential result.  Checks every prefix (so every o_t) and hT."""
    rng = np.random.default_rng(seed)
    q, k, v, la, be = _rand_inputs(rng, 1, 1, T, dk, dv)
    h0 = rng.standard_normal((1, 1, dv, dk))
    o, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib)
    A, Bm = _affine_maps(k[0, 0], v[0, 0], la[0, 0], be[0, 0])
    err = 0.0
    for _ in range(trials):
        for t in range(1, T + 1):
            At, Bt = _fold(A, Bm, 0, t, rng)
            St = h0[0, 0] @ At + Bt
            err = max(err, _rel(St @ q[0, 0, t - 1], o[0, 0, t - 1]))
            if t == T:
                err = max(err, _rel(St, hT[0, 0]))
    return err


def reversed_order_error(lib, dk=4, dv=4, T=13, seed=3):
    """How far the wrong composition order lands from the oracle (must be
    large: it shows the bracketing pin has teeth)."""
    rng = np.random.default_rng(seed)
    q, k, v, la, be = _rand_inputs(rng, 1, 1, T, dk, dv)
    h0 = rng.standard_normal((1, 1, dv, dk))
    _, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib)
    A, Bm = _affine_maps(k[0, 0], v[0, 0], la[0, 0], be[0, 0])
    Ar, Br = _fold(A, Bm, 0, T, rng, reverse=True)
    return _rel(h0[0, 0] @ Ar + Br, hT[0, 0])


def pin_t1_closed_form(lib, dk=5, dv=7, seed=4):
    """T = 1: S_1 = alpha h0 (I - beta k k^T) + beta v k^T, o = S_1 q."""
    rng = np.random.default_rng(seed)
    q, k, v, la, be = _rand_inputs(rng, 1, 1, 1, dk, dv, unit_k=False)
    h0 = rng.standard_normal((1, 1, dv, dk))
    o, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib)
    kk = k[0, 0, 0]
    S1 = (np.exp(la[0, 0, 0]) * h0[0, 0] @ (np.eye(dk) - be[0, 0, 0] * np.outer(kk, kk))
          + be[0, 0, 0] * np.outer(v[0, 0, 0], kk))
    return max(_rel(hT[0, 0], S1), _rel(o[0, 0, 0], S1 @ q[0, 0, 0]))


def _orthogonal_keys(rng, T, dk):
    """T <= dk mutually orthogonal keys with random (non-unit) norms."""
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    scale = rng.uniform(0.3, 2.0, size=T)
    return Qm[:, :T].T * scale[:, None]


def pin_linear_attention(lib, dk=8, dv=5, T=8, seed=5):
    """Mutually orthogonal keys and h0 = 0 make the erase term vanish
    (S_{t-1} k_t = 0), leaving gated linear attention with write strength
    beta:  o_t = sum_{j<=t} (prod_{j<i<=t} alpha_i) beta_j (k_j . q_t) v_j.
    With alpha = 1 this is the dense causal form (Q K^T * mask) diag(beta) V."""
    rng = np.random.default_rng(seed)
    k = _orthogonal_keys(rng, T, dk)[None, None]
    q = rng.standard_normal((1, 1, T, dk))
    v = rng.standard_normal((1, 1, T, dv))
    be = rng.uniform(0.05, 0.95, size=(1, 1, T))
    err = 0.0
    # ungated: dense masked matmul
    la = np.zeros((1, 1, T))
    o, hT = oracle.gdn_fwd(q, k, v, la, be, None, lib=lib)
    mask = np.tril(np.ones((T, T)))
    o_ref = ((q[0, 0] @ k[0, 0].T) * mask) @ (be[0, 0][:, None] * v[0, 0])
    hT_ref = (be[0, 0][:, None] * v[0, 0]).T @ k[0, 0]
    err = max(err, _rel(o[0, 0], o_ref), _rel(hT[0, 0], hT_ref))
    # gated: decay matrix D[t, j] = exp(sum_{j<i<=t} log_alpha_i) for j <= t
    la = -rng.uniform(0.05, 0.8, size=(1, 1, T))
    o, hT = oracle.gdn_fwd(q, k, v, la, be, None, lib=lib)
    c = np.cumsum(la[0, 0])
    D = np.exp(c[:, None] - c[None, :]) * mask
    o_ref = ((q[0, 0] @ k[0, 0].T) * D) @ (be[0, 0][:, None] * v[0, 0])
    hT_ref = (D[-1][:, None] * be[0, 0][:, None] * v[0, 0]).T @ k[0, 0]
    err = max(err, _rel(o[0, 0], o_ref), _rel(hT[0, 0], hT_ref))
    return err


def pin_linearity(lib, dk=5, dv=4, T=17, seed=6):
    """For fixed (q, k, alpha, beta) the map (h0, V) -> (o, hT) is linear."""
    rng = np.random.default_rng(seed)
    q, k, va, la, be = _rand_inputs(rng, 1, 2, T, dk, dv)
    vb = rng.standard_normal(va.shape)
    ha = rng.standard_normal((1, 2, dv, dk))
    hb = rng.standard_normal((1, 2, dv, dk))
    c = 0.37
    oa, Ha = oracle.gdn_fwd(q, k, va, la, be, ha, lib=lib)
    ob, Hb = oracle.gdn_fwd(q, k, vb, la, be, hb, lib=lib)
    oc, Hc = oracle.gdn_fwd(q, k, va + c * vb, la, be, ha + c * hb, lib=lib)
    return max(_rel(oc, oa + c * ob), _rel(Hc, Ha + c * Hb))


def pin_continuation(lib, dk=6, dv=5, T1=7, T2=10, seed=7):
    """fwd(T1) then fwd(T2, h0 = hT) equals fwd(T1 + T2): the state is the
    whole carried context."""
    rng = np.random.default_rng(seed)
    q, k, v, la, be = _rand_inputs(rng, 2, 1, T1 + T2, dk, dv)
    h0 = rng.standard_normal((2, 1, dv, dk))
    o, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib)
    s1 = np.s_[:, :, :T1]
    s2 = np.s_[:, :, T1:]
    o1, h1 = oracle.gdn_fwd(q[s1], k[s1], v[s1], la[s1], be[s1], h0, lib=lib)
    o2, h2 = oracle.gdn_fwd(q[s2], k[s2], v[s2], la[s2], be[s2], h1, lib=lib)
    return max(_rel(np.concatenate([o1, o2], axis=2), o), _rel(h2, hT))


def pin_varlen_split(lib, dk=4, dv=6, H=2, seed=8):
    """A packed batch equals independent dense calls per sequence, including
    empty sequences."""
    rng = np.random.default_rng(seed)
    lens = [5, 0, 1, 9, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    TT = int(cu[-1])
    q = rng.standard_normal((H, TT, dk))
    k = rng.standard_normal((H, TT, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((H, TT, dv))
    la = -rng.uniform(0.0, 1.0, size=(H, TT))
    be = rng.uniform(0.0, 1.0, size=(H, TT))
    h0 = rng.standard_normal((len(lens), H, dv, dk))
    o, hT = oracle.gdn_fwd_varlen(q, k, v, la, be, cu, h0, lib=lib)
    err = 0.0
    for n in range(len(lens)):
        a, b = int(cu[n]), int(cu[n + 1])
        od, hd = oracle.gdn_fwd(q[None, :, a:b], k[None, :, a:b], v[None, :, a:b],
                                la[None, :, a:b], be[None, :, a:b], h0[n][None], lib=lib)
        if b > a:
            err = max(err, _rel(o[:, a:b], od[0]))
        err = max(err, _rel(hT[n], hd[0]))
    return err


def pin_norm_bound(lib, dk=6, dv=4, T=25, seed=9):
    """Unit k, beta in (0,1): (I - beta k k^T) is a contraction, so
    ||S_t||_F <= alpha_t ||S_{t-1}||_F + beta_t ||v_t||.  Returns the largest
    violation (0 when the bound holds), checked through prefix runs."""
    rng = np.random.default_rng(seed)
    q, k, v, la, be = _rand_inputs(rng, 1, 1, T, dk, dv)
    h0 = rng.standard_normal((1, 1, dv, dk))
    prev = np.linalg.norm(h0)
    worst = 0.0
    for t in range(1, T + 1):
        s = np.s_[:, :, :t]
        _, hT = oracle.gdn_fwd(q[s], k[s], v[s], la[s], be[s], h0, lib=lib)
        cur = np.linalg.norm(hT)
        bound = np.exp(la[0, 0, t - 1]) * prev + be[0, 0, t - 1] * np.linalg.norm(v[0, 0, t - 1])
        worst = max(worst, (cur - bound) / max(bound, 1e-300))
        prev = cur
    return max(worst, 0.0)


def _gla_closed_form(q, k, v, la, be, h0):
    """Gated linear attention written out as masked decayed attention
    ("线性注意力机制与Gated DeltaNet的优化实践" sections 2.2-2.3 unrolled):
    o_t = sum_{s<=t} exp(G_t - G_s) beta_s (q_t . k_s) v_s + exp(G_t) h0 q_t,
    hT = exp(G_T) h0 + sum_s exp(G_T - G_s) beta_s v_s k_s^T, G the
    cumulative log gate."""
    T = la.shape[-1]
    if T == 0:
        dv, dk = v.shape[-1], q.shape[-1]
        o = np.zeros(q.shape[:-1] + (dv,))
        hT = np.zeros(q.shape[:2] + (dv, dk)) if h0 is None else h0.copy()
        return o, hT
    G = np.cumsum(la, axis=-1)                                     # [B,H,T]
    mask = np.tril(np.ones((T, T)))
    dec = np.exp(G[..., :, None] - G[..., None, :]) * mask         # [B,H,T,T]
    P = np.einsum("bhtd,bhsd->bhts", q, k) * dec * be[..., None, :]
    o = np.einsum("bhts,bhsi->bhti", P, v)
    hT = np.einsum("bhs,bhsi,bhsj->bhij", np.exp(G[..., -1:] - G) * be, v, k)
    if h0 is not None:
        o = o + np.exp(G)[..., None] * np.einsum("bhij,bhtj->bhti", h0, q)
        hT = hT + np.exp(G[..., -1])[..., None, None] * h0
    return o, hT


def pin_gla_closed_form(lib, dk=5, dv=4, T=13, seed=21):
    """The oracle's gated linear attention equals its unrolled closed form,
    with an initial state, gates and write strengths drawn at random."""
    rng = np.random.default_rng(seed)
    q, k, v, la, be = _rand_inputs(rng, 2, 2, T, dk, dv, unit_k=False)
    h0 = rng.standard_normal((2, 2, dv, dk))
    o, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib, erase=False)
    o_ref, hT_ref = _gla_closed_form(q, k, v, la, be, h0)
    return max(_rel(o, o_ref), _rel(hT, hT_ref))


def pin_gla_linear_attention(lib, dk=4, dv=6, T=11, seed=22):
    """alpha = beta = 1, no initial state: plain linear attention,
    z_i = sum_{j<=i} (q_i . k_j) v_j (the first formula of section 2.2),
    i.e. the causally masked (Q K^T) V."""
    rng = np.random.default_rng(seed)
    q, k, v, _, _ = _rand_inputs(rng, 1, 1, T, dk, dv, unit_k=False)
    ones = np.ones((1, 1, T))
    o, hT = oracle.gdn_fwd(q, k, v, 0 * ones, ones, None, lib=lib, erase=False)
    o_ref = np.tril(q[0, 0] @ k[0, 0].T) @ v[0, 0]
    hT_ref = v[0, 0].T @ k[0, 0]
    return max(_rel(o[0, 0], o_ref), _rel(hT[0, 0], hT_ref))


def pin_gla_equals_delta_on_orthogonal_keys(lib, dk=8, dv=5, T=8, seed=23):
    """With a zero initial state and mutually orthogonal keys the delta rule
    never erases anything (S_{t-1} k_t = 0), so both loops must agree."""
    rng = np.random.default_rng(seed)
    q, _, v, la, be = _rand_inputs(rng, 1, 1, T, dk, dv)
    k = _orthogonal_keys(rng, T, dk)[None, None]
    a = oracle.gdn_fwd(q, k, v, la, be, None, lib=lib)
    b = oracle.gdn_fwd(q, k, v, la, be, None, lib=lib, erase=False)
    return max(_rel(b[0], a[0]), _rel(b[1], a[1]))


def pin_gla_varlen_split(lib, dk=4, dv=3, H=2, seed=24):
    """Packed gated linear attention equals per-sequence dense calls."""
    rng = np.random.default_rng(seed)
    lens = [5, 0, 9, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    TT = int(cu[-1])
    q = rng.standard_normal((H, TT, dk))
    k = rng.standard_normal((H, TT, dk))
    v = rng.standard_normal((H, TT, dv))
    la = -rng.uniform(0, 1, (H, TT))
    be = rng.uniform(0, 1, (H, TT))
    h0 = rng.standard_normal((len(lens), H, dv, dk))
    o, hT = oracle.gdn_fwd_varlen(q, k, v, la, be, cu, h0, lib=lib, erase=False)
    worst = 0.0
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        s = np.s_[:, a:b]
        od, hd = _gla_closed_form(q[s][None], k[s][None], v[s][None], la[s][None],
                                  be[s][None], h0[n][None])
        worst = max(worst, _rel(hT[n], hd[0]))
        if b > a:
            worst = max(worst, _rel(o[:, a:b], od[0]))
    return worst


def _vg_inputs(rng, B, H, T, dk, dv):
    q, k, v, _, be = _rand_inputs(rng, B, H, T, dk, dv)
    la = -np.log1p(np.exp(rng.standard_normal((B, H, T, dk)))) * 0.5   # a gate per key dimension
    return q, k, v, la, be


def pin_vg_scalar_reduction(lib, dk=5, dv=4, T=12, seed=31):
    """A per-dimension gate whose entries are all equal is the scalar gate:
    the vector-gate loop must agree with the scalar loops, with and without
    the erase term."""
    rng = np.random.default_rng(seed)
    q, k, v, la, be = _rand_inputs(rng, 1, 2, T, dk, dv)
    h0 = rng.standard_normal((1, 2, dv, dk))
    lav = np.repeat(la[..., None], dk, axis=-1)
    worst = 0.0
    for erase in (True, False):
        a = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib, erase=erase)
        b = oracle.gdn_fwd(q, k, v, lav, be, h0, lib=lib, erase=erase, vector_gate=True)
        worst = max(worst, _rel(b[0], a[0]), _rel(b[1], a[1]))
    return worst


def _vg_affine_maps(k, v, la, be, erase=True):
    """Per-token maps S -> S A_t + B_t with a diagonal gate: A_t =
    diag(alpha_t) (I - beta_t k k^T) (the decay acts on the old state first),
    B_t = beta_t v_t k_t^T; section 2.2's extra diagonal factor."""
    T, dk = k.shape
    A = np.empty((T, dk, dk))
    Bm = np.empty((T, v.shape[1], dk))
    for t in range(T):
        E = np.eye(dk) - (be[t] * np.outer(k[t], k[t]) if erase else 0.0)
        A[t] = np.diag(np.exp(la[t])) @ E
        Bm[t] = be[t] * np.outer(v[t], k[t])
    return A, Bm


def pin_vg_bracketing(lib, dk=4, dv=3, T=11, seed=32, trials=4):
    """Section 2.3 with the diagonal factor: any bracketing of the explicit
    affine maps equals the vector-gate loop, at every prefix, with and
    without the erase term."""
    rng = np.random.default_rng(seed)
    q, k, v, la, be = _vg_inputs(rng, 1, 1, T, dk, dv)
    h0 = rng.standard_normal((1, 1, dv, dk))
    err = 0.0
    for erase in (True, False):
        o, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib, erase=erase, vector_gate=True)
        A, Bm = _vg_affine_maps(k[0, 0], v[0, 0], la[0, 0], be[0, 0], erase)
        for _ in range(trials):
            for t in range(1, T + 1):
                At, Bt = _fold(A, Bm, 0, t, rng)
                St = h0[0, 0] @ At + Bt
                err = max(err, _rel(St @ q[0, 0, t - 1], o[0, 0, t - 1]))
                if t == T:
                    err = max(err, _rel(St, hT[0, 0]))
    return err


def pin_vg_beta_zero(lib, dk=5, dv=3, T=9, seed=33):
    """beta = 0: each key dimension j of the state only decays,
    S_t[:, j] = exp(sum_{i<=t} log_alpha_i[j]) h0[:, j]."""
    rng = np.random.default_rng(seed)
    q, k, v, la, _ = _vg_inputs(rng, 1, 2, T, dk, dv)
    be = np.zeros(la.shape[:-1])
    h0 = rng.standard_normal((1, 2, dv, dk))
    o, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib, vector_gate=True)
    cum = np.exp(np.cumsum(la, axis=2))                               # [1,2,T,dk]
    o_ref = np.einsum("bhij,bhtj,bhtj->bhti", h0, cum, q)
    hT_ref = h0 * cum[:, :, -1][:, :, None, :]
    return max(_rel(o, o_ref), _rel(hT, hT_ref))


def pin_vg_varlen_split(lib, dk=4, dv=3, H=2, seed=34):
    """Packed vector-gate batches equal per-sequence dense calls."""
    rng = np.random.default_rng(seed)
    lens = [6, 0, 8, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    TT = int(cu[-1])
    q = rng.standard_normal((H, TT, dk))
    k = rng.standard_normal((H, TT, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((H, TT, dv))
    la = -rng.uniform(0, 1, (H, TT, dk))
    be = rng.uniform(0, 1, (H, TT))
    h0 = rng.standard_normal((len(lens), H, dv, dk))
    o, hT = oracle.gdn_fwd_varlen(q, k, v, la, be, cu, h0, lib=lib, vector_gate=True)
    worst = 0.0
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        s = np.s_[:, a:b]
        od, hd = oracle.gdn_fwd(q[s][None], k[s][None], v[s][None], la[s][None], be[s][None],
                                h0[n][None], lib=lib, vector_gate=True)
        worst = max(worst, _rel(hT[n], hd[0]))
        if b > a:
            worst = max(worst, _rel(o[:, a:b], od[0]))
    return worst



# ------------------------------------------------------------------ gradient

_FD_STEP = 1e-3
_FD_TOL = 1e-9     # five-point stencil: truncation O(h^4), rounding ~1e-13 / h


def _bwd_inputs(rng, T, dk, dv, H=1):
    q, k, v, la, be = _rand_inputs(rng, 1, H, T, dk, dv)
    h0 = rng.standard_normal((1, H, dv, dk))
    dO = rng.standard_normal((1, H, T, dv))
    dhT = rng.standard_normal((1, H, dv, dk))
    return q, k, v, la, be, h0, dO, dhT


def _loss(lib, xs, dO, dhT, erase):
    q, k, v, la, be, h0 = xs
    if erase:
        o, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib)
    else:
        o, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib, erase=False)
    return float(np.sum(dO * o) + np.sum(dhT * hT))


def pin_bwd_finite_differences(lib, dk=4, dv=3, T=7, seed=51, erase=True):
    """Each gradient against the five-point central difference of the
    forward loss along a random direction: (-L(x+2hD) + 8L(x+hD) - 8L(x-hD)
    + L(x-2hD)) / 12h  =  <grad, D>."""
    rng = np.random.default_rng(seed)
    q, k, v, la, be, h0, dO, dhT = _bwd_inputs(rng, T, dk, dv)
    xs = [q, k, v, la, be, h0]
    grads = oracle.gdn_bwd(q, k, v, la, be, h0, dO, dhT, lib=lib, erase=erase)
    worst = 0.0
    for i, x in enumerate(xs):
        D = rng.standard_normal(x.shape)
        f = []
        for m in (2, 1, -1, -2):
            ys = list(xs)
            ys[i] = x + m * _FD_STEP * D
            f.append(_loss(lib, ys, dO, dhT, erase))
        fd = (-f[0] + 8 * f[1] - 8 * f[2] + f[3]) / (12 * _FD_STEP)
        an = float(np.sum(grads[i] * D))
        err = abs(fd - an) / max(abs(an), abs(fd), 1e-3)
        worst = max(worst, err / _FD_TOL * PIN_TOL)   # reported on the PIN_TOL scale
    return worst


def pin_bwd_fd_no_erase(lib, **kw):
    return pin_bwd_finite_differences(lib, erase=False, seed=52, **kw)


def pin_bwd_adjoint(lib, dk=5, dv=4, T=11, seed=53):
    """L = <dO, O> + <dhT, hT> is linear in (h0, V), so L = <dV, V> + <dh0, h0>;
    O is linear in q and hT does not depend on it, so <dO, O> = <dq, q>.
    Both modes (with and without the erase term)."""
    rng = np.random.default_rng(seed)
    q, k, v, la, be, h0, dO, dhT = _bwd_inputs(rng, T, dk, dv, H=2)
    worst = 0.0
    for erase in (True, False):
        o, hT = oracle.gdn_fwd(q, k, v, la, be, h0, lib=lib, erase=erase)
        dq, _, dv_, _, _, dh0 = oracle.gdn_bwd(q, k, v, la, be, h0, dO, dhT, lib=lib,
                                              erase=erase)
        L_o, L_h = float(np.sum(dO * o)), float(np.sum(dhT * hT))
        scale = max(abs(L_o) + abs(L_h), 1e-300)
        worst = max(worst,
                    abs(L_o + L_h - float(np.sum(dv_ * v) + np.sum(dh0 * h0))) / scale,
                    abs(L_o - float(np.sum(dq * q))) / max(abs(L_o), 1e-300))
    return worst


def pin_bwd_varlen_split(lib, dk=4, dv=3, H=2, seed=54):
    """Packed gradients equal the per-sequence dense gradients (both modes)."""
    rng = np.random.default_rng(seed)
    lens = [3, 0, 7, 1, 5]
    cu = np.concatenate([[0], np.cumsum(lens)])
    TT = int(cu[-1])
    q, k, v, la, be = (x[0] for x in _rand_inputs(rng, 1, H, TT, dk, dv))
    dO = rng.standard_normal((H, TT, dv))
    h0 = rng.standard_normal((len(lens), H, dv, dk))
    dhT = rng.standard_normal((len(lens), H, dv, dk))
    worst = 0.0
    for erase in (True, False):
        g = oracle.gdn_bwd_varlen(q, k, v, la, be, cu, h0, dO, dhT, lib=lib, erase=erase)
        for n in range(len(lens)):
            a, b = int(cu[n]), int(cu[n + 1])
            gd = oracle.gdn_bwd(q[None, :, a:b], k[None, :, a:b], v[None, :, a:b],
                                la[None, :, a:b], be[None, :, a:b], h0[n][None],
                                dO[None, :, a:b], dhT[n][None], lib=lib, erase=erase)
            for i in range(5):
                if b > a:
                    worst = max(worst, _rel(g[i][:, a:b], gd[i][0]))
            worst = max(worst, _rel(g[5][n], gd[5][0]))
    return worst


ALL_PINS = {
    "beta_zero": pin_beta_zero,
    "exact_recall": pin_exact_recall,
    "bracketing": pin_bracketing,
    "t1_closed_form": pin_t1_closed_form,
    "linear_attention": pin_linear_attention,
    "linearity": pin_linearity,
    "continuation": pin_continuation,
    "varlen_split": pin_varlen_split,
    "norm_bound": pin_norm_bound,
    "gla_closed_form": pin_gla_closed_form,
    "gla_linear_attention": pin_gla_linear_attention,
    "gla_equals_delta_on_orthogonal_keys": pin_gla_equals_delta_on_orthogonal_keys,
    "gla_varlen_split": pin_gla_varlen_split,
    "vg_scalar_reduction": pin_vg_scalar_reduction,
    "vg_bracketing": pin_vg_bracketing,
    "vg_beta_zero": pin_vg_beta_zero,
    "vg_varlen_split": pin_vg_varlen_split,
    "bwd_finite_differences": pin_bwd_finite_differences,
    "bwd_fd_no_erase": pin_bwd_fd_no_erase,
    "bwd_adjoint": pin_bwd_adjoint,
    "bwd_varlen_split": pin_bwd_varlen_split,
}
