"""Hand-worked examples of the recurrence (text fixtures in tests/golden/).

No source page prints a numeric example of the gated delta rule, so each
fixture is a tiny case (d_k = d_v = 2) whose values were worked out on paper
from the page's definition, in dyadic numbers that fp64 holds exactly; the
derivation sits in the fixture's comments next to its citation.  They pin the
oracle to numbers that come from neither its code nor a retyped formula, and
the GPU path to the same numbers through zero padding (extra key and value
dimensions that stay zero leave the recurrence on the first two untouched).
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
FORWARD = ("delta_rule_d2_t3", "gated_linear_attention_d2_t3", "vector_gate_d2_t3")
GRADIENT = "gradient_d2_t1"
# the gradient's output names in the order gdn_bwd returns them
GRAD_NAMES = ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dh0")


def load(name: str) -> dict:
    """Parse one fixture: `name value value ...` lines, `#` starts a comment.
    Arrays come back in the oracle's per-head shapes (fp64)."""
    raw = {}
    with open(os.path.join(GOLDEN_DIR, name + ".txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                raw[line[0]] = [float(x) for x in line[1:]]
    dk, dv, T = (int(raw.pop(n)[0]) for n in ("d_k", "d_v", "T"))
    shapes = {"h0": (dv, dk), "hT": (dv, dk), "dhT": (dv, dk), "dh0": (dv, dk),
              "q": (T, dk), "k": (T, dk), "dq": (T, dk), "dk": (T, dk),
              "v": (T, dv), "o": (T, dv), "dO": (T, dv), "dv": (T, dv),
              "beta": (T,), "dlog_alpha": (T,), "dbeta": (T,)}
    out = {"d_k": dk, "d_v": dv, "T": T}
    for key, vals in raw.items():
        a = np.array(vals, dtype=np.float64)
        if key == "alpha":
            # one gate per token, or one per token and key dimension
            shape = (T,) if a.size == T else (T, dk)
        else:
            shape = shapes[key]
        out[key] = a.reshape(shape)
    out["log_alpha"] = np.log(out["alpha"])
    out["vector_gate"] = out["alpha"].ndim == 2
    out["erase"] = not name.startswith("gated_linear_attention")
    return out


def pad(a: np.ndarray, dims: tuple) -> np.ndarray:
    """Zero-pad the trailing axes of `a` up to `dims` (one size per axis)."""
    width = [(0, 0)] * (a.ndim - len(dims)) + [(0, d - s) for s, d in zip(a.shape[-len(dims):],
                                                                           dims)]
    return np.pad(a, width)


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def oracle_forward_errors(lib, name: str) -> dict:
    """The oracle's dense and packed forward on one fixture against its
    values; the packed call holds the sequence twice, both from h0."""
    import oracle
    g = load(name)
    one = lambda a: a[None, None]  # noqa: E731
    kw = dict(lib=lib, erase=g["erase"], vector_gate=g["vector_gate"])
    o, hT = oracle.gdn_fwd(one(g["q"]), one(g["k"]), one(g["v"]), one(g["log_alpha"]),
                           one(g["beta"]), one(g["h0"]), **kw)
    two = lambda a: np.concatenate([a, a])[None]  # noqa: E731
    T = g["T"]
    ov, hv = oracle.gdn_fwd_varlen(two(g["q"]), two(g["k"]), two(g["v"]), two(g["log_alpha"]),
                                   two(g["beta"]), np.array([0, T, 2 * T]),
                                   np.stack([g["h0"], g["h0"]])[:, None], **kw)
    return {"o": rel(o[0, 0], g["o"]), "hT": rel(hT[0, 0], g["hT"]),
            "o_packed": rel(ov[0], np.concatenate([g["o"], g["o"]])),
            "hT_packed": max(rel(hv[n, 0], g["hT"]) for n in range(2))}


def oracle_gradient_errors(lib) -> dict:
    """The oracle's gradient on the hand-worked one-token fixture."""
    import oracle
    g = load(GRADIENT)
    one = lambda a: a[None, None]  # noqa: E731
    got = oracle.gdn_bwd(one(g["q"]), one(g["k"]), one(g["v"]), one(g["log_alpha"]),
                         one(g["beta"]), one(g["h0"]), one(g["dO"]), one(g["dhT"]), lib=lib)
    return {n: rel(a[0, 0], g[n]) for n, a in zip(GRAD_NAMES, got)}


def oracle_packed_gradient_errors(lib) -> dict:
    """The gradient fixture packed as two sequences x two heads.  Head 1 has
    v and h0 doubled: every state doubles (the states are linear in (h0, v)
    jointly), so dq, dk, dlog_alpha and dbeta double while dv and dh0, which
    depend only on dO, dhT, q and the gates, stay as they are.  Distinct
    heads make a mix-up of the (sequence, head) state offsets visible."""
    import oracle
    g = load(GRADIENT)
    scale = {"dq": 2.0, "dk": 2.0, "dv": 1.0, "dlog_alpha": 2.0, "dbeta": 2.0, "dh0": 1.0}
    heads = lambda a, b: np.stack([np.concatenate([a, a]), np.concatenate([b, b])])  # noqa: E731
    same = lambda n: heads(g[n], g[n])  # noqa: E731
    h0 = np.stack([np.stack([g["h0"], 2 * g["h0"]])] * 2)          # [N=2][H=2]
    dhT = np.stack([np.stack([g["dhT"], g["dhT"]])] * 2)
    got = oracle.gdn_bwd_varlen(same("q"), same("k"), heads(g["v"], 2 * g["v"]),
                                same("log_alpha"), same("beta"), np.array([0, 1, 2]), h0,
                                same("dO"), dhT, lib=lib)
    errs = {}
    for n, a in zip(GRAD_NAMES, got):
        for h in range(2):
            want = g[n] * (scale[n] if h else 1.0)
            if n == "dh0":
                errs["dh0[h%d]" % h] = max(rel(a[s, h], want) for s in range(2))
            else:
                errs["%s[h%d]" % (n, h)] = rel(a[h], np.concatenate([want, want]))
    return errs
