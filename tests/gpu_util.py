"""Helpers shared by the GPU tests: run the CUDA path and the oracle on the
same seeded inputs and compare with the relative max-norm the tolerances are
stated in (max|delta| / max|reference|)."""
from __future__ import annotations

import numpy as np
import torch

import gated_deltanet_recurrence_gdn_gb300 as gdn
import oracle
import synth

# Every GPU test runs with poisoned scratch: blocks the library hands out are
# filled with NaN bytes first, so a kernel that reads scratch nobody wrote
# fails its parity check instead of passing on leftovers of an earlier call.
gdn.set_option(gdn.GDN_OPT_POISON_SCRATCH, 1)

# fp32 I/O: 1e-4 on o and hT; bf16 I/O: 1e-2 on o, 2e-2 on hT.
TOL = {"f32": (1e-4, 1e-4), "bf16": (1e-2, 2e-2)}
ORACLE_THREADS = 16


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if b.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def f64(t):
    return synth.to_f64(t)


def oracle_dense(x, heads=None, T=None):
    """Oracle on a subset of (b, h) heads (list of pairs) and/or a token
    prefix.  Returns (o, hT) stacked over the selected heads."""
    q, k, v, la, be = (f64(t) for t in (x.q, x.k, x.v, x.log_alpha, x.beta))
    h0 = f64(x.h0)
    if heads is None:
        heads = [(b, h) for b in range(q.shape[0]) for h in range(q.shape[1])]
    s = slice(None) if T is None else slice(0, T)
    sel = lambda a: np.stack([a[b, h][s] for b, h in heads])[None]  # noqa: E731
    o, hT = oracle.gdn_fwd(sel(q), sel(k), sel(v), sel(la), sel(be),
                           None if h0 is None else np.stack([h0[b, h] for b, h in heads])[None],
                           threads=ORACLE_THREADS)
    return o[0], hT[0]


def oracle_dense_heads_gpu(x, heads):
    """Like oracle_dense but copying only the selected heads off the device."""
    def sel(t, s=slice(None)):
        return np.stack([f64(t[b, h][s]) for b, h in heads])[None]
    h0 = None if x.h0 is None else np.stack([f64(x.h0[b, h]) for b, h in heads])[None]
    o, hT = oracle.gdn_fwd(sel(x.q), sel(x.k), sel(x.v), sel(x.log_alpha), sel(x.beta), h0,
                           threads=ORACLE_THREADS)
    return o[0], hT[0]


def oracle_dense_prefix_gpu(x, T):
    """Oracle on the first T tokens of every head (outputs are causal, so they
    equal the first T outputs of the full run)."""
    s = np.s_[:, :, :T]
    o, hT = oracle.gdn_fwd(f64(x.q[s]), f64(x.k[s]), f64(x.v[s]), f64(x.log_alpha[s]),
                           f64(x.beta[s]), f64(x.h0), threads=ORACLE_THREADS)
    return o, hT


def oracle_varlen_pairs_gpu(y, pairs):
    """Oracle for selected (sequence, head) pairs of a packed batch, run on
    several host threads.  Returns {(n, h): (o [len, d_v], hT [d_v, d_k])}."""
    from concurrent.futures import ThreadPoolExecutor
    cu = y.cu_seqlens.cpu().numpy().astype(np.int64)
    inputs = {}
    for n, h in pairs:
        a, b = int(cu[n]), int(cu[n + 1])
        sl = np.s_[h, a:b]
        h0 = None if y.h0 is None else f64(y.h0[n, h])[None, None]
        inputs[(n, h)] = (f64(y.q[sl])[None, None], f64(y.k[sl])[None, None],
                          f64(y.v[sl])[None, None], f64(y.log_alpha[sl])[None, None],
                          f64(y.beta[sl])[None, None], h0)

    def run(key):
        o, hT = oracle.gdn_fwd(*inputs[key])
        return key, (o[0, 0], hT[0, 0])

    with ThreadPoolExecutor(max_workers=ORACLE_THREADS) as ex:
        return dict(ex.map(run, list(inputs)))


def sync():
    torch.cuda.synchronize()
