"""Seeded synthetic inputs for the gated delta rule forward pass.

Shared by the oracle side and the CUDA side of tests and the benchmark; it
holds none of the method's arithmetic, only the input recipe:

* q, k ~ N(0, 1), then L2-normalised per token (over d_k);
* v ~ N(0, 1);
* beta = sigmoid(N(0, 1));
* log_alpha = -0.5 * softplus(N(0, 1))        ("fast" decay), or
  log_alpha = -softplus(N(-1, 1))              ("slow" decay, long context);
* with a gate per key dimension (vector_gate=True) log_alpha gets a trailing
  d_k axis, each entry drawn by the same rule independently;
* h0 = 0, or h0 ~ N(0, std^2) per (sequence, head);
* packed variable-length batches draw their lengths uniformly from
  [len_min, len_max] with a seeded numpy generator.

Tensors are drawn in fp32 with a seeded torch generator on the requested
device, then q, k, v are cast to the I/O dtype; gates and h0 stay fp32.
Values drawn on a CUDA device differ from values drawn on the CPU for the same
seed; callers that compare two implementations hand both the SAME tensors
(the oracle gets a host copy widened to fp64 via ``to_f64``).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

# The workloads, by name.  "gdn_fwd_b4_h16_t4096_d128_bf16" is the headline
# throughput workload; the other gdn_fwd ones are parity cases, and the
# gdn_decode one times the single-token step.
WORKLOADS = {
    "gdn_fwd_b1_h1_t256_d64_fp32": dict(B=1, H=1, T=256, dk=64, dv=64, io="f32",
                                        decay="fast", h0_std=0.0, seed=1),
    "gdn_fwd_b4_h16_t4096_d128_bf16": dict(B=4, H=16, T=4096, dk=128, dv=128, io="bf16",
                                           decay="fast", h0_std=0.0, seed=2),
    "gdn_fwd_b8_h8_t8192_d64_bf16_h0": dict(B=8, H=8, T=8192, dk=64, dv=64, io="bf16",
                                            decay="fast", h0_std=0.02, seed=3),
    "gdn_fwd_b1_h16_t131072_d128_bf16": dict(B=1, H=16, T=131072, dk=128, dv=128, io="bf16",
                                             decay="slow", h0_std=0.0, seed=4),
    "gdn_fwd_varlen_n64_h32_dk128_dv256_bf16": dict(N=64, len_min=128, len_max=16384, H=32,
                                                    dk=128, dv=256, io="bf16", decay="fast",
                                                    h0_std=0.02, seed=5),
    # the headline batch at a quarter of its length: the case ncu captures run on
    "gdn_fwd_b4_h16_t1024_d128_bf16": dict(B=4, H=16, T=1024, dk=128, dv=128, io="bf16",
                                           decay="fast", h0_std=0.0, seed=7),
    # the headline shape at twice the batch: more two-CTA chains than a GB300
    # has SMs, the case the forward runs with both d_v halves in one CTA
    "gdn_fwd_b8_h16_t4096_d128_bf16": dict(B=8, H=16, T=4096, dk=128, dv=128, io="bf16",
                                           decay="fast", h0_std=0.0, seed=8),
    # one decode step over 256 sequences x 32 heads: 537 MB of fp32 state
    "gdn_decode_b256_h32_d128_bf16": dict(kind="decode", B=256, H=32, dk=128, dv=128,
                                          io="bf16", decay="fast", state_std=0.02, seed=6),
}

IO_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    log_alpha: torch.Tensor
    beta: torch.Tensor
    h0: torch.Tensor | None
    cu_seqlens: torch.Tensor | None = None   # int32, packed batches only
    meta: dict = field(default_factory=dict)
    slots: torch.Tensor | None = None        # int32 state slots, decode steps only

    def tensors(self):
        return dict(q=self.q, k=self.k, v=self.v, log_alpha=self.log_alpha, beta=self.beta,
                    h0=self.h0)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, g, device, mean=0.0, std=1.0):
    x = torch.empty(shape, dtype=torch.float32, device=device)
    x.normal_(mean=mean, std=std, generator=g)
    return x


def _unit_rows(x):
    # per-token L2 normalisation of the Gaussian draw (part of the recipe)
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def _gates(shape, g, device, decay, la_shape=None):
    beta = torch.sigmoid(_normal(shape, g, device))
    shape = la_shape if la_shape is not None else shape
    if decay == "fast":
        la = -0.5 * torch.nn.functional.softplus(_normal(shape, g, device))
    elif decay == "slow":
        la = -torch.nn.functional.softplus(_normal(shape, g, device, mean=-1.0))
    elif decay == "none":
        la = torch.zeros(shape, dtype=torch.float32, device=device)
    else:
        raise ValueError(decay)
    return la.contiguous(), beta.contiguous()


def make_dense(B, H, T, dk, dv, *, io="bf16", decay="fast", h0_std=0.0, seed=0,
               device="cpu", vector_gate=False) -> Inputs:
    """Dense batch: q,k [B,H,T,dk], v [B,H,T,dv], gates [B,H,T], h0 [B,H,dv,dk]
    (log_alpha [B,H,T,dk] with vector_gate)."""
    g = _gen(device, seed)
    dt = IO_DTYPES[io]
    q = _unit_rows(_normal((B, H, T, dk), g, device)).to(dt)
    k = _unit_rows(_normal((B, H, T, dk), g, device)).to(dt)
    v = _normal((B, H, T, dv), g, device).to(dt)
    la, beta = _gates((B, H, T), g, device, decay, (B, H, T, dk) if vector_gate else None)
    h0 = _normal((B, H, dv, dk), g, device, std=h0_std) if h0_std > 0 else None
    return Inputs(q, k, v, la, beta, h0, None,
                  dict(B=B, H=H, T=T, dk=dk, dv=dv, io=io, decay=decay, h0_std=h0_std,
                       seed=seed, vector_gate=vector_gate))


def varlen_lengths(N, len_min, len_max, seed):
    rng = np.random.default_rng(int(seed))
    return rng.integers(len_min, len_max + 1, size=N).astype(np.int64)


def make_varlen(lengths, H, dk, dv, *, io="bf16", decay="fast", h0_std=0.0, seed=0,
                device="cpu", vector_gate=False) -> Inputs:
    """Packed batch: q,k [H,T_total,dk], v [H,T_total,dv], gates [H,T_total],
    cu_seqlens int32 [N+1], h0 [N,H,dv,dk] (log_alpha [H,T_total,dk] with
    vector_gate)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    TT = int(cu[-1])
    N = len(lengths)
    g = _gen(device, seed)
    dt = IO_DTYPES[io]
    q = _unit_rows(_normal((H, TT, dk), g, device)).to(dt)
    k = _unit_rows(_normal((H, TT, dk), g, device)).to(dt)
    v = _normal((H, TT, dv), g, device).to(dt)
    la, beta = _gates((H, TT), g, device, decay, (H, TT, dk) if vector_gate else None)
    h0 = _normal((N, H, dv, dk), g, device, std=h0_std) if h0_std > 0 else None
    cu_t = torch.tensor(cu, dtype=torch.int32, device=device)
    return Inputs(q, k, v, la, beta, h0, cu_t,
                  dict(N=N, H=H, T_total=TT, dk=dk, dv=dv, io=io, decay=decay,
                       h0_std=h0_std, seed=seed, vector_gate=vector_gate))


def make_decode(B, H, dk, dv, *, io="bf16", decay="fast", state_std=0.02, n_slots=None,
                seed=0, device="cpu") -> Inputs:
    """One decode step: q,k [B,H,dk], v [B,H,dv], gates [B,H], and the fp32
    states in `h0`: [B,H,dv,dk], or a pool [n_slots,H,dv,dk] with `slots` a
    seeded choice of B distinct slots (int32 [B])."""
    g = _gen(device, seed)
    dt = IO_DTYPES[io]
    q = _unit_rows(_normal((B, H, dk), g, device)).to(dt)
    k = _unit_rows(_normal((B, H, dk), g, device)).to(dt)
    v = _normal((B, H, dv), g, device).to(dt)
    la, beta = _gates((B, H), g, device, decay)
    P = B if n_slots is None else n_slots
    state = _normal((P, H, dv, dk), g, device, std=state_std)
    slots = None
    if n_slots is not None:
        perm = np.random.default_rng(int(seed)).permutation(n_slots)[:B]
        slots = torch.tensor(perm, dtype=torch.int32, device=device)
    return Inputs(q, k, v, la, beta, state, None,
                  dict(kind="decode", B=B, H=H, dk=dk, dv=dv, io=io, decay=decay,
                       state_std=state_std, n_slots=n_slots, seed=seed), slots)


def make_workload(name, device="cpu", **override) -> Inputs:
    cfg = dict(WORKLOADS[name])
    cfg.update(override)
    if cfg.get("kind") == "decode":
        return make_decode(cfg["B"], cfg["H"], cfg["dk"], cfg["dv"], io=cfg["io"],
                           decay=cfg["decay"], state_std=cfg["state_std"], seed=cfg["seed"],
                           device=device)
    if "N" in cfg:
        lengths = cfg.pop("lengths", None)
        if lengths is None:
            lengths = varlen_lengths(cfg["N"], cfg["len_min"], cfg["len_max"], cfg["seed"])
        return make_varlen(lengths, cfg["H"], cfg["dk"], cfg["dv"], io=cfg["io"],
                           decay=cfg["decay"], h0_std=cfg["h0_std"], seed=cfg["seed"],
                           device=device, vector_gate=cfg.get("vector_gate", False))
    return make_dense(cfg["B"], cfg["H"], cfg["T"], cfg["dk"], cfg["dv"], io=cfg["io"],
                      decay=cfg["decay"], h0_std=cfg["h0_std"], seed=cfg["seed"],
                      device=device, vector_gate=cfg.get("vector_gate", False))


def to_f64(t):
    """Host fp64 numpy copy of exactly the values a kernel receives."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()
