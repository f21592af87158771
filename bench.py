"""Throughput benchmark of the gated delta rule forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-erase] [--backward]
                    [--vector-gate]

One step = one gdn_fwd call (every stage of the chunked forward pass) over the
whole synthetic batch of the workload (default: B=4, H=16, T=4096,
d_k=d_v=128, bf16 I/O, fp32 state).  Inputs are resident in HBM before the
timed region; L2 is flushed (a 256 MiB write) before every timed step and
each step is timed with CUDA events on the launching stream.  Rank 0 prints
one JSON line.  Under torchrun every rank runs an independent replica of the
workload (the path has no cross-GPU exchange), "scaling": "weak", and the
slowest rank's time is reported.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores (rank 0 only).

--no-erase times gated linear attention (the recurrence without the erase
term); --vector-gate draws a forget gate per key dimension; --backward times
the backward pass (gdn_bwd: the gradient of sum(dO * o) + sum(dhT * hT) for
fixed seeded weights dO, dhT) instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "GDN chunked fwd tokens/s (B·H·T/s) and % of roofline, bf16, d=128, 1×GB300"
UNIT = "tokens/s"
DECODE_METRIC = "GDN decode step tokens/s (B·H/s) and % of roofline, bf16, d=128, 1×GB300"
GLA_METRIC = ("gated linear attention (no erase term) chunked fwd tokens/s (B·H·T/s) and % of "
              "roofline, bf16, d=128, 1×GB300")
VG_METRIC = ("GDN chunked fwd with a forget gate per key dimension tokens/s (B·H·T/s) and % of "
             "roofline, bf16, d=128, 1×GB300")
BWD_METRIC = "GDN chunked bwd tokens/s (B·H·T/s) and % of roofline, bf16, d=128, 1×GB300"
DEFAULT_WORKLOAD = "gdn_fwd_b4_h16_t4096_d128_bf16"
# tf32 tensor rate relative to bf16 (nominal dense figures: 1.1 vs 2.25 PFLOP/s)
TF32_PER_BF16 = 1.1 / 2.25
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--vector-gate", action="store_true",
                    help="a forget gate per key dimension (log_alpha [.., T, d_k])")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (gdn_bwd) instead of the forward")
    ap.add_argument("--no-erase", action="store_true",
                    help="gated linear attention: the recurrence without the erase term")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--host-link", action="store_true",
                    help="measure the host <-> device copy rates that bound the e2e figure "
                         "(pinned and pageable, one and several streams) and exit")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers


def dist_setup(n_gpus):
    """One process per GPU (torchrun env).  NCCL on GPUs; gloo when there is
    no GPU (the CPU tests of this path)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Largest value over all ranks (the slowest rank's time)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, step_ms):
    """Whole-job tokens/s: every rank runs its own replica of the workload
    (weak scaling), timed by the slowest rank."""
    return tokens_per_rank * world / (step_ms * 1e-3)


def workload_shape(name):
    cfg = synth.WORKLOADS[name]
    if cfg.get("kind") == "decode":
        return dict(kind="decode", B=cfg["B"], H=cfg["H"], dk=cfg["dk"], dv=cfg["dv"],
                    io=cfg["io"], tokens=cfg["B"] * cfg["H"], N=cfg["B"], h0=True)
    if "N" in cfg:
        lens = synth.varlen_lengths(cfg["N"], cfg["len_min"], cfg["len_max"], cfg["seed"])
        return dict(kind="varlen", H=cfg["H"], dk=cfg["dk"], dv=cfg["dv"], io=cfg["io"],
                    lengths=lens, tokens=int(lens.sum()) * cfg["H"], N=cfg["N"],
                    h0=cfg["h0_std"] > 0)
    return dict(kind="dense", B=cfg["B"], H=cfg["H"], T=cfg["T"], dk=cfg["dk"], dv=cfg["dv"],
                io=cfg["io"], tokens=cfg["B"] * cfg["H"] * cfg["T"], N=cfg["B"],
                h0=cfg["h0_std"] > 0)


def algorithmic(shape):
    """Compulsory HBM bytes and chunked-algorithm FLOPs of one forward call.

    Bytes: every q, k, v, o element once at the I/O width, two fp32 gates per
    token-head, h0 (when given) read once and hT written once per
    (sequence, head).  FLOPs per token-head, counting full 64x64 chunk tiles
    as issued: 6*C*d_k + 4*C*d_v + 6*d_k*d_v (C = 64)."""
    io = 2 if shape["io"] == "bf16" else 4
    dk, dv, C = shape["dk"], shape["dv"], 64
    th = shape["tokens"]
    if shape["kind"] == "decode":
        # one token per (sequence, head): its q, k, v, o and gates, and the
        # fp32 state read and written once; 6 d_k d_v FLOPs (S k, S q, update)
        return th * ((2 * dk + 2 * dv) * io + 8 + 2 * dk * dv * 4), th * 6 * dk * dv
    seqheads = shape["N"] * shape["H"]
    state = seqheads * dk * dv * 4
    gates = 4 * (1 + dk) if VECTOR_GATE else 8
    by = th * ((2 * dk + 2 * dv) * io + gates) + state * (2 if shape["h0"] else 1)
    flops = th * (6 * C * dk + 4 * C * dv + 6 * dk * dv)
    return by, flops


def kernel_bytes(kernel, shape, call_bytes):
    """Compulsory bytes the timed kernel itself moves.  The fused forward
    kernel reads q, k, v, log_alpha and h0 and writes o and hT: the call's
    compulsory bytes less beta, which only the chunk-prep kernel reads."""
    if kernel == "k_gdn_fused":
        return call_bytes - 4 * shape["tokens"]
    return call_bytes


def algorithmic_bwd(shape):
    """Compulsory HBM bytes of one backward call and the FLOPs of its per-chunk
    gradient kernel (one tf32 product each; fp32 I/O issues three).

    Bytes: q, k, v, dO read and dq, dk, dv written once at the I/O width, the
    two gates read and their two gradients written (fp32), h0 and dhT read and
    dh0 written once per (sequence, head).  FLOPs of k_bwd_chunk per
    chunk-head (C = 64), as its loops issue them: the three d_v contractions
    against the chunk states (3 C d_k d_v), the two C x C ones over d_v and
    T^T dV' (2.5 C^2 d_v), eight C x C x d_k products of the gradient algebra
    (about 4 C^2 d_k) and the inverse and its adjoint (about C^3 / 2); two
    FLOPs per multiply-add."""
    io = 2 if shape["io"] == "bf16" else 4
    dk, dv, C = shape["dk"], shape["dv"], 64
    th = shape["tokens"]
    seqheads = shape["N"] * shape["H"]
    state = seqheads * dk * dv * 4
    by = th * ((4 * dk + 3 * dv) * io + 16) + state * (3 if shape["h0"] else 2)
    chunks = -(-th // C)
    fma = 3 * C * dk * dv + 2.5 * C * C * dv + 4 * C * C * dk + C ** 3 / 2
    return by, chunks * fma * 2


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# how the dominant kernel's duration is taken (the step time has no events
# between the call's kernels)
KERNEL_TIMING = "a second pass over the timed steps with per-kernel CUDA events"

# the sources each timed kernel is built from (its file and the headers it includes)
KERNEL_SOURCES = {
    "k_gdn_fused": ["gdn_fused.cu", "tc_common.cuh", "tc_ptx.cuh", "gdn_check.cuh", "gdn_internal.h"],
    "k_gdn_ut": ["gdn_ut.cu", "gdn_utw.cuh", "gdn_inv.cuh", "tc_common.cuh", "tc_ptx.cuh",
                 "gdn_check.cuh", "gdn_internal.h"],
    "k_gdn_utw": ["gdn_ut.cu", "gdn_utw.cuh", "gdn_inv.cuh", "tc_common.cuh", "tc_ptx.cuh",
                  "gdn_check.cuh", "gdn_internal.h"],
    "k_gdn_tc": ["gdn_tc.cu", "gdn_tcw.cuh", "gdn_utw.cuh", "gdn_inv.cuh", "gdn_bwd_tc.h",
                 "tc_common.cuh", "tc_ptx.cuh", "gdn_check.cuh", "gdn_internal.h"],
    "k_gdn_tc_ov": ["gdn_tc.cu", "gdn_tcw.cuh", "gdn_utw.cuh", "gdn_inv.cuh", "gdn_bwd_tc.h",
                    "tc_common.cuh", "tc_ptx.cuh", "gdn_check.cuh", "gdn_internal.h"],
    "k_gdn_tcw": ["gdn_tc.cu", "gdn_tcw.cuh", "gdn_utw.cuh", "gdn_inv.cuh", "gdn_bwd_tc.h",
                  "tc_common.cuh", "tc_ptx.cuh", "gdn_check.cuh", "gdn_internal.h"],
    "k_gdn_tcw_ov": ["gdn_tc.cu", "gdn_tcw.cuh", "gdn_utw.cuh", "gdn_inv.cuh", "gdn_bwd_tc.h",
                     "tc_common.cuh", "tc_ptx.cuh", "gdn_check.cuh", "gdn_internal.h"],
    "k_bwd_dstate_tc": ["gdn_bwd_tc.cu", "gdn_bwd_tc.h", "tc_common.cuh", "tc_ptx.cuh", "gdn_check.cuh",
                        "gdn_internal.h"],
    "k_gdn_prep": ["gdn_prep.cu", "gdn_inv.cuh", "gdn_bwd_tc.h", "tc_ptx.cuh", "gdn_check.cuh",
                   "gdn_internal.h"],
    "k_gdn_decode": ["gdn_decode.cu", "gdn_internal.h"],
    "k_bwd_chunk": ["gdn_bwd.cu", "gdn_internal.h", "gdn_mma.cuh", "gdn_tile.cuh"],
    "k_state_mma": ["gdn_simt.cu", "gdn_internal.h", "gdn_mma.cuh", "gdn_tile.cuh"],
    "k_state_vg": ["gdn_simt.cu", "gdn_internal.h", "gdn_mma.cuh", "gdn_tile.cuh"],
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_deltanet_recurrence_gdn_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel) or sorted(
        f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for f in files + ["../../include/gdn.h"]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is missing or was taken on different kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash(kernel)
    for line in open(p):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#"):
            k, w, src_hash, traffic = parts[:4]
            if k == kernel and w == workload and src_hash == want:
                return float(traffic)
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        load = [x for x in sm if mx and x >= 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ our GPU arm


def make_inputs(name, device):
    if VECTOR_GATE:
        return synth.make_workload(name, device=device, vector_gate=True)
    return synth.make_workload(name, device=device)


def is_decode(x):
    return x.meta.get("kind") == "decode"


def metric_for(shape):
    if BACKWARD:
        return BWD_METRIC
    if VECTOR_GATE:
        return VG_METRIC
    if NO_ERASE:
        return GLA_METRIC
    return DECODE_METRIC if shape["kind"] == "decode" else METRIC


NO_ERASE = False   # set from --no-erase
BACKWARD = False   # set from --backward
VECTOR_GATE = False   # set from --vector-gate
_BWD_WEIGHTS = {}


def bwd_weights(x):
    """Seeded output weights dO (I/O dtype) and dhT (fp32) of the backward."""
    key = (x.q.device, tuple(x.v.shape))
    if key not in _BWD_WEIGHTS:
        g = torch.Generator(device=x.q.device).manual_seed(1234)
        n_states = x.h0.shape[:2] if x.h0 is not None else (
            (x.meta["N"], x.meta["H"]) if x.cu_seqlens is not None else x.q.shape[:2])
        dout = torch.randn(x.v.shape, generator=g, device=x.q.device).to(x.q.dtype)
        dhT = torch.randn((*n_states, x.v.shape[-1], x.q.shape[-1]), generator=g,
                          device=x.q.device)
        _BWD_WEIGHTS[key] = (dout, dhT)
    return _BWD_WEIGHTS[key]


def call(gdn, x, out=None):
    if BACKWARD:
        dout, dhT = bwd_weights(x)
        if x.cu_seqlens is not None:
            g = gdn.gdn_bwd_varlen(x.q, x.k, x.v, x.log_alpha, x.beta, x.cu_seqlens, x.h0,
                                   dout, dhT, erase=not NO_ERASE)
        else:
            g = gdn.gdn_bwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, dout, dhT,
                            erase=not NO_ERASE)
        return g[0], g[5]
    if NO_ERASE:
        if x.cu_seqlens is not None:
            return gdn.gdn_fwd_varlen(x.q, x.k, x.v, x.log_alpha, x.beta, x.cu_seqlens, x.h0,
                                      out=out, erase=False)
        return gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, out=out, erase=False)
    if is_decode(x):
        return gdn.gdn_decode(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, slots=x.slots,
                              out=out), x.h0
    if x.cu_seqlens is not None:
        return gdn.gdn_fwd_varlen(x.q, x.k, x.v, x.log_alpha, x.beta, x.cu_seqlens, x.h0,
                                  out=out)
    return gdn.gdn_fwd(x.q, x.k, x.v, x.log_alpha, x.beta, x.h0, out=out)


def run_ours(args, world, rank, local):
    import gated_deltanet_recurrence_gdn_gb300 as gdn
    gdn.load()
    dev = torch.device("cuda", local)
    shape = workload_shape(args.workload)
    x = make_inputs(args.workload, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # the clock sampler starts first: its start-up pause then falls before the
    # warm-up instead of idling the GPU right before the timed steps
    clocks = ClockSampler(local)
    clocks.__enter__()
    try:
        out = torch.empty_like(x.v)
        for _ in range(max(args.warmup, 3)):
            flush.zero_()
            call(gdn, x, out=out)
        gdn.sync_check(dev)

        # ---- device-timed region: inputs resident, L2 flushed before each
        # step.  The step time is taken with events around each call only:
        # the library's per-kernel timer records events between the call's
        # kernels, which puts a stream dependency between them and lengthens
        # the step.  The dominant kernel's duration comes from a second pass
        # over the same steps with that timer on.
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        launches0 = gdn.kernel_launches()
        barrier(world)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            call(gdn, x, out=out)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    finally:
        clocks.__exit__(None, None, None)
    barrier(world)
    wall = time.perf_counter() - t_wall
    launches = gdn.kernel_launches() - launches0
    gdn.kernel_timer(True)
    gdn.kernel_timer_read()
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.zero_()
        call(gdn, x, out=out)
    torch.cuda.synchronize(dev)
    k_ms, k_n, k_name = gdn.kernel_timer_read()
    gdn.kernel_timer(False)
    if k_n == 0 or k_n % args.steps:
        # the same number of timed launches of the dominant kernel in every call
        # (two for a segment scan: its map pass and its output pass), or the
        # mean mixes kernels
        raise RuntimeError("kernel timer: %d launches of %s in %d steps" % (k_n, k_name,
                                                                          args.steps))
    k_per_call = k_n // args.steps
    gdn.sync_check(dev)
    step_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    step_ms = max_over_ranks(step_ms, world)
    kern_ms = max_over_ranks(k_ms / max(k_n, 1), world)

    # ---- end to end: pinned host inputs -> device, forward, result -> host.
    # A decode step keeps its states resident in device memory (a serving
    # loop's state cache): only the token's inputs go in and o comes back.
    dec = is_decode(x)
    src = {k: t for k, t in x.tensors().items() if not (dec and k == "h0")}
    if BACKWARD:
        src["dout"], src["dhT"] = bwd_weights(x)
    host = {k: (None if t is None else t.cpu().pin_memory()) for k, t in src.items()}
    dev_buf = {k: (None if t is None else torch.empty_like(t)) for k, t in src.items()}
    o_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hT_shape = ((shape["N"], shape["H"], shape["dv"], shape["dk"]) if shape["kind"] == "varlen"
                else (shape["B"], shape["H"], shape["dv"], shape["dk"]))
    h_host = None if dec else torch.empty(hT_shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = o_host.numel() * o_host.element_size() + (0 if dec else h_host.numel() * 4)
    g_host = None
    if BACKWARD:
        like = [x.q, x.k, x.v, x.log_alpha, x.beta]
        g_host = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in like]
        g_host.append(torch.empty(hT_shape, dtype=torch.float32).pin_memory())
        d2h = sum(t.numel() * t.element_size() for t in g_host)
    e2e_steps = max(3, min(args.steps, 10))

    dense = shape["kind"] == "dense" and not (NO_ERASE or BACKWARD or VECTOR_GATE)

    def e2e_step():
        if BACKWARD:
            for k_, t in host.items():
                if t is not None:
                    dev_buf[k_].copy_(t, non_blocking=True)
            kw = dict(erase=not NO_ERASE)
            if x.cu_seqlens is not None:
                g = gdn.gdn_bwd_varlen(dev_buf["q"], dev_buf["k"], dev_buf["v"],
                                       dev_buf["log_alpha"], dev_buf["beta"], x.cu_seqlens,
                                       dev_buf["h0"], dev_buf["dout"], dev_buf["dhT"], **kw)
            else:
                g = gdn.gdn_bwd(dev_buf["q"], dev_buf["k"], dev_buf["v"], dev_buf["log_alpha"],
                                dev_buf["beta"], dev_buf["h0"], dev_buf["dout"], dev_buf["dhT"],
                                **kw)
            for hb, t in zip(g_host, g):
                hb.copy_(t, non_blocking=True)
            return
        if dense:
            # the library's host-buffer entry point: it uploads, computes and
            # downloads, pipelined over time slices
            gdn.gdn_fwd_host(host["q"], host["k"], host["v"], host["log_alpha"], host["beta"],
                             host["h0"], out=o_host, final_out=h_host, sync=False)
            return
        for k_, t in host.items():
            if t is not None:
                dev_buf[k_].copy_(t, non_blocking=True)
        y = synth.Inputs(dev_buf["q"], dev_buf["k"], dev_buf["v"], dev_buf["log_alpha"],
                         dev_buf["beta"], x.h0 if dec else dev_buf["h0"], x.cu_seqlens, x.meta,
                         x.slots)
        o, hT = call(gdn, y, out=out)
        o_host.copy_(o, non_blocking=True)
        if not dec:
            h_host.copy_(hT, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)

    by, flops = algorithmic_bwd(shape) if BACKWARD else algorithmic(shape)
    hbm, tf, src = load_peaks()
    # the call's compulsory bytes split over its timed launches: a segment
    # scan's two chain launches together read every input and write every output
    kby = kernel_bytes(k_name, shape, by) / k_per_call
    achieved = kby / (kern_ms * 1e-3) / 1e9
    res = {
        "metric": metric_for(shape),
        "value": job_throughput(shape["tokens"], world, step_ms),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if shape["io"] == "bf16" else "f32",
        "data": "synthetic (seeded; q,k L2-normalised Gaussian, v Gaussian, sigmoid beta, "
                "-softplus log-gates)",
        "config": {"workload": args.workload, "token_heads": shape["tokens"],
                   "d_k": shape["dk"], "d_v": shape["dv"],
                   "chunk": None if shape["kind"] == "decode" else 64,
                   "l2": "flushed before every timed step (256 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "wall_s_timed_region": wall},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_source": src + " (MEASURED_PEAKS.json hbm_gbs)"
                     if src == "measured" else "fallback 6.8 TB/s",
                     "traffic": recorded_traffic(k_name, args.workload),
                     "kernel": k_name, "kernel_ms": kern_ms,
                     "kernel_timing": KERNEL_TIMING, "launches_per_call": k_per_call,
                     "algorithmic_bytes": kby, "algorithmic_flops": flops,
                     "call_bytes": by,
                     "step_frac": by / (step_ms * 1e-3) / 1e9 / hbm,
                     "tensor_frac_of_peak": flops / k_per_call / (kern_ms * 1e-3) / (tf * 1e12)},
        "clocks": clocks.summary(),
        "e2e": {"value": job_throughput(shape["tokens"], world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "impl_used": "decode" if shape["kind"] == "decode" else
                     {1: "simt", 2: "tc"}.get(gdn.last_impl(), "none"),
    }
    if BACKWARD or VECTOR_GATE:
        # the dominant kernel's products run on tf32 tensor cores (mma.sync):
        # its roof is the tf32 rate, the measured bf16 peak times the nominal ratio
        tf32 = tf * TF32_PER_BF16
        ach = flops / k_per_call / (kern_ms * 1e-3) / 1e12
        res["roofline"] = {
            "bound": "tensor", "achieved": ach, "peak": tf32, "unit": "TFLOP/s",
            "frac": ach / tf32,
            "peak_source": "tf32 = %s bf16 peak %.1f TFLOP/s x 1.1/2.25 (nominal ratio)"
                           % (src, tf),
            "traffic": recorded_traffic(k_name, args.workload),
            "kernel": k_name, "kernel_ms": kern_ms, "kernel_timing": KERNEL_TIMING,
            "algorithmic_flops": flops,
            "algorithmic_bytes": by,
            "issued_tf32_products": 3 if shape["io"] == "f32" else 1,
            "step_hbm_frac": by / (step_ms * 1e-3) / 1e9 / hbm,
        }
        res["config"]["pass"] = ("backward (state recomputed)" if BACKWARD
                                 else "forward, a forget gate per key dimension")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.workload, x, args.cpu_seconds)
    elif rank == 0 and world == 1:
        res["cpu_baseline"] = None
    return res


# ------------------------------------------------------------- the oracle


def oracle_sample(name, x, budget_s, max_heads=None):
    """Run the fp64 oracle (1 thread) on whole heads of the workload until
    about budget_s seconds of CPU time; returns (token-heads, seconds, desc)."""
    import oracle
    oracle.build()
    f64 = synth.to_f64
    if is_decode(x):
        units = [(b, h) for b in range(x.q.shape[0]) for h in range(x.q.shape[1])]

        def one(u):
            b, h = u
            args = [f64(t[b, h])[None, None, None] for t in (x.q, x.k, x.v)]
            args += [f64(t[b, h]).reshape(1, 1, 1) for t in (x.log_alpha, x.beta)]
            t0 = time.perf_counter()
            oracle.gdn_fwd(*args, f64(x.h0[b, h])[None, None])
            return 1, time.perf_counter() - t0
    elif BACKWARD and x.cu_seqlens is None:
        dout, dhT = (t.cpu() for t in bwd_weights(x))
        units = [(b, h) for b in range(x.q.shape[0]) for h in range(x.q.shape[1])]

        def one(u):
            b, h = u
            args = [f64(t[b, h])[None, None] for t in (x.q, x.k, x.v, x.log_alpha, x.beta)]
            h0 = None if x.h0 is None else f64(x.h0[b, h])[None, None]
            t0 = time.perf_counter()
            oracle.gdn_bwd(*args, h0, f64(dout[b, h])[None, None], f64(dhT[b, h])[None, None],
                           erase=not NO_ERASE)
            return x.q.shape[2], time.perf_counter() - t0
    elif x.cu_seqlens is not None:
        cu = x.cu_seqlens.cpu().numpy()
        units = [(n, h) for n in range(len(cu) - 1) for h in range(x.q.shape[0])]

        def one(u):
            n, h = u
            a, b = int(cu[n]), int(cu[n + 1])
            s = np.s_[h, a:b]
            args = [f64(t[s])[None, None] for t in (x.q, x.k, x.v, x.log_alpha, x.beta)]
            h0 = None if x.h0 is None else f64(x.h0[n, h])[None, None]
            t0 = time.perf_counter()
            if BACKWARD:
                dout, dhT = (t.cpu() for t in bwd_weights(x))
                oracle.gdn_bwd(*args, h0, f64(dout[s])[None, None], f64(dhT[n, h])[None, None],
                               erase=not NO_ERASE)
            else:
                oracle.gdn_fwd(*args, h0, erase=not NO_ERASE, vector_gate=VECTOR_GATE)
            return b - a, time.perf_counter() - t0
    else:
        units = [(b, h) for b in range(x.q.shape[0]) for h in range(x.q.shape[1])]

        def one(u):
            b, h = u
            args = [f64(t[b, h])[None, None] for t in (x.q, x.k, x.v, x.log_alpha, x.beta)]
            h0 = None if x.h0 is None else f64(x.h0[b, h])[None, None]
            t0 = time.perf_counter()
            oracle.gdn_fwd(*args, h0, erase=not NO_ERASE, vector_gate=VECTOR_GATE)
            return x.q.shape[2], time.perf_counter() - t0

    toks, secs, used = 0, 0.0, 0
    for u in units[: max_heads or len(units)]:
        n, s = one(u)
        toks += n
        secs += s
        used += 1
        if secs >= budget_s:
            break
    return toks, secs, "%d of %d (sequence, head) problems, whole length each" % (used, len(units))


def cpu_baseline(name, x, budget_s):
    toks, secs, desc = oracle_sample(name, x, budget_s)
    return {"value": toks / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": desc + "; fp64 single-threaded C, %.1f s" % secs,
            "host_cpus": os.cpu_count()}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    shape = workload_shape(args.workload)
    x = make_inputs(args.workload, "cpu")
    per_step = max(1.0, min(args.cpu_seconds, 60.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        oracle_sample(args.workload, x, per_step / 4, max_heads=1)
    toks, secs = 0, 0.0
    desc = ""
    for _ in range(args.steps):
        t, s, desc = oracle_sample(args.workload, x, per_step)
        toks += t
        secs += s
    value = toks / secs
    return {
        "metric": metric_for(shape), "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "token_heads": shape["tokens"],
                   "d_k": shape["dk"], "d_v": shape["dv"],
                   "chunk": None if shape["kind"] == "decode" else 64},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "per step: " + desc + " (fp64 single-threaded C)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def host_link(nbytes=256 << 20, reps=5):
    """Copy rates between host and device memory (GB/s, best of `reps`, CUDA
    events on the copying streams): what bounds `e2e`, whose timed region
    moves the step's inputs up and its outputs down."""
    dev = torch.device("cuda", torch.cuda.current_device())
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    pin = torch.ones(nbytes, dtype=torch.uint8).pin_memory()
    pin2 = torch.ones(nbytes, dtype=torch.uint8).pin_memory()
    pag = torch.ones(nbytes, dtype=torch.uint8)

    def rate(fn, moved):
        fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return moved / (best * 1e-3) / 1e9

    def split(n, pairs):
        # n streams, each copying its share of every (dst, src) pair
        cur = torch.cuda.current_stream()
        streams = [torch.cuda.Stream() for _ in range(n)]

        def run():
            ev = cur.record_event()
            for i, st in enumerate(streams):
                st.wait_event(ev)
                with torch.cuda.stream(st):
                    for dst, src in pairs:
                        part = dst.numel() // n
                        dst[i * part:(i + 1) * part].copy_(src[i * part:(i + 1) * part],
                                                           non_blocking=True)
            for st in streams:
                cur.wait_stream(st)
        return run

    out = {"bytes_per_copy": nbytes}
    out["h2d_pinned_gbs"] = rate(lambda: d.copy_(pin, non_blocking=True), nbytes)
    out["d2h_pinned_gbs"] = rate(lambda: pin.copy_(d, non_blocking=True), nbytes)
    out["h2d_pageable_gbs"] = rate(lambda: d.copy_(pag), nbytes)
    out["d2h_pageable_gbs"] = rate(lambda: pag.copy_(d), nbytes)
    for n in (2, 4, 8):
        out["h2d_pinned_%d_streams_gbs" % n] = rate(split(n, [(d, pin)]), nbytes)
    both = [torch.cuda.Stream(), torch.cuda.Stream()]

    def up_and_down():
        cur = torch.cuda.current_stream()
        ev = cur.record_event()
        for st in both:
            st.wait_event(ev)
        with torch.cuda.stream(both[0]):
            d.copy_(pin, non_blocking=True)
        with torch.cuda.stream(both[1]):
            pin2.copy_(d2, non_blocking=True)
        for st in both:
            cur.wait_stream(st)
    out["h2d_plus_d2h_at_once_gbs"] = rate(up_and_down, 2 * nbytes)
    return {k: (round(v, 1) if isinstance(v, float) else v) for k, v in out.items()}


def main():
    global NO_ERASE, BACKWARD, VECTOR_GATE
    args = parse()
    if args.host_link:
        torch.cuda.set_device(0)
        print(json.dumps({"host_link": host_link()}), flush=True)
        return
    NO_ERASE = args.no_erase
    BACKWARD = args.backward
    VECTOR_GATE = args.vector_gate
    if VECTOR_GATE and (BACKWARD or synth.WORKLOADS[args.workload].get("kind") == "decode"):
        raise SystemExit("--vector-gate times the chunked forward only")
    if BACKWARD and synth.WORKLOADS[args.workload].get("kind") == "decode":
        raise SystemExit("--backward needs a chunked workload")
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
