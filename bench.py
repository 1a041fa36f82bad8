#!/usr/bin/env python
"""Benchmark of the DFlash drafting hot path on GB300.

Default workload: the 9B-shaped DFlash v1 drafter at batch 1 (8 taps of
hidden 4096, 6 layers of 32/8 heads x 128, SwiGLU 12288, vocab 151936,
layers 0-4 sliding over 2048 positions, layer 5 full) over a 4096-token
context. One step is one decode round of the whole hot path:
  fuse the round's 16 committed tap rows (fc + hidden_norm + ring + K/V
  injection into all six layers), draft one block of 16 rows (anchor + 15
  mask rows), top-8 per position, greedy verification against the target's
  logits for the 16 verify rows.
The context grows by 16 rows a step, as a fully accepted decode loop does.

Printed: one JSON line (rank 0). `value` is draft blocks/s over all ranks
(weak scaling: every rank drafts its own stream; batch 1 does not shard, so
ranks are replicas). Weights (3.8 GB) exceed L2 (129 MB), so no flush is
needed between steps.

--impl reference times the CPU oracle (float64 NumPy, one BLAS thread) on the
same workload, on the host cores, as the reference arm.

--workload serve32 | dflash2geom runs a multi-stream round instead (32
streams of the 9B-shaped drafter with contexts of 1024..16384 rows and greedy
verification; 8 streams of the DFlash2-geometry drafter at 8192 rows with
sampling verification). Under torchrun the streams are split into contiguous
groups, one per rank, with the weights replicated; each rank drafts and
verifies its own streams with no collective, and the round's results (accept
lengths and committed tokens) are gathered to rank 0 on the host once the
timing is over. `value` is then stream-blocks/s of all ranks (strong
scaling: the round's streams are fixed as ranks are added).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft blocks/s (block 16) and fused tap rows/s; % of HBM/tensor-core roofline"
UNIT = "blocks/s"
WORKLOAD = (
    "9B-shaped DFlash v1 drafter, batch 1: 8 taps x hidden 4096, 6 layers (32q/8kv x 128, SwiGLU 12288), "
    "vocab 151936, 4096-token context, decode round = 16-row tap fusion + K/V injection, block-16 draft, "
    "top-8, greedy verify"
)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def blas_threads(n=None):
    """Thread count of the BLAS library NumPy loaded, read (and with n, set)
    through that library's own exported calls; (None, None) if no known BLAS
    is loaded. Returns (threads, library path)."""
    import ctypes

    import numpy as np

    np.dot(np.ones((2, 2)), np.ones((2, 2)))  # the BLAS is loaded by now
    names = [
        ("scipy_openblas_get_num_threads64_", "scipy_openblas_set_num_threads64_"),
        ("scipy_openblas_get_num_threads", "scipy_openblas_set_num_threads"),
        ("openblas_get_num_threads64_", "openblas_set_num_threads64_"),
        ("openblas_get_num_threads", "openblas_set_num_threads"),
    ]
    seen = set()
    try:
        with open("/proc/self/maps") as f:
            paths = [ln.split()[-1] for ln in f if len(ln.split()) >= 6]
    except OSError:
        return None, None
    for path in paths:
        if "blas" not in os.path.basename(path).lower() or path in seen:
            continue
        seen.add(path)
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for get, put in names:
            if hasattr(lib, get):
                if n is not None:
                    getattr(lib, put)(int(n))
                return int(getattr(lib, get)()), path
    return None, None


def bench_config(world):
    """The `config` object of the default workload's JSON line: the same for
    the GPU arm and the reference arm (run-dependent numbers go elsewhere)."""
    return {
        "workload": WORKLOAD,
        "streams_per_gpu": 1,
        "context_start": 4096,
        "context_growth_per_step": 16,
        "l2": "no flush: 3.8 GB of weights stream through a 129 MB L2 every step",
        "parallelism": f"replicas x{world}",
    }


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = (
        "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
        "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
        "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"
    )

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True,
            )
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons),
            "samples": len(sm),
        }


# ---------------------------------------------------------------- DRAM traffic from ncu
GEMM_SOURCES = ["gemm.cu", "internal.h", "ptx.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_dram_9b_decode.json")


def gemm_source_hash():
    import hashlib

    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "block_diffusion_speculative_tap_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def gemm_traffic():
    """DRAM bytes (read + write) per GEMM launch of the decode step, from the
    committed ncu capture summary; null when the GEMM source has changed
    since the counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        if d.get("gemm_source_sha256") != gemm_source_hash():
            return None
        return d["dram_bytes_per_launch"]
    except Exception:
        return None


# ---------------------------------------------------------------- other configs
def measure_config(name, dev, pk, steps, dr=None):
    """Supplementary measurements of the parity workloads (not the headline):
    draft stream-blocks/s and its HBM roofline fraction, the LM head's
    TFLOP/s, and verification time, at the workload's streams and contexts."""
    import ctypes as C

    import torch

    import block_diffusion_speculative_tap_gb300 as D
    import synthetic_inputs as SI
    from block_diffusion_speculative_tap_gb300 import _abi as A

    P = SI.preset(name)
    m = P["model"]
    ctx = P["context"]
    S = len(ctx)
    if dr is None:
        w = SI.make_weights(m, P["seed"], device=dev)
        dr = D.Drafter(m, w)
    st = dr.new_state(S, P["ring"])
    for s_ in range(S):  # one stream at a time keeps the tap planes small
        taps = SI.make_taps(m, ctx[s_], P["seed"] + 1 + s_, device=dev)
        st.fuse_taps(taps, [(s_, 0, ctx[s_])])
        del taps
    anchors = SI.anchor_ids(S, m["vocab"], m["mask_token"], P["seed"] + 2, device=dev)
    V = m["vocab"]
    k = P["topk"]
    logits = torch.empty(S * 15, V, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(S * 15, k, dtype=torch.int32, device=dev)
    vals = torch.empty(S * 15, k, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def draft():
        st.draft(anchors, k=k, logits=logits, ids=ids, vals=vals)

    for _ in range(3):
        draft()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        draft()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    A.lib.dflash_trace_enable(1)
    draft()
    torch.cuda.synchronize()
    A.lib.dflash_trace_enable(0)
    tot_b, lm_ms, lm_fl = 0.0, 0.0, 0.0
    per = {}
    for i in range(A.lib.dflash_trace_count()):
        nm, t, b, fl = C.c_char_p(), C.c_float(), C.c_double(), C.c_double()
        if A.lib.dflash_trace_get(i, C.byref(nm), C.byref(t), C.byref(b), C.byref(fl)) == 0:
            tot_b += b.value
            key = nm.value.decode()
            per[key] = per.get(key, 0.0) + t.value
            if key == "gemm.lm_head":
                lm_ms += t.value
                lm_fl += fl.value
    out = {
        "streams": S,
        "context": [min(ctx), max(ctx)],
        "topk": k,
        "draft_stream_blocks_per_s": S * 1e3 / ms,
        "draft_ms": ms,
        "draft_algorithmic_bytes": tot_b,
        "draft_frac_of_hbm_peak": tot_b / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
        "lm_head_tflops": lm_fl / (lm_ms * 1e-3) / 1e12 if lm_ms else None,
        "lm_head_frac_of_bf16_peak": (lm_fl / (lm_ms * 1e-3) / 1e12 / pk["bf16_tflops"]) if lm_ms else None,
        "kernels_ms_traced": {k: round(v, 4) for k, v in sorted(per.items(), key=lambda kv: -kv[1])},
    }
    # verification of the drafted rows against seeded target logits
    tl = SI.make_logits((S, 16, V), P["target_logit_std"], P["seed"] + 3, device=dev)
    if P["verify"] == "greedy":
        def ver():
            D.verify_greedy(ids, tl)
    else:
        T = P.get("temperature", 1.0)
        u = SI.make_uniforms((S, 16, 2), P["seed"] + 5, device=dev)
        draft_ids = ids[:, 0].reshape(S, 15).contiguous()

        def ver():
            D.verify_sample(draft_ids, tl, logits.view(S, 15, V), u, T)
    for _ in range(3):
        ver()
    torch.cuda.synchronize()
    v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    v0.record(stream)
    for _ in range(steps):
        ver()
    v1.record(stream)
    torch.cuda.synchronize()
    vms = v0.elapsed_time(v1) / steps
    vbytes = S * 16 * V * 2 * (1 if P["verify"] == "greedy" else 2)
    out["verify_mode"] = P["verify"]
    out["verify_ms"] = vms
    out["verify_rows_per_s"] = S * 16 * 1e3 / vms
    out["verify_frac_of_hbm_peak"] = vbytes / (vms * 1e-3) / 1e9 / pk["hbm_gbs"]
    if name == "tiny":
        # the tiny drafter's fill of its whole context (fc + hidden_norm + K/V
        # injection), absolute only: its 5 MB of weights stay in L2
        st3 = dr.new_state(S, P["ring"])
        ftaps = SI.make_taps(m, ctx[0], P["seed"] + 1, device=dev)
        for _ in range(3):
            st3.fuse_taps(ftaps, [(0, 0, ctx[0])])
            st3.truncate(0, 0)
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(steps):
            st3.fuse_taps(ftaps, [(0, 0, ctx[0])])
            st3.truncate(0, 0)
        f1.record(stream)
        torch.cuda.synchronize()
        fms = f0.elapsed_time(f1) / steps
        out["fill_rows"] = ctx[0]
        out["fill_ms"] = fms
        out["fused_tap_rows_per_s"] = ctx[0] * 1e3 / fms
        out["note"] = "absolute only: the weights (5.2 MB) are L2-resident, so no roofline fraction is claimed"
        del st3, ftaps
    rc, bits = st.status()
    if rc != 0:
        raise RuntimeError(f"{name}: device status {rc} bits {bits}")
    del st, logits
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- the rows after the draft
def measure_next_rows(dev, pk, steps):
    """The DFlash2 candidate-path selector (32 streams x 15 positions x top-16
    over a 151936-token vocabulary, rank-256 codebooks), tree verification
    (32 streams, 93-node trees of widths 4, 2, 2, 1, 1, 1, 1: the arg-max scan
    of every node's target row and the walk) and the two-tap convolution
    stage (8 streams of the DFlash2 geometry, hidden 5120, 16 groups): each
    timed with CUDA events over `steps` back-to-back calls, with its
    algorithmic bytes (each input and output touched once) against the HBM
    peak."""
    import torch

    import block_diffusion_speculative_tap_gb300 as D
    import synthetic_inputs as SI

    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    out = {}
    S, P, k, V, r = 32, 15, 16, 151936, 256
    logits = SI.make_logits((S * P, V), 2.0, 4242, device=dev)
    ids, vals, _ = D.topk(logits, k)
    del logits
    U, W = SI.make_codebooks(V, r, 4243, device=dev)
    pid = torch.empty(S, P, dtype=torch.int32, device=dev)
    prk = torch.empty(S, P, dtype=torch.int32, device=dev)
    psc = torch.empty(S, dtype=torch.float32, device=dev)
    ws = torch.empty(S * (P - 1) * k * k * 4, dtype=torch.uint8, device=dev)
    ms = timed(lambda: D.select_path(ids, vals, U, W, positions=P, path_ids=pid, path_ranks=prk, path_score=psc, ws=ws))
    b = S * (P - 1) * 2 * k * r * 2 + S * P * k * 8 + 2 * S * (P - 1) * k * k * 4 + S * P * 8 + S * 4
    out["selector"] = {
        "workload": "32 streams x 15 positions x top-16, vocabulary 151936, rank-256 codebooks",
        "ms": ms, "streams_per_s": S * 1e3 / ms, "algorithmic_bytes": b,
        "achieved_gbs": b / (ms * 1e-3) / 1e9, "frac_of_hbm_peak": b / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
        "bound": "latency (14 pair tables and a 15-step recursion a stream)",
    }
    del U, W, ws
    widths = [4, 2, 2, 1, 1, 1, 1]
    topk_ids, _, _ = D.topk(SI.make_logits((S * 15, V), 2.0, 800, device=dev), 8)
    anchors = SI.anchor_ids(S, V, V - 1, 801, device=dev)
    N = D.tree_size(widths, 8)
    tokens, parents, depths, mask = D.tree_build(anchors, topk_ids, widths)
    tl = SI.make_logits((S, N, V), 2.0, 802, device=dev)
    acc = torch.empty(S, dtype=torch.int32, device=dev)
    toks = torch.empty(S, 16, dtype=torch.int32, device=dev)
    node = torch.empty(S, dtype=torch.int32, device=dev)
    tws = torch.empty(S * N * 8, dtype=torch.uint8, device=dev)
    ms_b = timed(lambda: D.tree_build(anchors, topk_ids, widths))
    ms_v = timed(lambda: D.tree_verify(tokens, tl, widths, accept=acc, tokens=toks, node=node, ws=tws))
    bv = S * N * V * 2 + S * N * 4 + S * 17 * 4
    out["tree"] = {
        "workload": f"32 streams, {N}-node trees (widths {widths}), vocabulary 151936",
        "build_ms": ms_b, "verify_ms": ms_v, "verify_rows_per_s": S * N * 1e3 / ms_v,
        "verify_algorithmic_bytes": bv, "verify_achieved_gbs": bv / (ms_v * 1e-3) / 1e9,
        "verify_frac_of_hbm_peak": bv / (ms_v * 1e-3) / 1e9 / pk["hbm_gbs"], "bound": "hbm (target rows scanned once)",
    }
    del tl, tws
    base = SI.preset("dflash2geom")["model"]
    m = SI.shrink(base, n_layers=1, layer_kinds=[SI.FULL], vocab=1024, variant=2, conv_groups=16)
    dr = D.Drafter(m, SI.make_weights(m, 831, device=dev))
    Sc = 8
    st = dr.new_state(Sc, 64)
    X = torch.randn(Sc * 16, m["hidden"], device=dev)
    ms_c = timed(lambda: st.draft_conv(X))
    T, H, G = Sc * 16, m["hidden"], 16
    bc = T * H * (4 + 4) + 2 * G * H * 2 + H * 2  # the residual read and written once, the weights once
    out["conv"] = {
        "workload": "8 streams x 16 rows, hidden 5120, 16 groups (the whole stage: norm, tap logits, mix, "
        "sums of squares for the final norm)",
        "ms": ms_c, "algorithmic_bytes": bc, "achieved_gbs": bc / (ms_c * 1e-3) / 1e9,
        "frac_of_hbm_peak": bc / (ms_c * 1e-3) / 1e9 / pk["hbm_gbs"], "bound": "latency (5 MB a call)",
    }
    del st, dr
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- our arm
def max_over_ranks(value, world, device):
    """The largest of every rank's value (the slowest replica's time), as
    every rank sees it; the value itself on a single rank."""
    if world <= 1:
        return value
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def run_ours(args, rank, world):
    import torch

    import block_diffusion_speculative_tap_gb300 as D
    import synthetic_inputs as SI
    from block_diffusion_speculative_tap_gb300 import _abi as A

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    P = SI.preset("9b")
    m = P["model"]
    C0 = P["context"][0]
    seed = P["seed"] + rank
    w = SI.make_weights(m, seed, device=dev)
    dr = D.Drafter(m, w)
    total_steps = args.warmup + 2 * args.steps + args.e2e_steps + 2
    max_settle = 400
    R = C0 + 16 * (max(total_steps, max_settle) + 2)
    st = dr.new_state(1, max(R, P["ring"]))
    ctx = SI.make_taps(m, C0, seed + 1, device=dev)
    st.fuse_taps(ctx, [(0, 0, C0)])
    del ctx
    # a round's 16 tap rows of every tap layer in one buffer [n_taps, 16, H]
    # (one host-to-device copy a round end to end); the planes are its slices
    taps_buf = torch.stack(SI.make_taps(m, 16, seed + 2, device=dev)).contiguous()
    step_taps = [taps_buf[i] for i in range(taps_buf.shape[0])]
    anchor = SI.anchor_ids(1, m["vocab"], m["mask_token"], seed + 3, device=dev)
    tl = SI.make_logits((1, 16, m["vocab"]), 1.0, seed + 4, device=dev)
    logits = torch.empty(15, m["vocab"], dtype=torch.bfloat16, device=dev)
    # a round's int32 results in one buffer (one readback end to end):
    # accept length [1], tokens [1, 16], top-8 draft ids [15, 8]
    results = torch.empty(1 + 16 + 15 * 8, dtype=torch.int32, device=dev)
    ids = results[17:].view(15, 8)
    vals = torch.empty(15, 8, dtype=torch.float32, device=dev)
    acc = results[0:1]
    toks = results[1:17].view(1, 16)
    stream = torch.cuda.current_stream()

    def step():
        C = st.length(0)
        st.fuse_taps(step_taps, [(0, C, 16)])
        st.draft(anchor, k=8, logits=logits, ids=ids, vals=vals)
        D.verify_greedy(ids, tl, accept=acc, tokens=toks)

    # clocks settle: untimed steps for at least 0.3 s (an idle GPU ramps its
    # clocks over tens of milliseconds), then the W warm-up steps
    t_settle = time.perf_counter()
    settle = 0
    while time.perf_counter() - t_settle < 0.3 and settle < max_settle:
        step()
        torch.cuda.synchronize()
        settle += 1
    st.truncate(0, C0)  # back to the workload's starting context
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    def timed(n, trace):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        if trace:
            A.lib.dflash_trace_enable(1)
        l0 = D.launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        if trace:
            A.lib.dflash_trace_enable(0)
        if world > 1:
            torch.distributed.barrier()
        return e0.elapsed_time(e1), D.launch_count() - l0

    clocks = ClockSampler(dev.index)
    clocks.start()
    ms, launches = timed(args.steps, trace=False)
    clk = clocks.stop()
    ms_tr, _ = timed(args.steps, trace=True)
    # per-launch durations of the traced region
    import ctypes as C

    recs = []
    for i in range(A.lib.dflash_trace_count()):
        nm, t, b, fl = C.c_char_p(), C.c_float(), C.c_double(), C.c_double()
        if A.lib.dflash_trace_get(i, C.byref(nm), C.byref(t), C.byref(b), C.byref(fl)) == 0:
            recs.append((nm.value.decode(), t.value, b.value, fl.value))
    by = {}
    for nm, t, b, fl in recs:
        e = by.setdefault(nm, [0, 0.0, 0.0, 0.0])
        e[0] += 1
        e[1] += t
        e[2] += b
        e[3] += fl
    ms_max = max_over_ranks(ms, world, dev)

    # ---- the draft alone (block forward + LM head + top-8) at the current
    # context: blocks/s and its fraction of the weight-streaming roofline
    def draft_only():
        st.draft(anchor, k=8, logits=logits, ids=ids, vals=vals)

    for _ in range(3):
        draft_only()
    torch.cuda.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for _ in range(args.steps):
        draft_only()
    d1.record(stream)
    torch.cuda.synchronize()
    draft_ms = d0.elapsed_time(d1) / args.steps
    A.lib.dflash_trace_enable(1)
    draft_only()
    torch.cuda.synchronize()
    A.lib.dflash_trace_enable(0)
    draft_bytes = 0.0
    for i in range(A.lib.dflash_trace_count()):
        nm, t, b, fl = C.c_char_p(), C.c_float(), C.c_double(), C.c_double()
        if A.lib.dflash_trace_get(i, C.byref(nm), C.byref(t), C.byref(b), C.byref(fl)) == 0:
            draft_bytes += b.value

    # ---- fused tap rows/s: a 4096-row prompt fill (fc + hidden_norm + K/V injection)
    fill_rows = 4096
    st2 = dr.new_state(1, fill_rows)
    fill_taps = SI.make_taps(m, fill_rows, seed + 5, device=dev)
    for _ in range(2):
        st2.fuse_taps(fill_taps, [(0, 0, fill_rows)])
        st2.truncate(0, 0)
    torch.cuda.synchronize()
    A.lib.dflash_trace_enable(1)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nfill = 3
    f0.record(stream)
    for _ in range(nfill):
        st2.fuse_taps(fill_taps, [(0, 0, fill_rows)])
        st2.truncate(0, 0)
    f1.record(stream)
    torch.cuda.synchronize()
    A.lib.dflash_trace_enable(0)
    fill_ms = f0.elapsed_time(f1) / nfill
    # the same fill without K/V injection (fc + hidden_norm + ring only)
    for _ in range(2):
        st2.fuse_taps(fill_taps, [(0, 0, fill_rows)], inject=False)
        st2.truncate(0, 0)
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(nfill):
        st2.fuse_taps(fill_taps, [(0, 0, fill_rows)], inject=False)
        st2.truncate(0, 0)
    g1.record(stream)
    torch.cuda.synchronize()
    fill_noinj_ms = g0.elapsed_time(g1) / nfill
    fill_recs = {}
    for i in range(A.lib.dflash_trace_count()):
        nm, t, b, fl = C.c_char_p(), C.c_float(), C.c_double(), C.c_double()
        if A.lib.dflash_trace_get(i, C.byref(nm), C.byref(t), C.byref(b), C.byref(fl)) == 0:
            e = fill_recs.setdefault(nm.value.decode(), [0, 0.0, 0.0, 0.0])
            e[0] += 1
            e[1] += t.value
            e[2] += b.value
            e[3] += fl.value
    del st2, fill_taps

    # ---- e2e: host buffers, copies inside the timed region, one readback a step
    h_taps = taps_buf.cpu().pin_memory()
    h_anchor = anchor.cpu().pin_memory()
    h_tl = tl.cpu().pin_memory()
    h_results = torch.empty(results.numel(), dtype=torch.int32).pin_memory()
    h2d = h_taps.numel() * 2 + 4 + h_tl.numel() * 2
    # the target logits (the bulk of the bytes; needed only by verification)
    # travel on a side stream, queued behind the tap copy, under the draft
    side = torch.cuda.Stream(device=dev)
    e_go, e_tl = torch.cuda.Event(), torch.cuda.Event()
    d2h = h_results.numel() * 4
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        # the fill goes first, so the GPU starts while the host queues the rest
        taps_buf.copy_(h_taps, non_blocking=True)
        e_go.record(stream)
        C = st.length(0)
        st.fuse_taps(step_taps, [(0, C, 16)])
        with torch.cuda.stream(side):
            side.wait_event(e_go)
            tl.copy_(h_tl, non_blocking=True)
            e_tl.record(side)
        anchor.copy_(h_anchor, non_blocking=True)
        st.draft(anchor, k=8, logits=logits, ids=ids, vals=vals)
        stream.wait_event(e_tl)
        D.verify_greedy(ids, tl, accept=acc, tokens=toks)
        h_results.copy_(results, non_blocking=True)
        stream.synchronize()  # the next round's anchor depends on this round's result
    e2e_s = time.perf_counter() - t0
    rc, bits = st.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {bits}")

    pk, src = peaks()
    gemm = [v for k, v in by.items() if k.startswith("gemm.")]
    g_ms = sum(v[1] for v in gemm)
    g_b = sum(v[2] for v in gemm)
    g_n = sum(v[0] for v in gemm)
    # The trace brackets every launch with events, which breaks the launch
    # chaining: each traced launch pays a launch latency and a dependency gap
    # the untraced step hides, about the same for a small kernel as for a
    # large one. That cost per launch is the traced step's excess over the
    # untraced one, divided by the launches; taking it off each GEMM launch
    # gives the GEMMs' time in the timed region (the raw traced durations
    # give a lower bound of their bandwidth).
    ovh = max(0.0, (ms_tr - ms) / launches) if launches else 0.0
    g_ms_live = g_ms - g_n * ovh
    if g_ms_live <= 0 or g_ms_live > ms:
        g_ms_live = None
    share = g_ms_live / ms if g_ms_live else None
    achieved = (g_b / g_n) / ((g_ms_live / g_n) * 1e-3) / 1e9 if g_n and g_ms_live else None
    achieved_traced = (g_b / g_n) / ((g_ms / g_n) * 1e-3) / 1e9 if g_n else None
    fc = fill_recs.get("gemm.fc", [0, 0.0, 0.0, 0.0])
    fc_tflops = fc[3] / (fc[1] * 1e-3) / 1e12 if fc[0] else None
    step_ms = ms_max / args.steps
    out = {
        "metric": METRIC,
        "value": world * args.steps / (ms_max * 1e-3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) taps, N(0,1) target logits)",
        "config": bench_config(world),
        "run": {"ring": st.ring, "settle_steps": settle},
        "fused_tap_rows_per_s": fill_rows / (fill_ms * 1e-3),
        "fused_tap_rows_per_s_without_kv_injection": fill_rows / (fill_noinj_ms * 1e-3),
        "fill": {
            "rows": fill_rows,
            "ms": fill_ms,
            "ms_without_kv_injection": fill_noinj_ms,
            "fc_tflops": fc_tflops,
            "fc_frac_of_bf16_peak": (fc_tflops / pk["bf16_tflops"]) if fc_tflops else None,
            "peak_source": src,
            "kernels_ms": {k: v[1] / nfill for k, v in fill_recs.items()},
        },
        "roofline": {
            "kernel": "gemm_kernel (tcgen05, every GEMM launch of the decode step)",
            "bound": "hbm",
            "achieved": achieved,
            "peak": pk["hbm_gbs"],
            "unit": "GB/s",
            "frac": (achieved / pk["hbm_gbs"]) if achieved else None,
            "traffic": gemm_traffic(),
            "peak_source": src,
            "method": "algorithmic bytes per GEMM launch / its CUDA-event duration in a traced pass less the "
            "trace's cost per launch ((traced step - untraced step) / launches); the raw traced durations "
            "give the lower bound",
            "trace_cost_per_launch_us": ovh * 1e3,
            "gemm_ms_per_step": g_ms_live / args.steps if g_ms_live else None,
            "gemm_share_of_step": share,
            "gemm_ms_per_step_traced": g_ms / args.steps,
            "achieved_traced_lower_bound": achieved_traced,
            "frac_traced_lower_bound": (achieved_traced / pk["hbm_gbs"]) if achieved_traced else None,
            "gemm_ms_le_step": bool(g_ms_live is not None and g_ms_live <= ms + 1e-9),
            "gemm_bytes_per_step": g_b / args.steps,
            "gemm_launches_per_step": g_n / args.steps,
            "step_bytes_per_step": sum(v[2] for v in by.values()) / args.steps,
            "step_frac_of_hbm_peak": sum(v[2] for v in by.values()) / args.steps / (step_ms * 1e-3) / 1e9
            / pk["hbm_gbs"],
        },
        "draft_only": {
            "blocks_per_s": 1e3 / draft_ms,
            "ms": draft_ms,
            "algorithmic_bytes": draft_bytes,
            "achieved_gbs": draft_bytes / (draft_ms * 1e-3) / 1e9,
            "frac_of_hbm_peak": draft_bytes / (draft_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "note": "dflash_draft_block alone (weights once, K/V of the visible context, activations), "
            "CUDA events around K back-to-back drafts at a fixed context",
        },
        "step_kernels_ms": {k: v[1] / args.steps for k, v in sorted(by.items(), key=lambda kv: -kv[1][1])},
        "ms_per_step_traced": ms_tr / args.steps,
        "e2e": {
            "value": args.e2e_steps / e2e_s * world,
            "unit": UNIT,
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps,
        },
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if world == 1 and not args.no_other_configs:
        others = {"tiny": measure_config("tiny", dev, pk, 50)}
        for name in ("long32k", "serve32"):
            others[name] = measure_config(name, dev, pk, 20, dr=dr)
        del st
        torch.cuda.empty_cache()
        others["dflash2geom"] = measure_config("dflash2geom", dev, pk, 20)
        others["next_rows"] = measure_next_rows(dev, pk, 20)
        out["other_configs"] = {
            "note": "supplementary: the parity workloads measured at their own streams and contexts "
            "(draft = block forward + LM head + top-k; verify = the workload's mode); not the headline",
            **others,
        }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args, m, w, seed, C0)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return out


# ---------------------------------------------------------------- multi-stream rounds split by stream
SHARDED = {
    "serve32": (
        "32 streams of the 9B-shaped DFlash v1 drafter (8 taps x hidden 4096, 6 layers 32q/8kv x 128, "
        "SwiGLU 12288, layers 0-4 sliding 2048, vocab 151936), contexts uniform in [1024, 16384] (seeded), "
        "one shared round a step: block-16 draft, top-8, greedy verify against N(0,2) target logits with "
        "planted accept lengths"
    ),
    "dflash2geom": (
        "8 streams of the DFlash2-geometry drafter (5 taps x hidden 5120, 5 layers 40q/8kv x 128, "
        "SwiGLU 17408, vocab 151936) at context 8192, one shared round a step: block-16 draft, top-8, "
        "drafted ids sampled at T=1, sampling verify (accept min(1,p/q), residual max(0,p-q))"
    ),
}


def partition_streams(S, world, rank):
    """Contiguous stream range [lo, hi) of `rank` when S streams are split
    over `world` ranks; the first S % world ranks take one stream more."""
    base, extra = divmod(int(S), int(world))
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def gather_streams(lo, accept, tokens, world):
    """Host gather of one round's results to rank 0. Each rank passes the
    first stream of its range, its accept lengths [n] and committed tokens
    [n][16]; rank 0 gets (accept [S], tokens [S][16]) in stream order, the
    other ranks None. No collective runs during the timed rounds."""
    item = (int(lo), [int(a) for a in accept], [[int(t) for t in row] for row in tokens])
    if world <= 1:
        parts = [item]
    else:
        import torch.distributed as dist

        parts = [None] * world if dist.get_rank() == 0 else None
        dist.gather_object(item, parts, dst=0)
        if dist.get_rank() != 0:
            return None
    parts = sorted(parts, key=lambda p: p[0])
    return [a for p in parts for a in p[1]], [t for p in parts for t in p[2]]


def trace_groups(A):
    """Per kernel group (the label before its first dot) of the last trace:
    [launches, traced ms, algorithmic bytes, flops]."""
    import ctypes as C

    by = {}
    for i in range(A.lib.dflash_trace_count()):
        nm, t, b, fl = C.c_char_p(), C.c_float(), C.c_double(), C.c_double()
        if A.lib.dflash_trace_get(i, C.byref(nm), C.byref(t), C.byref(b), C.byref(fl)) == 0:
            e = by.setdefault(nm.value.decode().split(".")[0], [0, 0.0, 0.0, 0.0])
            e[0] += 1
            e[1] += t.value
            e[2] += b.value
            e[3] += fl.value
    return by


def run_sharded(args, rank, world):
    """One multi-stream round a step, the round's streams split over ranks."""
    import ctypes

    import torch

    import block_diffusion_speculative_tap_gb300 as D
    import synthetic_inputs as SI
    from block_diffusion_speculative_tap_gb300 import _abi as A

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    name = args.workload
    P = SI.preset(name)
    m = P["model"]
    ctx = P["context"]
    S, V, k = len(ctx), m["vocab"], P["topk"]
    lo, hi = partition_streams(S, world, rank)
    n = hi - lo
    w = SI.make_weights(m, P["seed"], device=dev)  # replicated: the same weights on every rank
    dr = D.Drafter(m, w)
    st = dr.new_state(n, P["ring"])
    for j, s_ in enumerate(range(lo, hi)):  # stream s_ draws its context from its own seed on any rank
        taps = SI.make_taps(m, ctx[s_], P["seed"] + 1 + s_, device=dev)
        st.fuse_taps(taps, [(j, 0, ctx[s_])])
        del taps
    anchors = SI.anchor_ids(S, V, m["mask_token"], P["seed"] + 2, device=dev)[lo:hi].contiguous()
    tl = SI.make_logits((S, 16, V), P["target_logit_std"], P["seed"] + 3, device=dev)[lo:hi].contiguous()
    logits = torch.empty(n * 15, V, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(n * 15, k, dtype=torch.int32, device=dev)
    vals = torch.empty(n * 15, k, dtype=torch.float32, device=dev)
    results = torch.empty(n * 17, dtype=torch.int32, device=dev)  # accept [n], tokens [n, 16]
    acc, toks = results[:n], results[n:].view(n, 16)
    sample = P["verify"] == "sample"
    lengths = None
    if sample:
        T = P.get("temperature", 1.0)
        ud = SI.make_uniforms((S * 15,), P["seed"] + 4, device=dev)[lo * 15 : hi * 15].contiguous()
        u = SI.make_uniforms((S, 16, 2), P["seed"] + 5, device=dev)[lo:hi].contiguous()
        drafted = torch.empty(n * 15, dtype=torch.int32, device=dev)
        nb = ctypes.c_size_t()
        A.check(A.lib.dflash_verify_workspace_bytes(A.VERIFY_SAMPLE, n, V, ctypes.byref(nb)), "workspace")
        vws = torch.empty(max(nb.value, 256), dtype=torch.uint8, device=dev)
    else:
        # planted accept lengths: the target's argmax follows the draft for L rows
        st.draft(anchors, k=k, logits=logits, ids=ids, vals=vals)
        lengths = SI.make_accept_lengths(S, P["seed"] + 4)
        tl_h = tl.cpu()
        SI.plant_accepts(tl_h, ids[:, 0].reshape(n, 15).cpu(), lengths[lo:hi])
        tl.copy_(tl_h)
    stream = torch.cuda.current_stream()

    def step():
        st.draft(anchors, k=k, logits=logits, ids=ids, vals=vals)
        if sample:
            D.topk(logits, 0, temperature=T, uniforms=ud, sampled=drafted)
            D.verify_sample(drafted.view(n, 15), tl, logits.view(n, 15, V), u, T, accept=acc, tokens=toks, ws=vws)
        else:
            D.verify_greedy(ids, tl, accept=acc, tokens=toks)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    def timed(steps, trace):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        if trace:
            A.lib.dflash_trace_enable(1)
        l0 = D.launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        if trace:
            A.lib.dflash_trace_enable(0)
        if world > 1:
            torch.distributed.barrier()
        return e0.elapsed_time(e1), D.launch_count() - l0

    clocks = ClockSampler(dev.index)
    clocks.start()
    ms, launches = timed(args.steps, trace=False)
    clk = clocks.stop()
    ms_tr, _ = timed(1, trace=True)
    by = trace_groups(A)
    ms_max = max_over_ranks(ms, world, dev)
    # the round's results, gathered on the host after the timing
    got = gather_streams(lo, acc.cpu().tolist(), toks.cpu().tolist(), world)
    check = None
    if got is not None and lengths is not None:
        check = {"planted_accepts_recovered": got[0] == [min(L, 15) for L in lengths], "streams": len(got[0])}

    # end to end: target logits (and uniforms) from pinned host memory, the
    # round's accept lengths and tokens read back, every step
    h_tl = tl.cpu().pin_memory()
    h_anchor = anchors.cpu().pin_memory()
    h_res = torch.empty(results.numel(), dtype=torch.int32).pin_memory()
    h2d = h_tl.numel() * 2 + h_anchor.numel() * 4
    if sample:
        h_ud, h_u = ud.cpu().pin_memory(), u.cpu().pin_memory()
        h2d += h_ud.numel() * 4 + h_u.numel() * 4
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        anchors.copy_(h_anchor, non_blocking=True)
        tl.copy_(h_tl, non_blocking=True)
        if sample:
            ud.copy_(h_ud, non_blocking=True)
            u.copy_(h_u, non_blocking=True)
        step()
        h_res.copy_(results, non_blocking=True)
        stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    rc, bits = st.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {bits}")
    pk, src = peaks()
    top = max(by.items(), key=lambda kv: kv[1][1])
    per_round = launches / args.steps if args.steps else 0
    ovh = max(0.0, (ms_tr - ms / args.steps) / per_round) if per_round else 0.0
    top_ms = top[1][1] - top[1][0] * ovh
    if top_ms <= 0 or top_ms > ms / args.steps:
        top_ms = None
    achieved = top[1][2] / (top_ms * 1e-3) / 1e9 if top_ms else None
    round_bytes = sum(v[2] for v in by.values())
    out = {
        "metric": METRIC,
        "value": S * args.steps / (ms_max * 1e-3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps,
        "higher_is_better": True,
        "scaling": "strong",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) taps, seeded contexts and target logits)",
        "config": {
            "workload": SHARDED[name],
            "streams": S,
            "parallelism": f"streams split contiguously over {world} rank(s), weights replicated, no collective",
            "l2": "no flush: every round streams the weights (3.8-4.9 GB) through the 129 MB L2",
        },
        "run": {"streams_this_rank": [lo, hi], "result_check": check},
        "roofline": {
            "kernel": f"{top[0]} (the kernel group with the largest share of the round)",
            "bound": "hbm",
            "achieved": achieved,
            "peak": pk["hbm_gbs"],
            "unit": "GB/s",
            "frac": (achieved / pk["hbm_gbs"]) if achieved else None,
            "traffic": None,
            "peak_source": src,
            "method": "algorithmic bytes of the group's launches in a round / their CUDA-event durations in a "
            "traced round less the trace's cost per launch ((traced round - untraced round) / launches)",
            "group_ms_per_round": top_ms,
            "round_bytes": round_bytes,
            "round_frac_of_hbm_peak": round_bytes / (ms / args.steps * 1e-3) / 1e9 / pk["hbm_gbs"],
        },
        "round_kernels_ms_traced": {kk: round(v[1], 4) for kk, v in sorted(by.items(), key=lambda kv: -kv[1][1])},
        "e2e": {
            "value": S * args.e2e_steps / e2e_s,
            "unit": UNIT,
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": h_res.numel() * 4,
            "steps": args.e2e_steps,
        },
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return out


# ---------------------------------------------------------------- oracle (reference / baseline)
def oracle_step_setup(m, w64, C0, ctx_planes, step_planes):
    import oracle as O

    ref = O.OracleStreams(m, w64, 1)
    ref.append(0, ctx_planes)
    return ref


def cpu_baseline(args, m, w, seed, C0):
    """Time the oracle on a bounded sample of the same workload: a fixed
    number of decode rounds (16-row fusion + K/V injection, block draft,
    top-8, greedy verify) from the 4096-row context, on one BLAS thread (the
    context fill before them uses every core and is not timed)."""
    import oracle as O
    import synthetic_inputs as SI

    t_setup = time.perf_counter()
    w64 = O.weights_to_f64(w)
    ctx = [O.to_f64(p) for p in SI.make_taps(m, C0, seed + 1, device="cuda")]
    ref = O.OracleStreams(m, w64, 1)
    ref.append(0, ctx)
    del ctx
    step = [O.to_f64(p) for p in SI.make_taps(m, 16, seed + 2, device="cuda")]
    anchor = int(SI.anchor_ids(1, m["vocab"], m["mask_token"], seed + 3)[0])
    tl = O.to_f64(SI.make_logits((1, 16, m["vocab"]), 1.0, seed + 4))[0]
    setup_s = time.perf_counter() - t_setup
    before, _ = blas_threads()
    threads, lib = blas_threads(1)
    n = args.cpu_rounds
    t0 = time.perf_counter()
    for _ in range(n):
        ref.append(0, step)
        logits, _ = ref.draft(0, anchor)
        ids = [O.topk(logits[r], 8)[0] for r in range(15)]
        O.greedy_verify([int(i[0]) for i in ids], tl)
    dt = time.perf_counter() - t0
    if before:
        blas_threads(before)
    return {
        "value": n / dt,
        "unit": UNIT,
        "cores": threads if threads else 1,
        "kind": "oracle",
        "sample": f"{n} decode rounds of the same workload from the 4096-row context (float64 NumPy oracle; "
        f"BLAS threads as its runtime reports: {threads} ({os.path.basename(lib) if lib else 'no BLAS found'}); "
        f"context set-up {setup_s:.1f} s on all cores, not timed)",
    }


def run_reference(args):
    import numpy as np

    import oracle as O
    import synthetic_inputs as SI

    P = SI.preset("9b")
    m = P["model"]
    C0 = P["context"][0]
    seed = P["seed"]
    w = SI.make_weights(m, seed, device="cpu")
    w64 = O.weights_to_f64(w)
    del w
    ref = O.OracleStreams(m, w64, 1)
    ref.append(0, [O.to_f64(p) for p in SI.make_taps(m, C0, seed + 1)])
    step = [O.to_f64(p) for p in SI.make_taps(m, 16, seed + 2)]
    anchor = int(SI.anchor_ids(1, m["vocab"], m["mask_token"], seed + 3)[0])
    tl = O.to_f64(SI.make_logits((1, 16, m["vocab"]), 1.0, seed + 4))[0]

    def one():
        ref.append(0, step)
        logits, _ = ref.draft(0, anchor)
        ids = [O.topk(logits[r], 8)[0] for r in range(15)]
        O.greedy_verify([int(i[0]) for i in ids], tl)

    # the context fill above used every core; the rounds run on one thread
    threads, lib = blas_threads(1)
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    threads = threads if threads else 1
    v = args.steps / dt
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": v,
        "unit": UNIT,
        "n_gpus": 0,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": bench_config(int(os.environ.get("WORLD_SIZE", 1))),
        "cpu_baseline": {
            "value": v,
            "unit": UNIT,
            "cores": threads,
            "kind": "oracle",
            "sample": f"{args.steps} timed decode rounds after {args.warmup} untimed ones from the 4096-row "
            f"context (float64 NumPy oracle, BLAS threads as its runtime reports: {threads})",
        },
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def profile_workload(name):
    """A small workload for an ncu capture of one kernel (no timing, no JSON
    line): 'attention32' drafts 32 streams x 2048 context rows through a
    two-layer 9B-shaped drafter (both layers sliding) three times, so the
    many-stream attention launch is captured at a few GB of device memory;
    'fill4096' runs a 4096-row prompt fill of the 9B-shaped drafter three
    times (fc GEMM, hidden_norm, K/V injection); 'attention8d2' drafts 8
    streams x 8192 context rows through a one-layer drafter of the DFlash2
    geometry (40 q / 8 kv heads of 128) three times, so the tensor-memory
    attention launch is captured; 'treeverify' verifies 32 streams of
    93-node draft trees over a 151936-token vocabulary three times (the
    arg-max scan of 2976 target rows, 904 MB); 'topk480' takes the top 8 of
    480 rows of 151936 logits three times (the vocabulary scan of a
    32-stream draft, 146 MB); 'sampleverify' runs sampling verification of
    8 streams over a 151936-token vocabulary three times (the DFlash2
    geometry's round: 31 rows of statistics and the cluster draw a stream)."""
    import torch

    import block_diffusion_speculative_tap_gb300 as D
    import synthetic_inputs as SI

    torch.cuda.set_device(0)
    if name == "fill4096":
        # a 4096-row prompt fill of the 9B-shaped drafter, three times
        m = SI.preset("9b")["model"]
        dr = D.Drafter(m, SI.make_weights(m, 5, device="cuda"))
        st = dr.new_state(1, 4096)
        taps = SI.make_taps(m, 4096, 6, device="cuda")
        for _ in range(3):
            st.fuse_taps(taps, [(0, 0, 4096)])
            st.truncate(0, 0)
        torch.cuda.synchronize()
        rc, bits = st.status()
        if rc != 0:
            raise RuntimeError(f"device status {rc} bits {bits}")
        return
    if name == "treeverify":
        S, V, widths = 32, 151936, [4, 2, 2, 1, 1, 1, 1]
        topk_ids, _, _ = D.topk(SI.make_logits((S * 15, V), 2.0, 800, device="cuda"), 8)
        anchors = SI.anchor_ids(S, V, V - 1, 801, device="cuda")
        tokens, _, _, _ = D.tree_build(anchors, topk_ids, widths, want_mask=False)
        tl = SI.make_logits((S, D.tree_size(widths, 8), V), 2.0, 802, device="cuda")
        for _ in range(3):
            D.tree_verify(tokens, tl, widths)
        torch.cuda.synchronize()
        return
    if name == "topk480":
        lg = SI.make_logits((480, 151936), 2.0, 810, device="cuda")
        for _ in range(3):
            D.topk(lg, 8)
        torch.cuda.synchronize()
        return
    if name == "sampleverify":
        S, V = 8, 151936
        tl = SI.make_logits((S, 16, V), 1.0, 820, device="cuda")
        dl = (tl[:, :15].float() + 0.5 * SI.make_logits((S, 15, V), 1.0, 821, device="cuda").float()).to(torch.bfloat16)
        draft = SI.make_token_ids((S, 15), V, 822, device="cuda")
        u = SI.make_uniforms((S, 16, 2), 823, device="cuda")
        for _ in range(3):
            D.verify_sample(draft, tl, dl, u, 1.0)
        torch.cuda.synchronize()
        return
    if name == "attention8d2":
        m = SI.shrink(SI.preset("dflash2geom")["model"], n_layers=1, layer_kinds=[SI.FULL], vocab=8192)
        S, C = 8, 8192
    elif name == "attention32":
        m = SI.shrink(SI.preset("9b")["model"], n_layers=2, layer_kinds=[SI.SLIDING] * 2)
        S, C = 32, 2048
    else:
        raise SystemExit(f"unknown profile workload {name}")
    dr = D.Drafter(m, SI.make_weights(m, 5, device="cuda"))
    st = dr.new_state(S, C + 1024)
    for s in range(S):
        st.fuse_taps(SI.make_taps(m, C, 100 + s, device="cuda"), [(s, 0, C)])
    anchors = SI.anchor_ids(S, m["vocab"], m["mask_token"], 7, device="cuda")
    for _ in range(3):
        st.draft(anchors, k=8)
    torch.cuda.synchronize()
    rc, bits = st.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {bits}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--e2e-steps", type=int, default=60)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rounds", type=int, default=4, help="decode rounds of the CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true", help="skip the supplementary workloads")
    ap.add_argument("--workload", default="9b", choices=["9b"] + sorted(SHARDED),
                    help="9b: the batch-1 decode round (default); serve32 / dflash2geom: a multi-stream round, "
                    "streams split over ranks")
    ap.add_argument("--profile-workload", default=None, help="run a small workload for ncu (attention32, attention8d2, fill4096, treeverify, topk480, sampleverify) and exit")
    args = ap.parse_args()
    if args.profile_workload:
        profile_workload(args.profile_workload)
        return 0
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if rank != 0:
            return 0
        if args.workload != "9b":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the default workload "
                              "(the 9B-shaped batch-1 decode round) only"}), flush=True)
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    out = run_ours(args, rank, world) if args.workload == "9b" else run_sharded(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
