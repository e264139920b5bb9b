"""Benchmark of the low-batch MXFP8 decode projections on one GB300 per rank.

Workload (one "step"): the single decode-projection GEMM at M = 1, 2, 4, 8
activation rows, N = 2048, K = 5120 - each activation arrives as bf16, goes
through mx_quantize_rows (128x4-swizzled scales) and then mx_gemm (launched
with programmatic dependent launch). value = algorithmic HBM bytes of the step
/ step time (GB/s). Weights rotate over enough copies (>= 3x L2) that every
GEMM streams its weight from HBM. Extras on the same line: per-M GEMM time and
bandwidth, the three-projection chain (M = 1..64), the grouped WO-A + wo_b
pair (T = 1, 8, 32), the kernel roofline, an end-to-end number through the
Python API with host buffers, SM clocks, and the CPU oracle's time on a
bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --profile gemm|bf16|chain|wo_a|sweep   (a few plain launches for ncu)
  python bench.py --timeline   (per-CTA phase timeline, timeline build of the library)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "small-M MXFP8 GEMM µs & HBM GB/s vs GB300 peak; 3-projection chain µs/step"
M_LIST = (1, 2, 4, 8)
N1, K1 = 2048, 5120
CHAIN_SHAPES = [(2048, 5120), (8192, 1536), (5120, 8192)]
CHAIN_G1_COLS = 1536
CHAIN_M = (1, 4, 8, 16, 32, 48, 64)
WOA = dict(G=4, H=8, R=1024, D=512)
WOA_T = (1, 8, 16, 32)
WOB = (5120, 4096)
SWEEP_M = (64, 96, 128, 192, 256)
SWEEP_SHAPES = [(8192, 5120), (5120, 8192)]


def w_bytes(n, k):
    return n * k + n * k // 32


def gemm_bytes(m, n, k):
    """Algorithmic bytes of one GEMM: W + W scales + A + A scales + bf16 out."""
    return w_bytes(n, k) + m * k + m * k // 32 + 2 * m * n


def quant_bytes(m, k):
    return 2 * m * k + m * k + m * k // 32


def step_bytes():
    return sum(gemm_bytes(m, N1, K1) + quant_bytes(m, K1) for m in M_LIST)


# DRAM bytes per gemm_kernel launch from an ncu capture of the decode-projection
# workload, keyed by the sha256 prefix of the kernel source it was taken on; a
# changed kernel reports null until it is captured again.
NCU_TRAFFIC = {"ef44984828dd5bdb": 10.893e6, "21856ef7ae979106": 10.907e6, "1d452fa6645ff44c": 10.902e6,
               "93ee1b1e31bdd36e": 10.901e6, "9ec494b77ea113c6": 10.902e6}


def gemm_source_sha():
    """Hash of the GEMM kernel's code (comments and blank lines dropped), which
    keys the DRAM traffic an ncu capture measured for that code."""
    import hashlib
    path = os.path.join(ROOT, "mxfp8_block_scaled_06_gb300", "csrc", "gemm.cu")
    lines = []
    for line in open(path).read().splitlines():
        line = line.split("//", 1)[0].rstrip()
        if line.strip():
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# --------------------------------------------------------------------- device
class Rig:
    """Device buffers of the benchmark: rotating weight copies and activations."""

    def __init__(self, torch, mx, h, l2_bytes):
        self.torch, self.mx, self.h = torch, mx, h
        self.dev = torch.device("cuda", torch.cuda.current_device())
        self.l2 = l2_bytes

    def copies(self, bytes_per_set):
        return max(4, -(-3 * self.l2 // bytes_per_set) + 1)

    def weight_set(self, shapes, seed, ncopies):
        """ncopies independent MXFP8 weight sets (quantized by the library)."""
        torch, mx = self.torch, self.mx
        out = []
        base = []
        for i, (n, k) in enumerate(shapes):
            bits = synth.block_scaled_bf16(seed, synth.TAG_W + i, n, k, -6, 6)
            x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(self.dev)
            base.append(mx.mx_quantize_rows(self.h, x))
        for c in range(ncopies):
            out.append([(q.clone(), s.clone()) for q, s in base])
        torch.cuda.synchronize()
        return out

    def activation(self, m, k, seed, umin=-6, umax=6):
        bits = synth.block_scaled_bf16(seed, synth.TAG_A + m, m, k, umin, umax)
        return self.torch.from_numpy(bits.view(np.int16)).view(self.torch.bfloat16).to(self.dev)


REPLAYS = 10  # every timing is the median of at least this many graph replays


def time_graph(torch, fn, reps, per_graph, stream):
    """Capture per_graph calls of fn into a CUDA graph and replay it reps times,
    each replay bracketed by CUDA events on the capturing stream; returns the
    per-replay device milliseconds and the graph."""
    with torch.cuda.stream(stream):
        fn(0)  # make sure everything is initialized outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(per_graph):
                fn(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        g.replay()
        torch.cuda.synchronize()
        for st, sp in ev:
            st.record(stream)
            g.replay()
            sp.record(stream)
    ev[-1][1].synchronize()
    return [st.elapsed_time(sp) for st, sp in ev], g


def median_us(torch, fn, per_graph, stream, reps=REPLAYS):
    """Median over reps replays of a per_graph-call graph, in us per call."""
    times, _ = time_graph(torch, fn, reps, per_graph, stream)
    return statistics.median(times) * 1e3 / per_graph


def step_replays(k):
    """Replays of a fixed-size graph that time exactly k steps: the smallest
    divisor of k that is at least min(10, k)."""
    return next(d for d in range(min(REPLAYS, k), k + 1) if k % d == 0)


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a window."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows if len(r) >= 9 for j in range(4)
                          if r[5 + j].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(sm)}


class Replicas:
    """N independent replicas, one process per GPU (launched by torchrun): the
    path has no exchange step, so the ranks share only host-side coordination
    over gloo - a barrier before the timed region and the maximum of the timed
    region over ranks. Rank 0 alone reports."""

    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        if self.world > 1:
            import torch.distributed as dist
            if not dist.is_initialized():
                dist.init_process_group("gloo", init_method="env://")

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(self, x: float) -> float:
        if self.world == 1:
            return x
        import torch
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def job_value(self, bytes_per_rank_step: float, ms_step: float) -> float:
        """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
        return self.world * bytes_per_rank_step / (ms_step * 1e-3) / 1e9

    @property
    def reports(self) -> bool:
        return self.rank == 0


def run_ours(args):
    import torch

    import mxfp8_block_scaled_06_gb300 as mx
    from mxfp8_block_scaled_06_gb300 import build as mxbuild

    rep = Replicas()
    world, rank, local = rep.world, rep.rank, rep.local
    mxbuild.build()
    torch.cuda.set_device(local)
    h = mx.mx_create(local)
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20)
    rig = Rig(torch, mx, h, l2)
    stream = torch.cuda.Stream()
    pk, pk_kind = peaks()
    K, W = args.steps, args.warmup

    # ---------------------------------------------------------------- main step
    nset = rig.copies(w_bytes(N1, K1))
    wts = rig.weight_set([(N1, K1)], seed=1, ncopies=nset)
    xs = {m: rig.activation(m, K1, seed=1) for m in M_LIST}
    qa = {m: (torch.empty((m, K1), dtype=torch.uint8, device=rig.dev),
              torch.empty(mx.mx_scale_bytes(m, K1), dtype=torch.uint8, device=rig.dev)) for m in M_LIST}
    outs = {m: torch.empty((m, N1), dtype=torch.bfloat16, device=rig.dev) for m in M_LIST}

    def step(i, quant=True):
        for j, m in enumerate(M_LIST):
            wq, ws = wts[(i * len(M_LIST) + j) % nset][0]
            if quant:
                mx.mx_quantize_rows(h, xs[m], q=qa[m][0], scales=qa[m][1], stream=stream)
            mx.mx_gemm(h, qa[m][0], qa[m][1], wq, ws, out=outs[m], pdl=True, stream=stream)

    # exactly K steps timed: `reps` replays of a graph of K / reps steps, each
    # replay bracketed by events; ms per step = the median replay / its steps
    reps = step_replays(K)
    per_graph = K // reps
    k_eff = reps * per_graph
    # warm-up: W steps untimed, then a sustained window so the clock sampler sees load
    for i in range(max(W, 3)):
        with torch.cuda.stream(stream):
            step(i)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    t_end = time.time() + 1.0
    _, g_step = time_graph(torch, step, 1, per_graph, stream)
    with torch.cuda.stream(stream):
        while time.time() < t_end:
            g_step.replay()
    torch.cuda.synchronize()
    rep.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for st, sp in ev:
            st.record(stream)
            g_step.replay()
            sp.record(stream)
    ev[-1][1].synchronize()
    torch.cuda.synchronize()
    rep.barrier()
    clk = clocks.stop()
    replay_ms = [st.elapsed_time(sp) for st, sp in ev]
    ms_step = rep.max_over_ranks(statistics.median(replay_ms) / per_graph)
    st, sp = ev[0]
    value = rep.job_value(step_bytes(), ms_step)

    # ------------------------------------------------- per-kernel GEMM timing
    gemm_us, gemm_gbs = {}, {}
    for m in M_LIST:
        def only(i, m=m):
            wq, ws = wts[i % nset][0]
            mx.mx_gemm(h, qa[m][0], qa[m][1], wq, ws, out=outs[m], pdl=True, stream=stream)
        us = median_us(torch, only, 100, stream)
        gemm_us[m] = us
        gemm_gbs[m] = gemm_bytes(m, N1, K1) / (us * 1e-6) / 1e9
    # the same step with the quantization inside the GEMM (mx_gemm_bf16: one
    # launch per projection instead of two)
    fused_us = {}
    for m in M_LIST:
        def fused(i, m=m):
            wq, ws = wts[i % nset][0]
            mx.mx_gemm_bf16(h, xs[m], wq, ws, out=outs[m], pdl=True, stream=stream)
        fused_us[m] = median_us(torch, fused, 100, stream)
    # dominant kernel: mx_gemm over the step's mix of M
    gemm_launch_us = median_us(torch, lambda i: step(i, quant=False), 100, stream) / len(M_LIST)
    gemm_mix_bytes = sum(gemm_bytes(m, N1, K1) for m in M_LIST) / len(M_LIST)
    achieved = gemm_mix_bytes / (gemm_launch_us * 1e-6) / 1e9
    quant_us = {}
    for m in (1, 8):
        quant_us[m] = median_us(torch, lambda i, m=m: mx.mx_quantize_rows(
            h, xs[m], q=qa[m][0], scales=qa[m][1], stream=stream), 100, stream)

    # ----------------------------------------------------------------- chain
    chain = {}
    if not args.quick:
        cset = rig.copies(sum(w_bytes(n, k) for n, k in CHAIN_SHAPES))
        cw = rig.weight_set(CHAIN_SHAPES, seed=2, ncopies=cset)
        wbytes = sum(w_bytes(n, k) for n, k in CHAIN_SHAPES)
        for m in CHAIN_M:
            a1 = rig.activation(m, CHAIN_SHAPES[0][1], seed=2, umin=-4, umax=4)
            q1 = mx.mx_quantize_rows(h, a1)
            bufs = dict(out=torch.empty((m, CHAIN_SHAPES[2][0]), dtype=torch.bfloat16, device=rig.dev),
                        a2=torch.empty((m, CHAIN_G1_COLS), dtype=torch.uint8, device=rig.dev),
                        a2_scales=torch.empty(mx.mx_scale_bytes(m, CHAIN_G1_COLS), dtype=torch.uint8, device=rig.dev),
                        a3=torch.empty((m, CHAIN_SHAPES[1][0]), dtype=torch.uint8, device=rig.dev),
                        a3_scales=torch.empty(mx.mx_scale_bytes(m, CHAIN_SHAPES[1][0]), dtype=torch.uint8, device=rig.dev))

            def run_chain(i, m=m, q1=q1, bufs=bufs):
                mx.mx_gemm_chain(h, q1[0], q1[1], cw[i % cset], g1_cols=CHAIN_G1_COLS, stream=stream, **bufs)
            us = median_us(torch, run_chain, 30, stream)
            chain[m] = {"us": round(us, 3), "weight_gbs": round(wbytes / (us * 1e-6) / 1e9, 1),
                        "vs_weight_read_at_peak": round(us / (wbytes / (pk["hbm_gbs"] * 1e9) * 1e6), 3)}
            # the same chain with the RMS-norm split between G1 and G2 (one more launch)
            out1 = torch.empty((m, CHAIN_SHAPES[0][0]), dtype=torch.bfloat16, device=rig.dev)
            nwb = synth.norm_weight_bf16(4, CHAIN_G1_COLS)
            nw = torch.from_numpy(nwb.view(np.int16)).view(torch.bfloat16).to(rig.dev)

            def run_norm(i, m=m, q1=q1, bufs=bufs, out1=out1, nw=nw):
                mx.mx_gemm_chain_norm(h, q1[0], q1[1], cw[i % cset], nw, 1e-6, g1_cols=CHAIN_G1_COLS,
                                      out1=out1, stream=stream, **bufs)
            chain[m]["with_rms_norm_split_us"] = round(median_us(torch, run_norm, 30, stream), 3)

    # ------------------------------------------------------- WO-A and wo_b
    woa = {}
    if not args.quick:
        G, H, R, D = WOA["G"], WOA["H"], WOA["R"], WOA["D"]
        pair = [(G * R, H * D), WOB]
        wset = rig.copies(sum(w_bytes(n, k) for n, k in pair))
        ww = rig.weight_set(pair, seed=3, ncopies=wset)
        cs = torch.from_numpy(synth.rope_cos_sin_cache(65536)).to(rig.dev)
        for t in WOA_T:
            xb = synth.normal_bf16(3 + t, synth.TAG_X, (t, G * H, D))
            x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(rig.dev)
            pos = torch.from_numpy(synth.positions(3 + t, synth.TAG_POS, t)).to(rig.dev)
            q = torch.empty((t, G * R), dtype=torch.uint8, device=rig.dev)
            qs = torch.empty(mx.mx_scale_bytes(t, G * R), dtype=torch.uint8, device=rig.dev)
            ob = torch.empty((t, WOB[0]), dtype=torch.bfloat16, device=rig.dev)

            def run_woa(i, t=t, x=x, pos=pos, q=q, qs=qs):
                wq, ws = ww[i % wset][0]
                mx.wo_a_grouped(h, x, pos, cs, wq, ws, G, H, R, q=q, q_scales=qs, early_trigger=True,
                                stream=stream)

            def run_pair(i, t=t, x=x, pos=pos, q=q, qs=qs, ob=ob):
                run_woa(i)
                wq, ws = ww[i % wset][1]
                mx.mx_gemm(h, q, qs, wq, ws, out=ob, pdl=True, stream=stream)
            xq = torch.empty((t, G * H * D), dtype=torch.uint8, device=rig.dev)
            xqs = torch.empty(mx.mx_scale_bytes(t, G * H * D), dtype=torch.uint8, device=rig.dev)

            def run_unfused(i, t=t, x=x, pos=pos, q=q, qs=qs, xq=xq, xqs=xqs):
                wq, ws = ww[i % wset][0]
                mx.wo_a_grouped_unfused(h, x, pos, cs, wq, ws, G, H, R, q=q, q_scales=qs, xq=xq,
                                        xq_scales=xqs, stream=stream)
            ua = median_us(torch, run_woa, 30, stream)
            up = median_us(torch, run_pair, 30, stream)
            uu = median_us(torch, run_unfused, 30, stream)
            wa = w_bytes(*pair[0])
            woa[t] = {"wo_a_us": round(ua, 3), "wo_a_weight_gbs": round(wa / (ua * 1e-6) / 1e9, 1),
                      "wo_a_plus_wo_b_us": round(up, 3),
                      "pair_weight_gbs": round((wa + w_bytes(*WOB)) / (up * 1e-6) / 1e9, 1),
                      "wo_a_unfused_us": round(uu, 3),
                      "wo_a_path": "fused kernel" if t <= 8 else "two launches on the handle's scratch"}

    # --------------------------------------------------------------- sweep
    sweep = {}
    mxfp8_peak = 2 * pk["bf16_tflops"]  # the nominal fp8 : bf16 dense ratio times the measured bf16 burst
    if not args.quick:
        for n, k in SWEEP_SHAPES:
            sset = rig.copies(w_bytes(n, k))
            sw = rig.weight_set([(n, k)], seed=4, ncopies=sset)
            for m in SWEEP_M:
                a = mx.mx_quantize_rows(h, rig.activation(m, k, seed=4))
                o = torch.empty((m, n), dtype=torch.bfloat16, device=rig.dev)
                us = median_us(torch, lambda i, a=a, o=o: mx.mx_gemm(
                    h, a[0], a[1], *sw[i % sset][0], out=o, pdl=True, stream=stream), 50, stream)
                tf = 2 * m * n * k / (us * 1e-6) / 1e12
                gbs = gemm_bytes(m, n, k) / (us * 1e-6) / 1e9
                sweep[f"M{m}_N{n}_K{k}"] = {"us": round(us, 3), "gbs": round(gbs, 1),
                                            "hbm_frac": round(gbs / pk["hbm_gbs"], 3),
                                            "tflops": round(tf, 1),
                                            "tensor_frac": round(tf / mxfp8_peak, 3)}

    # --------------------------------------------------- end to end (host I/O)
    # the step's four activations travel as one pinned host buffer and its four
    # outputs come back as one: one copy each way per step
    rows = sum(M_LIST)
    hx_all = torch.cat([xs[m].cpu() for m in M_LIST]).pin_memory()
    dx_all = torch.empty_like(hx_all, device=rig.dev)
    out_all = torch.empty((rows, N1), dtype=torch.bfloat16, device=rig.dev)
    hout_all = torch.empty((rows, N1), dtype=torch.bfloat16).pin_memory()
    offs = {m: sum(M_LIST[:j]) for j, m in enumerate(M_LIST)}
    h2d = rows * K1 * 2
    d2h = rows * N1 * 2

    def e2e_copy_step(i):
        # copy-engine transfers: one pinned host-to-device copy of the activations,
        # one device-to-host copy of the outputs
        with torch.cuda.stream(stream):
            dx_all.copy_(hx_all, non_blocking=True)
            for j, m in enumerate(M_LIST):
                o = offs[m]
                q, s = mx.mx_quantize_rows(h, dx_all[o:o + m], q=qa[m][0], scales=qa[m][1], stream=stream)
                wq, ws = wts[(i * len(M_LIST) + j) % nset][0]
                mx.mx_gemm(h, q, s, wq, ws, out=out_all[o:o + m], pdl=True, stream=stream)
            hout_all.copy_(out_all, non_blocking=True)

    def e2e_step(i):
        # zero-copy: the quantizer reads the activations from the pinned host buffer
        # and the GEMM writes its outputs into the pinned host buffer (the same
        # bytes cross the CPU-GPU link, with no copy-engine transfer in between)
        with torch.cuda.stream(stream):
            for j, m in enumerate(M_LIST):
                o = offs[m]
                q, s = mx.mx_quantize_rows(h, hx_all[o:o + m], q=qa[m][0], scales=qa[m][1], stream=stream)
                wq, ws = wts[(i * len(M_LIST) + j) % nset][0]
                mx.mx_gemm(h, q, s, wq, ws, out=hout_all[o:o + m], pdl=True, stream=stream)
    for i in range(3):
        e2e_step(i)
        e2e_copy_step(i)
    torch.cuda.synchronize()
    # eager: every step issued from Python (host-bound: ~8 calls per step)
    e_steps = min(K, 200)
    st.record(stream)
    for i in range(e_steps):
        e2e_step(i)
    sp.record(stream)
    sp.synchronize()
    e_ms_eager = st.elapsed_time(sp) / e_steps
    # as a decode server runs it: the same calls, copies included, captured once in
    # a CUDA graph (per_graph steps) and replayed
    e_ms = median_us(torch, e2e_step, per_graph, stream, reps) / 1e3
    c_ms = median_us(torch, e2e_copy_step, per_graph, stream, reps) / 1e3
    e2e = {"value": round(world * step_bytes() / (e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
           "ms_per_step": round(e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "path": "public API (mx_quantize_rows, mx_gemm) through the Python binding; the "
                   "quantizer reads each step's activations straight from pinned host memory and "
                   "the GEMM writes its outputs straight into pinned host memory (zero-copy over "
                   "the CPU-GPU link), captured in a CUDA graph and replayed",
           "with_copy_engine": {"value": round(world * step_bytes() / (c_ms * 1e-3) / 1e9, 1),
                                "ms_per_step": round(c_ms, 4),
                                "path": "one pinned host-to-device copy of the activations and one "
                                        "device-to-host copy of the outputs per step"},
           "eager_value": round(world * step_bytes() / (e_ms_eager * 1e-3) / 1e9, 1),
           "eager_ms_per_step": round(e_ms_eager, 4)}

    status = mx.mx_device_status(h)

    # --------------------------------------------------------- CPU baseline
    cpu = None
    if rep.reports and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(args.cpu_seconds)

    if not rep.reports:
        return None
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / pk["hbm_gbs"], 4),
            "traffic": args.traffic if args.traffic is not None else NCU_TRAFFIC.get(gemm_source_sha()),
            "kernel": "gemm_kernel (mx_gemm), mean over M in {1,2,4,8}",
            "peak_kind": f"{pk_kind} hbm_gbs (burst copy)",
            "bytes_per_launch": round(gemm_mix_bytes), "launch_us": round(gemm_launch_us, 3)}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": k_eff,
        "warmup": max(W, 3), "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (x e4m3, fp32 accumulate, bf16 out)",
        "data": "synthetic (SplitMix64/Box-Muller, N(0,1) x 2^U[-6,6] per 32-block)",
        "config": {"workload": "single decode-projection GEMM: mx_quantize_rows + mx_gemm at M in "
                               "{1,2,4,8}, N=2048, K=5120 (one step = the four M values)",
                   "step_bytes": step_bytes(), "pdl": True, "parallelism": f"replicas x{world}",
                   "l2": f"weights rotate over {nset} copies ({nset * w_bytes(N1, K1) / 1e6:.0f} MB "
                         f">= 3x L2 {l2 / 1e6:.0f} MB): inputs larger than L2",
                   "timing": f"median of {reps} replays of a CUDA graph of {per_graph} steps (CUDA "
                             f"events per replay); per-kernel, chain, WO-A and sweep figures: median "
                             f"of {REPLAYS} replays"},
        "gemm_us": {str(m): round(v, 3) for m, v in gemm_us.items()},
        "gemm_gbs": {str(m): round(v, 1) for m, v in gemm_gbs.items()},
        "gemm_frac_of_peak": {str(m): round(v / pk["hbm_gbs"], 3) for m, v in gemm_gbs.items()},
        "quantize_us": {str(m): round(v, 3) for m, v in quant_us.items()},
        "quantize_plus_gemm_fused_us": {str(m): round(v, 3) for m, v in fused_us.items()},
        "chain_us_per_step": chain, "wo_a": woa, "sweep": sweep,
        "sweep_peaks": {"hbm_gbs": pk["hbm_gbs"], "mxfp8_tflops": mxfp8_peak,
                        "mxfp8_peak_kind": f"2 x {pk_kind} bf16 burst"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": k_eff * 2 * len(M_LIST), "clocks": clk, "device_status": status,
    }
    return line


def cpu_baseline(seconds=15.0):
    """The oracle as it stands on the host cores: quantize + fp64 dequantized
    GEMM of the same step, as many whole M values as fit in the time budget."""
    import oracle

    wbits = synth.block_scaled_bf16(1, synth.TAG_W, N1, K1, -6, 6)
    wq, ws = oracle.mx_quantize(synth.bf16_bits_to_f64(wbits))  # offline weight quantization
    done_bytes, t_used, n_gemm = 0, 0.0, 0
    t0 = time.perf_counter()
    while True:
        for m in M_LIST:
            x = synth.bf16_bits_to_f64(synth.block_scaled_bf16(1, synth.TAG_A + m, m, K1, -6, 6))
            ts = time.perf_counter()
            aq, as_ = oracle.mx_quantize(x)
            oracle.round_bf16(oracle.mx_gemm(aq, as_, wq, ws))
            t_used += time.perf_counter() - ts
            done_bytes += gemm_bytes(m, N1, K1) + quant_bytes(m, K1)
            n_gemm += 1
        if time.perf_counter() - t0 > seconds or n_gemm >= 40:
            break
    threads = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        pass
    return {"value": round(done_bytes / t_used / 1e9, 3), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{n_gemm} oracle quantize+GEMM calls of the step's M values "
                      f"({t_used:.1f} s CPU wall); weight quantized once outside the timing",
            "ms_per_step": round(t_used / (n_gemm / len(M_LIST)) * 1e3, 1)}


def run_reference(args):
    """--impl reference: the CPU oracle on the same workload and metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle

    wbits = synth.block_scaled_bf16(1, synth.TAG_W, N1, K1, -6, 6)
    wq, ws = oracle.mx_quantize(synth.bf16_bits_to_f64(wbits))
    xs = {m: synth.bf16_bits_to_f64(synth.block_scaled_bf16(1, synth.TAG_A + m, m, K1, -6, 6))
          for m in M_LIST}

    def one_step():
        for m in M_LIST:
            aq, as_ = oracle.mx_quantize(xs[m])
            oracle.round_bf16(oracle.mx_gemm(aq, as_, wq, ws))
    for _ in range(args.warmup):
        one_step()
    steps = max(1, args.steps)
    t0 = time.perf_counter()
    budget = 120.0
    done = 0
    for _ in range(steps):
        one_step()
        done += 1
        if time.perf_counter() - t0 > budget:
            break
    sec = (time.perf_counter() - t0) / done
    value = step_bytes() / sec / 1e9
    threads = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        pass
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": done, "warmup": args.warmup,
            "ms_per_step": round(sec * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "single decode-projection GEMM: quantize + GEMM at M in "
                                   "{1,2,4,8}, N=2048, K=5120 (CPU oracle, numpy float64)"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": f"{done} whole steps"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_profile(args):
    """A few plain (non-graph) launches of one kernel family for ncu."""
    import torch

    import mxfp8_block_scaled_06_gb300 as mx
    from mxfp8_block_scaled_06_gb300 import build as mxbuild

    mxbuild.build()
    torch.cuda.set_device(0)
    h = mx.mx_create(0)
    rig = Rig(torch, mx, h, 126 * 2**20)
    if args.profile == "gemm":
        w = rig.weight_set([(N1, K1)], 1, 4)
        for m in (1, 8):
            q = mx.mx_quantize_rows(h, rig.activation(m, K1, 1))
            for i in range(3):
                mx.mx_gemm(h, q[0], q[1], *w[i % 4][0], pdl=True)
    elif args.profile == "bf16":
        w = rig.weight_set([(N1, K1)], 1, 4)
        for m in (1, 8):
            x = rig.activation(m, K1, 1)
            for i in range(3):
                mx.mx_gemm_bf16(h, x, *w[i % 4][0], pdl=True)
    elif args.profile == "chain":
        cw = rig.weight_set(CHAIN_SHAPES, 2, 2)
        for m in (8, 64):
            q = mx.mx_quantize_rows(h, rig.activation(m, CHAIN_SHAPES[0][1], 2, -4, 4))
            for i in range(2):
                mx.mx_gemm_chain(h, q[0], q[1], cw[i % 2], g1_cols=CHAIN_G1_COLS)
    elif args.profile == "wo_a":
        G, H, R, D = WOA["G"], WOA["H"], WOA["R"], WOA["D"]
        ww = rig.weight_set([(G * R, H * D)], 3, 2)
        cs = torch.from_numpy(synth.rope_cos_sin_cache(65536)).cuda()
        for t in WOA_T:
            x = torch.from_numpy(synth.normal_bf16(3, synth.TAG_X, (t, G * H, D)).view(np.int16)).view(torch.bfloat16).cuda()
            pos = torch.from_numpy(synth.positions(3, synth.TAG_POS, t)).cuda()
            for i in range(2):
                mx.wo_a_grouped(h, x, pos, cs, *ww[i % 2][0], G, H, R)
    elif args.profile == "sweep":
        for n, k in SWEEP_SHAPES:
            w = rig.weight_set([(n, k)], 4, 2)
            for m in (64, 256):
                q = mx.mx_quantize_rows(h, rig.activation(m, k, 4))
                for i in range(2):
                    mx.mx_gemm(h, q[0], q[1], *w[i % 2][0])
    torch.cuda.synchronize()
    assert mx.mx_device_status(h) == mx.MX_OK
    print(json.dumps({"profile": args.profile, "ok": True}))


TIMELINE_SLOTS = {"entry": 0, "setup": 1, "w_issued": 2, "wsf_landed": 3, "wait_ret": 4,
                  "rms_done": 13, "x_landed": 14, "act_quantized": 12, "first_full": 5, "last_full": 15,
                  "second_full": 18, "mma_issued": 16, "accum": 6, "red_pass": 7, "red_done": 8,
                  "exit": 9}
TIMELINE_EXIT = TIMELINE_SLOTS["exit"]


def run_timeline(args):
    """--timeline: per-CTA %globaltimer stamps of GEMM launches (the timeline
    build of libmx, -DMX_TIMELINE) in CUDA graphs of back-to-back launches with
    PDL. For every launch after the first, each phase is reported relative to the
    previous launch's last CTA exit (median and range over the launch's CTAs,
    then the median over launches); the weights rotate over >= 3x L2."""
    import ctypes

    import torch

    import mxfp8_block_scaled_06_gb300 as mx
    from mxfp8_block_scaled_06_gb300 import build as mxbuild

    lib = mx.load_library(mxbuild.build_timeline())
    lib.mx_timeline_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                     ctypes.POINTER(ctypes.c_int)]
    lib.mx_timeline_reset.argtypes = [ctypes.c_void_p]
    ctas, slots, launches = 512, 20, 256
    torch.cuda.set_device(0)
    h = mx.mx_create(0)
    props = torch.cuda.get_device_properties(0)
    rig = Rig(torch, mx, h, getattr(props, "L2_cache_size", 126 * 2**20))
    stream = torch.cuda.Stream()

    def record(fn, per_graph, period=1, names=None):
        """Timeline of per_graph calls of fn. period > 1: each call makes
        `period` launches, reported separately (by `names`)."""
        with torch.cuda.stream(stream):
            fn(0)  # tensor maps and plans outside the capture
        torch.cuda.synchronize()
        assert lib.mx_timeline_reset(h.ptr) == 0  # slots from here on belong to the captured launches
        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(per_graph):
                    fn(i)
        torch.cuda.synchronize()
        st, sp = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            st.record(stream)
            for _ in range(5):
                g.replay()
            sp.record(stream)
        sp.synchronize()
        ms = st.elapsed_time(sp)
        n = ctypes.c_int(0)
        buf = np.zeros(launches * ctas * slots, dtype=np.uint64)
        assert lib.mx_timeline_read(h.ptr, buf.ctypes.data, buf.nbytes, ctypes.byref(n)) == 0
        tl = buf.reshape(launches, ctas, slots)[: n.value]
        e = TIMELINE_EXIT
        res = {}
        for pos in range(period):
            phases = {k: [] for k in TIMELINE_SLOTS}
            spread = {k: [] for k in TIMELINE_SLOTS}
            dur, early, landed_early = [], [], []
            for i in range(pos if pos > 0 else period, len(tl), period):
                prev = tl[i - 1][tl[i - 1][:, e] > 0]
                cur = tl[i][tl[i][:, e] > 0]
                if len(prev) == 0 or len(cur) == 0:
                    continue
                p_end = int(prev[:, e].max())
                rel = cur.astype(np.int64) - p_end
                dur.append((int(cur[:, e].max()) - p_end) / 1e3)
                early.append(float((rel[:, 0] < 0).mean()))
                landed_early.append(float(((rel[:, 3] < 0) & (cur[:, 3] > 0)).mean()))
                for k, j in TIMELINE_SLOTS.items():
                    v = rel[:, j][cur[:, j] > 0]
                    if len(v):
                        phases[k].append(float(np.median(v)))
                        spread[k].append(float(v.max() - v.min()))
            landed = [float(np.median(tl[i][tl[i][:, e] > 0][:, 17])) for i in range(max(1, pos), len(tl), period)
                      if (tl[i][:, e] > 0).any()]
            res[names[pos] if names else pos] = {
                "stages_landed_at_wait_median": float(np.median(landed)) if landed else None,
                "launch_us_median": round(float(np.median(dur)), 3) if dur else None,
                "ctas_started_before_previous_end": round(float(np.median(early)), 3) if early else None,
                "weight_scales_landed_before_previous_end": round(float(np.median(landed_early)), 3)
                if landed_early else None,
                "phase_ns_vs_previous_end": {k: int(np.median(v)) for k, v in phases.items() if v},
                "phase_spread_ns_over_ctas": {k: int(np.median(v)) for k, v in spread.items() if v}}
        out = {"us_per_graph_item": round(ms * 1e3 / (5 * per_graph), 3)}
        if period == 1:
            out.update(res[0])
        else:
            out["launches"] = res
        return out

    out = {}
    nset = rig.copies(w_bytes(N1, K1))
    wts = rig.weight_set([(N1, K1)], seed=1, ncopies=nset)
    for m in (1, 8, 64):
        q = mx.mx_quantize_rows(h, rig.activation(m, K1, seed=1))
        o = torch.empty((m, N1), dtype=torch.bfloat16, device=rig.dev)
        for pdl in (True, False):
            out[f"gemm_M{m}" + ("" if pdl else "_no_pdl")] = record(
                lambda i, q=q, o=o, pdl=pdl: mx.mx_gemm(h, q[0], q[1], *wts[i % nset][0], out=o, pdl=pdl,
                                                        stream=stream), 12)
    xs = {m: rig.activation(m, K1, seed=1) for m in M_LIST}
    qa = {m: mx.mx_quantize_rows(h, xs[m]) for m in M_LIST}
    outs = {m: torch.empty((m, N1), dtype=torch.bfloat16, device=rig.dev) for m in M_LIST}

    def step(i):
        for j, m in enumerate(M_LIST):
            mx.mx_quantize_rows(h, xs[m], q=qa[m][0], scales=qa[m][1], stream=stream)
            mx.mx_gemm(h, qa[m][0], qa[m][1], *wts[(i * len(M_LIST) + j) % nset][0], out=outs[m],
                       pdl=True, stream=stream)
    out["step"] = record(step, 3)
    cset = rig.copies(sum(w_bytes(n, k) for n, k in CHAIN_SHAPES))
    cw = rig.weight_set(CHAIN_SHAPES, seed=2, ncopies=cset)
    for m in (1, 4, 16, 64):
        q1 = mx.mx_quantize_rows(h, rig.activation(m, CHAIN_SHAPES[0][1], seed=2, umin=-4, umax=4))
        bufs = dict(out=torch.empty((m, CHAIN_SHAPES[2][0]), dtype=torch.bfloat16, device=rig.dev),
                    a2=torch.empty((m, CHAIN_G1_COLS), dtype=torch.uint8, device=rig.dev),
                    a2_scales=torch.empty(mx.mx_scale_bytes(m, CHAIN_G1_COLS), dtype=torch.uint8, device=rig.dev),
                    a3=torch.empty((m, CHAIN_SHAPES[1][0]), dtype=torch.uint8, device=rig.dev),
                    a3_scales=torch.empty(mx.mx_scale_bytes(m, CHAIN_SHAPES[1][0]), dtype=torch.uint8,
                                          device=rig.dev))
        out[f"chain_M{m}"] = record(lambda i, q1=q1, bufs=bufs: mx.mx_gemm_chain(
            h, q1[0], q1[1], cw[i % cset], g1_cols=CHAIN_G1_COLS, stream=stream, **bufs), 4,
            period=3, names=("G1", "G2", "G3"))
        out1 = torch.empty((m, CHAIN_SHAPES[0][0]), dtype=torch.bfloat16, device=rig.dev)
        nw = torch.from_numpy(synth.norm_weight_bf16(4, CHAIN_G1_COLS).view(np.int16)).view(
            torch.bfloat16).to(rig.dev)
        out[f"chain_norm_M{m}"] = record(lambda i, q1=q1, bufs=bufs, out1=out1, nw=nw: mx.mx_gemm_chain_norm(
            h, q1[0], q1[1], cw[i % cset], nw, 1e-6, g1_cols=CHAIN_G1_COLS, out1=out1, stream=stream,
            **bufs), 4, period=3,
            names=("G1", "G2+norm", "G3") if m <= 16 else ("G1", "G2 (after the norm kernel)", "G3"))
    # WO-A (fused, with the push exchange up to 16 tokens), alone and followed by wo_b
    G, H, R, D = WOA["G"], WOA["H"], WOA["R"], WOA["D"]
    pair = [(G * R, H * D), WOB]
    wset = rig.copies(sum(w_bytes(n, k) for n, k in pair))
    ww = rig.weight_set(pair, seed=3, ncopies=wset)
    cs = torch.from_numpy(synth.rope_cos_sin_cache(65536)).to(rig.dev)
    for t in (1, 8):
        x = torch.from_numpy(synth.normal_bf16(3 + t, synth.TAG_X, (t, G * H, D)).view(np.int16)).view(
            torch.bfloat16).to(rig.dev)
        pos = torch.from_numpy(synth.positions(3 + t, synth.TAG_POS, t)).to(rig.dev)
        q = torch.empty((t, G * R), dtype=torch.uint8, device=rig.dev)
        qs = torch.empty(mx.mx_scale_bytes(t, G * R), dtype=torch.uint8, device=rig.dev)
        ob = torch.empty((t, WOB[0]), dtype=torch.bfloat16, device=rig.dev)

        def woa(i, x=x, pos=pos, q=q, qs=qs):
            mx.wo_a_grouped(h, x, pos, cs, *ww[i % wset][0], G, H, R, q=q, q_scales=qs, early_trigger=True,
                            stream=stream)

        def woa_wob(i, q=q, qs=qs, ob=ob):
            woa(i)
            mx.mx_gemm(h, q, qs, *ww[i % wset][1], out=ob, pdl=True, stream=stream)
        out[f"wo_a_T{t}"] = record(woa, 12)
        out[f"wo_a_wo_b_T{t}"] = record(woa_wob, 6, period=2, names=("WO-A", "wo_b"))
    for n, k in SWEEP_SHAPES:
        ws = rig.weight_set([(n, k)], seed=4, ncopies=rig.copies(w_bytes(n, k)))
        for m in (32, 64, 128, 192, 256):
            q = mx.mx_quantize_rows(h, rig.activation(m, k, seed=4))
            o = torch.empty((m, n), dtype=torch.bfloat16, device=rig.dev)
            out[f"gemm_M{m}_N{n}_K{k}"] = record(
                lambda i, q=q, o=o, ws=ws: mx.mx_gemm(h, q[0], q[1], *ws[i % len(ws)][0], out=o, pdl=True,
                                                      stream=stream), 6)
    torch.cuda.synchronize()
    assert mx.mx_device_status(h) == mx.MX_OK
    print(json.dumps({"timeline": out}))


TUNE_M = (1, 2, 4, 8, 16, 32, 48, 64, 96, 128, 192, 256)


def run_tune_chain(args):
    """--tune-chain: the K-split count and ring depth of each chain projection,
    timed inside the graph-replayed mx_gemm_chain (not as isolated launches).
    Per row count, greedily G1, then G2, then G3: each candidate (splits in
    1..8, ring depth as planned or every chunk of the K-range resident) is set
    for that projection alone through MX_PLAN_AT (on a handle created for the
    candidate: overrides are read at mx_create), the projections already
    chosen keep their pick, the rest their current plan; weights rotate over
    >= 3x L2; each time is the median of 10 replays of 20 chained calls."""
    import torch

    import mxfp8_block_scaled_06_gb300 as mx
    from mxfp8_block_scaled_06_gb300 import build as mxbuild

    mxbuild.build()
    torch.cuda.set_device(0)
    h = mx.mx_create(0)
    props = torch.cuda.get_device_properties(0)
    rig = Rig(torch, mx, h, getattr(props, "L2_cache_size", 126 * 2**20))
    stream = torch.cuda.Stream()
    cset = rig.copies(sum(w_bytes(n, k) for n, k in CHAIN_SHAPES))
    cw = rig.weight_set(CHAIN_SHAPES, seed=2, ncopies=cset)
    spec = lambda picks: ",".join(f"{n}x{k}:{s}" + (f":{st}" if st else "")
                                  for (n, k), (s, st) in picks.items())
    out = {}
    for m in (TUNE_M if not args.tune_rows else [int(v) for v in args.tune_rows.split(",")]):
        q1 = mx.mx_quantize_rows(h, rig.activation(m, CHAIN_SHAPES[0][1], seed=2, umin=-4, umax=4))
        bufs = dict(out=torch.empty((m, CHAIN_SHAPES[2][0]), dtype=torch.bfloat16, device=rig.dev),
                    a2=torch.empty((m, CHAIN_G1_COLS), dtype=torch.uint8, device=rig.dev),
                    a2_scales=torch.empty(mx.mx_scale_bytes(m, CHAIN_G1_COLS), dtype=torch.uint8,
                                          device=rig.dev),
                    a3=torch.empty((m, CHAIN_SHAPES[1][0]), dtype=torch.uint8, device=rig.dev),
                    a3_scales=torch.empty(mx.mx_scale_bytes(m, CHAIN_SHAPES[1][0]), dtype=torch.uint8,
                                          device=rig.dev))

        def timed(plan_at, q1=q1, bufs=bufs):
            # a handle reads the plan overrides once, when it is created
            if plan_at:
                os.environ["MX_PLAN_AT"] = plan_at
            else:
                os.environ.pop("MX_PLAN_AT", None)
            hc = mx.mx_create(0)
            os.environ.pop("MX_PLAN_AT", None)
            try:
                return median_us(torch, lambda i: mx.mx_gemm_chain(
                    hc, q1[0], q1[1], cw[i % cset], g1_cols=CHAIN_G1_COLS, stream=stream, **bufs), 20, stream)
            finally:
                hc.close()

        current = timed("")
        picks, cands = {}, {}
        # ring depth candidates: 0 = as planned, 3 = shallow (room for the next
        # kernel's CTAs beside this one's), 12 = the whole K-range resident
        depths = (0, 3, 12) if args.tune_rounds > 1 else (0, 12)
        for rnd in range(args.tune_rounds):
            for n, k in CHAIN_SHAPES:
                times = {}
                for s in range(1, min(8, k // 128) + 1):
                    for st in depths:
                        try:
                            times[(s, st)] = timed(spec({**picks, (n, k): (s, st)}))
                        except mx.MxError:  # no plan fits shared memory: the library rejects it
                            pass
                best = min(times, key=times.get)
                picks[(n, k)] = best
                cands[f"{n}x{k}" + (f"_round{rnd + 1}" if args.tune_rounds > 1 else "")] = {
                    f"s{s}" + (f"_st{st}" if st else ""): round(t, 3) for (s, st), t in times.items()}
        tuned = timed(spec(picks))
        out[m] = {"current_us": round(current, 3), "tuned_us": round(tuned, 3), "MX_PLAN_AT": spec(picks),
                  "candidates_us": cands}
        print(json.dumps({m: out[m]}), file=sys.stderr, flush=True)
    torch.cuda.synchronize()
    assert mx.mx_device_status(h) == mx.MX_OK
    print(json.dumps({"tune_chain": out}))


def launch_replicas(n):
    """bench.py --gpus N outside torchrun: N processes of this script, rank i on
    GPU i (RANK = LOCAL_RANK = i, WORLD_SIZE = N, rendezvous on 127.0.0.1), with
    the same arguments; rank 0 alone prints. Returns the largest exit code."""
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    procs = []
    for i in range(n):
        env = dict(os.environ, RANK=str(i), LOCAL_RANK=str(i), WORLD_SIZE=str(n),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__)] + sys.argv[1:], env=env))
    return max(p.wait() for p in procs)


def replica_selftest():
    """--replica-selftest: the replicas' host-side coordination without a GPU (a
    gloo barrier and the maximum over ranks of rank + 1); rank 0 prints it."""
    rep = Replicas()
    rep.barrier()
    top = rep.max_over_ranks(float(rep.rank + 1))
    if rep.reports:
        print(json.dumps({"n_gpus": rep.world, "max_over_ranks": top}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="skip the chain and WO-A extras")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per GEMM launch from an ncu capture of the current kernel")
    ap.add_argument("--profile", default=None, choices=["gemm", "bf16", "chain", "wo_a", "sweep"])
    ap.add_argument("--timeline", action="store_true",
                    help="per-CTA phase timeline of GEMM launches (builds the -DMX_TIMELINE library)")
    ap.add_argument("--tune-chain", action="store_true",
                    help="time each chain projection's K-split / ring-depth candidates inside the chain")
    ap.add_argument("--tune-rows", default="", help="row counts for --tune-chain, e.g. 64,128")
    ap.add_argument("--tune-rounds", type=int, default=1,
                    help="greedy rounds of --tune-chain (more than one also tries a 3-stage ring)")
    ap.add_argument("--replica-selftest", action="store_true",
                    help="the replicas' host-side coordination only (no GPU), e.g. with --gpus 2")
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_replicas(args.gpus))
    if args.replica_selftest:
        replica_selftest()
        return
    if args.timeline:
        run_timeline(args)
        return
    if args.tune_chain:
        run_tune_chain(args)
        return
    if args.profile:
        run_profile(args)
        return
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
