#!/usr/bin/env python
"""Benchmark of the LM-head loss path on GB300.

One step = one call of each entry point on its largest workload:
  ce_fwd_f32       logits fp32 [16384, 131072] ~ N(0,1)           (8.6 GB)
  ce_fwd_sbv_bf16  logits bf16 [2048, 4, 131072] ~ N(0, 2^2)       (2.1 GB)
  flce_fwd_bf16    x bf16 [16*1024, 4096], W bf16 [128256, 4096]  (17.2 TFLOP)
  fljsd_fwd_bf16   xs, xt bf16 [8192, 4096], Ws, Wt [128256, 4096] (34.4 TFLOP)
Every input is larger than L2, and consecutive calls read different buffers,
so no L2 flush is needed between timed steps.  Inputs come from the seeded
generator (gen/), made on the host into pinned memory and copied to the GPU
once; `value` times device-resident inputs, `e2e` re-copies every input from
pinned host memory and reads the results back inside each timed step.

Prints ONE JSON line.  `--impl reference` times the fp64 CPU oracle on
bounded samples of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from lm_head_online_gb300 import roofline as rl  # noqa: E402

METRIC = "CE µs & HBM GB/s vs roofline; fused-linear µs & TFLOP/s vs bf16 peak (1 GB300)"
UNIT = "us/step"

CE = dict(T=16384, V=131072)
SBV = dict(S=2048, B=4, V=131072)
FLCE = dict(T=16 * 1024, H=4096, V=128256)
FLJSD = dict(T=8192, H=4096, V=128256)
WORKLOAD = ("ce_fwd_f32 fp32[16384,131072] + ce_fwd_sbv_bf16 bf16[2048,4,131072] + "
            "flce_fwd_bf16 x[16384,4096] W[128256,4096] + fljsd_fwd_bf16 T=8192 H=4096 V=128256 beta=0.5")
KERNELS_PER_STEP = 2 + 1 + 2 + 4   # ce_fwd_f32: row kernel + mean; sbv 1; flce 2; fljsd 4

# The workload table's smallest CE configurations (the pages' own "Estimated
# floor" workloads), timed after the step, each alone: fp32 [16384, 4096] and
# Megatron bf16 [2048, 4, V] for V = 4096 and 8192.
SMALL_CE = (("ce_fwd_f32", 16384, 4096), ("ce_fwd_sbv_bf16", 2048, 4096), ("ce_fwd_sbv_bf16", 2048, 8192))
L2_BYTES = 129 * 2 ** 20
# Host seconds of one timed oracle step, the same for the bench's cpu_baseline
# leg and every step of the reference arm (so the two time the same sample).
ORACLE_BUDGET_S = 6.0

# DRAM bytes (read + write) per launch of each main kernel at the bench sizes,
# scaled from small-case ncu captures of the same kernel sources (their summaries
# are under profiles/, named for the kernels and workloads):
# the tensor-core passes were captured at T = 4096 and their traffic follows T
# (W is re-read once per raster group of fixed token span): flce x 4 (T 16384),
# the log-sum-exp and divergence passes x 2 (T 8192).  The row kernels read the
# logits once (read / algorithmic = 1.0003 at V = 4096), so theirs is that ratio
# times the full-size logits and targets, plus the per-token losses written.
# The figures hold only for the sources they were taken from: a changed source
# makes the bench report null.
KERNEL_SOURCES = ("fused_linear.cu", "ce_rows.cu", "rowstats.cuh", "ptx.cuh", "lmho_internal.h")
TRAFFIC_SOURCE_DIGEST = "de5eec69d443197c"
TRAFFIC_BYTES = {
    "ce_fwd_f32.row_kernel_and_mean": int((16384 * 131072 * 4 + 16384 * 8) * 1.0003) + 16384 * 4 + 4,
    "ce_fwd_sbv_bf16.row_kernel": int((8192 * 131072 * 2 + 8192 * 8) * 1.0003) + 8192 * 4,
    "flce.tcgen05_gemm_ce": 4 * (1084856576 + 19516032),
    "fljsd.tcgen05_gemm_lse": 2 * (2169060352 + 35975936),
    "fljsd.tcgen05_gemm_jsd": 2 * (4777500672 + 20122880),
}


def kernel_source_digest():
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "lm_head_online_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_of(kernel):
    return TRAFFIC_BYTES.get(kernel) if kernel_source_digest() == TRAFFIC_SOURCE_DIGEST else None


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-small-ce", action="store_true", help="skip the small CE configurations after the step")
    ap.add_argument("--small-ce-only", action="store_true",
                    help="only the small CE configurations (timed back to back and flushed, with the bare read of "
                         "the same bytes); prints their JSON line (used for launch lists of the small calls)")
    ap.add_argument("--tp", action="store_true",
                    help="vocab-parallel Megatron CE: bf16 [2048, 4, 131072] with the vocab sharded over the N ranks "
                         "(partials, one NCCL all-gather, merge); prints its own JSON line")
    ap.add_argument("--tp-fused", action="store_true",
                    help="vocab-parallel fused linear + CE (x [16384, 4096]) and + JSD (xs, xt [8192, 4096]) with the "
                         "rows of W [128256, 4096] (both heads) sharded over the N ranks; prints its own JSON line")
    ap.add_argument("--e2e-clocks", action="store_true",
                    help="also sample clocks during the e2e region (nvidia-smi polling slows host copies)")
    ap.add_argument("--sweep", action="store_true",
                    help="time every configuration of the workload table (one JSON line each)")
    ap.add_argument("--case", choices=["ce", "sbv", "flce", "fljsd", "ce_fb", "sbv_fb", "flce_fb", "fljsd_fb", "cpo",
                                       "cpo_fb", "cublas"],
                    help="time one op alone at --T/--V/--H (profiling runs); prints one JSON line")
    ap.add_argument("--T", type=int, default=None, help="tokens (ce: rows; sbv: seq, batch 4)")
    ap.add_argument("--V", type=int, default=None)
    ap.add_argument("--H", type=int, default=4096)
    ap.add_argument("--ce-variant", default="auto")
    ap.add_argument("--raster-group", type=int, default=0, help="fused kernels: token tiles per raster group (0 = auto)")
    return ap.parse_args()


# ---------------------------------------------------------------- peaks
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p["bf16_tflops_sustained"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        if self.index < 0:
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            c = [x.strip() for x in ln.split(",")]
            if len(c) < 8:
                continue
            try:
                sm.append(float(c[0]))
                mx = max(mx, float(c[1]))
            except ValueError:
                continue
            for n, v in zip(names, c[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- inputs
def make_inputs(seed, torch, pinned=True):
    import gen
    thr = os.cpu_count() or 1

    def host(shape, dtype):
        t = torch.empty(shape, dtype=dtype)
        return t.pin_memory() if pinned else t

    h = {}
    h["ce_z"] = host((CE["T"], CE["V"]), torch.float32)
    gen.normal_f32(seed, gen.STREAM_LOGITS, h["ce_z"].shape, 1.0, out=h["ce_z"], threads=thr)
    h["ce_t"] = host((CE["T"],), torch.int64)
    gen.targets(seed, gen.STREAM_TARGET, h["ce_t"].shape, CE["V"], out=h["ce_t"], threads=thr)
    h["sbv_z"] = host((SBV["S"], SBV["B"], SBV["V"]), torch.bfloat16)
    gen.normal_bf16_bits(seed, gen.STREAM_LOGITS, h["sbv_z"].shape, 2.0, out=h["sbv_z"].view(torch.int16), threads=thr)
    h["sbv_t"] = host((SBV["S"], SBV["B"]), torch.int64)
    gen.targets(seed, gen.STREAM_TARGET, h["sbv_t"].shape, SBV["V"], out=h["sbv_t"], threads=thr)
    h["fl_x"] = host((FLCE["T"], FLCE["H"]), torch.bfloat16)
    gen.normal_bf16_bits(seed, gen.STREAM_X, h["fl_x"].shape, 1.0, out=h["fl_x"].view(torch.int16), threads=thr)
    h["fl_w"] = host((FLCE["V"], FLCE["H"]), torch.bfloat16)
    gen.normal_bf16_bits(seed, gen.STREAM_W, h["fl_w"].shape, 0.02, out=h["fl_w"].view(torch.int16), threads=thr)
    h["fl_t"] = host((FLCE["T"],), torch.int64)
    gen.targets(seed, gen.STREAM_TARGET, h["fl_t"].shape, FLCE["V"], out=h["fl_t"], threads=thr)
    for k, stream, shape, sig in (("js_xs", gen.STREAM_X, (FLJSD["T"], FLJSD["H"]), 1.0),
                                  ("js_ws", gen.STREAM_W, (FLJSD["V"], FLJSD["H"]), 0.02),
                                  ("js_xt", gen.STREAM_XT, (FLJSD["T"], FLJSD["H"]), 1.0),
                                  ("js_wt", gen.STREAM_WT, (FLJSD["V"], FLJSD["H"]), 0.02)):
        h[k] = host(shape, torch.bfloat16)
        gen.normal_bf16_bits(seed, stream, shape, sig, out=h[k].view(torch.int16), threads=thr)
    return h


# ---------------------------------------------------------------- small CE calls
def rotating_copies(x, torch, min_total=3 * L2_BYTES):
    """x and enough device copies of it that a call on copy i % R reads bytes
    not touched during the previous ~3 L2 capacities of reads."""
    nbytes = x.numel() * x.element_size()
    R = max(2, -(-min_total // nbytes))
    return [x] + [x.clone() for _ in range(R - 1)]


def time_flushed(fns, torch, warmup, steps, flush):
    """Per-call time: a 512 MB read (L2 flush) before each call, CUDA events
    recorded around the call on its stream."""
    for i in range(warmup):
        fns[i % len(fns)]()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i, (e0, e1) in enumerate(evs):
        flush.sum()
        e0.record()
        fns[i % len(fns)]()
        e1.record()
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) * 1e3 for e0, e1 in evs]


def time_back_to_back(fns, torch, warmup, steps):
    """Per-call time of `steps` calls issued back to back on one stream, call i
    reading copy i % R of the input (R copies > 3x L2), one event pair around
    all of them: no per-call event cost, every call's logits come from HBM.
    The calls are queued behind a sleeping kernel (~60 us of GPU time per
    call), so the host, which takes tens of microseconds per call, is ahead
    of the GPU and no call waits for its launch."""
    for i in range(warmup):
        fns[i % len(fns)]()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(2e6 + 1.2e5 * steps))
    e0.record()
    for i in range(steps):
        fns[i % len(fns)]()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / steps


def time_graph(fns, torch, steps, replays=3):
    """Per-call time of the same back-to-back sequence captured once into a
    CUDA graph (after an eager warm-up of every call on the capture stream's
    side) and replayed: median over `replays` replays of one event pair around
    the replay, graph launch included.  Inside a graph the next kernel is
    already staged when the previous one completes, so the gap between calls
    shrinks; the calls and their results are the same."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for f in fns:
            f()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(steps):
            fns[i % len(fns)]()
    g.replay()
    torch.cuda.synchronize()
    per = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        per.append(e0.elapsed_time(e1) * 1e3 / steps)
    del g
    return float(np.median(per))


def run_small_ce_only(args):
    import torch
    import lm_head_online_gb300 as lmho
    torch.cuda.set_device(0)
    lmho.load()
    pk = peaks()
    ops, roofs, _ = small_ce(lmho, torch, torch.device("cuda", 0), args.seed, pk, steps=args.steps)
    return {"metric": "small CE calls, us per call", "peaks": pk["src"], "ops": ops, "rooflines": roofs,
            "steps": args.steps}


def small_ce(lmho, torch, dev, seed, pk, steps=50):
    """The smallest CE workloads, each timed alone (see above): back to back
    on the stream (the roofline's time), the same calls replayed from one CUDA
    graph (a second roofline entry, "<op>.graph"), and one flushed call at a
    time, which adds a fixed event and launch cost of about 3 us; beside them
    the back-to-back time of a bare read of the same bytes with the same loads
    (lmho_probe_read): the stream floor at that size."""
    import gen
    thr = os.cpu_count() or 1
    flush = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    ops, roofs = {}, {}
    for name, T, V in SMALL_CE:
        if name == "ce_fwd_f32":
            z = torch.from_numpy(gen.normal_f32(seed, gen.STREAM_LOGITS, (T, V), 1.0, threads=thr)).to(dev)
            t = torch.from_numpy(gen.targets(seed, gen.STREAM_TARGET, (T,), V, threads=thr)).to(dev)
            ws = lmho.workspace(lmho.ce_workspace_bytes(T, V), dev)
            loss = torch.empty(1, device=dev)
            copies = rotating_copies(z, torch)
            fns = [lambda zz=zz: lmho.ce_fwd_f32(zz, t, loss=loss, ws=ws) for zz in copies]
            nbytes, key, shape = rl.ce_flat_bytes(T, V), f"ce_fwd_f32.T{T}_V{V}", f"fp32[{T},{V}]"
        else:
            z = torch.empty((T, 4, V), dtype=torch.bfloat16)
            gen.normal_bf16_bits(seed, gen.STREAM_LOGITS, (T, 4, V), 2.0, out=z.view(torch.int16), threads=thr)
            z = z.to(dev)
            t = torch.from_numpy(gen.targets(seed, gen.STREAM_TARGET, (T, 4), V, threads=thr)).to(dev)
            loss = torch.empty((T, 4), device=dev)
            copies = rotating_copies(z, torch)
            fns = [lambda zz=zz: lmho.ce_fwd_sbv_bf16(zz, t, loss=loss) for zz in copies]
            nbytes, key, shape = rl.ce_sbv_bytes(T, 4, V), f"ce_fwd_sbv_bf16.S{T}_B4_V{V}", f"bf16[{T},4,{V}]"
        b2b = time_back_to_back(fns, torch, 5, steps)
        gr = time_graph(fns, torch, steps)
        fl = time_flushed(fns, torch, 5, steps, flush)
        # the bare read of the same bytes with the same loads (nothing computed)
        seg = z.shape[-1] * z.element_size()
        probe_out = torch.empty(z.numel() * z.element_size() // seg, dtype=torch.int32, device=dev)
        reads = [lambda c=c: lmho.probe_read(c, seg, out=probe_out) for c in copies]
        floor = time_back_to_back(reads, torch, 5, steps)
        med = float(np.median(fl))
        gbs = nbytes / (b2b * 1e-6) / 1e9
        ops[key] = {"shape": shape, "bytes": nbytes, "copies": len(fns),
                    "us_back_to_back": round(b2b, 2), "GB/s_back_to_back": round(gbs, 1),
                    "us_graph": round(gr, 2), "GB/s_graph": round(nbytes / (gr * 1e-6) / 1e9, 1),
                    "us_bare_read_back_to_back": round(floor, 2),
                    "frac_of_bare_read": round(floor / b2b, 4),
                    "us_flushed_median": round(med, 2), "us_flushed_p10": round(float(np.percentile(fl, 10)), 2),
                    "GB/s_flushed": round(nbytes / (med * 1e-6) / 1e9, 1),
                    "frac_flushed": round(nbytes / (med * 1e-6) / 1e9 / pk["hbm"], 4)}
        roofs[key] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                      "frac": round(gbs / pk["hbm"], 4), "traffic": None,
                      "timing": f"back to back over {len(fns)} copies (> 3x L2), mean per call"}
        gg = nbytes / (gr * 1e-6) / 1e9
        roofs[key + ".graph"] = {"bound": "hbm", "achieved": round(gg, 1), "peak": pk["hbm"], "unit": "GB/s",
                                 "frac": round(gg / pk["hbm"], 4), "traffic": None,
                                 "timing": f"the same {steps} calls captured in one CUDA graph, median of 3 replays "
                                           f"(graph launch included), mean per call"}
        del fns, reads, copies, z
        torch.cuda.empty_cache()
    return ops, roofs, (2 + 3) * steps * sum(2 if n == "ce_fwd_f32" else 1 for n, _, _ in SMALL_CE)


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import lm_head_online_gb300 as lmho

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lmho.load()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    t_gen = time.time()
    h = make_inputs(args.seed + rank, torch)
    t_gen = time.time() - t_gen
    d = {k: v.to(dev, non_blocking=True) for k, v in h.items()}
    torch.cuda.synchronize()

    ws_ce = lmho.workspace(lmho.ce_workspace_bytes(CE["T"], CE["V"]), dev)
    ws_fl = lmho.workspace(lmho.flce_workspace_bytes(FLCE["T"], FLCE["H"], FLCE["V"]), dev)
    ws_js = lmho.workspace(lmho.fljsd_workspace_bytes(FLJSD["T"], FLJSD["H"], FLJSD["V"]), dev)
    out = {"ce": torch.empty(1, device=dev), "sbv": torch.empty((SBV["S"], SBV["B"]), device=dev),
           "fl": torch.empty(1, device=dev), "js": torch.empty(1, device=dev)}
    stream = torch.cuda.current_stream()

    # per-kernel events: ce 2, sbv 2, flce 3, fljsd 5
    K = args.steps
    ev = {op: [[torch.cuda.Event(enable_timing=True) for _ in range(n)] for _ in range(K)]
          for op, n in (("ce", 2), ("sbv", 2), ("fl", 3), ("js", 5))}

    for per_step in ev.values():       # create every event before the timed region
        for evs in per_step:
            for e in evs:
                e.record(stream)
    torch.cuda.synchronize()

    def nvtx(name, fn):
        # a named NVTX range around each call, for timeline profilers (no cost without one)
        def call():
            torch.cuda.nvtx.range_push(name)
            try:
                fn()
            finally:
                torch.cuda.nvtx.range_pop()
        return call

    op_fns = {
        "ce": nvtx("ce_fwd_f32", lambda: lmho.ce_fwd_f32(d["ce_z"], d["ce_t"], loss=out["ce"], ws=ws_ce)),
        "sbv": nvtx("ce_fwd_sbv_bf16", lambda: lmho.ce_fwd_sbv_bf16(d["sbv_z"], d["sbv_t"], loss=out["sbv"])),
        "fl": nvtx("flce_fwd_bf16",
                   lambda: lmho.flce_fwd_bf16(d["fl_x"], d["fl_w"], d["fl_t"], loss=out["fl"], ws=ws_fl)),
        "js": nvtx("fljsd_fwd_bf16", lambda: lmho.fljsd_fwd_bf16(d["js_xs"], d["js_ws"], d["js_xt"], d["js_wt"], 0.5,
                                                                 loss=out["js"], ws=ws_js)),
    }

    def step(i=None):
        for op in ("ce", "sbv", "fl", "js"):
            if i is not None:
                lmho.set_launch_events(ev[op][i])
            op_fns[op]()
            if i is not None:
                lmho.set_launch_events(None)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for w in (ws_fl, ws_js):
        st = lmho.ws_status(w)
        if st:
            raise RuntimeError(f"device status {st}: {lmho.strerror(st)}")

    def barrier():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x):
        if not dist:
            return x
        from lm_head_online_gb300 import dist as lmdist
        return lmdist.max_over_ranks(x)

    # -------- device-resident timing
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        barrier()
        e0.record(stream)
        for i in range(K):
            step(i)
        e1.record(stream)
        barrier()
    ms_total = e0.elapsed_time(e1)
    ms_step = max_over_ranks(ms_total / K)
    clock_dev = clocks.summary()

    def kern_ms(op, j):
        return float(np.mean([ev[op][i][j].elapsed_time(ev[op][i][j + 1]) for i in range(K)]))

    kern = {
        "ce_fwd_f32.row_kernel_and_mean": ("ce", 0), "ce_fwd_sbv_bf16.row_kernel": ("sbv", 0),
        "flce.tcgen05_gemm_ce": ("fl", 0), "flce.finalize": ("fl", 1),
        "fljsd.tcgen05_gemm_lse": ("js", 0), "fljsd.lse_finalize": ("js", 1),
        "fljsd.tcgen05_gemm_jsd": ("js", 2), "fljsd.jsd_finalize": ("js", 3),
    }
    kms = {k: kern_ms(*v) for k, v in kern.items()}
    call_ms = {op: float(np.mean([ev[op][i][0].elapsed_time(ev[op][i][-1]) for i in range(K)]))
               for op in ev}

    pk = peaks()
    ce_b = rl.ce_flat_bytes(CE["T"], CE["V"])
    sbv_b = rl.ce_sbv_bytes(SBV["S"], SBV["B"], SBV["V"])
    fl_f = rl.flce_flops(FLCE["T"], FLCE["H"], FLCE["V"])
    js_pf = rl.fljsd_pass_flops(FLJSD["T"], FLJSD["H"], FLJSD["V"])
    tf_peak = pk["bf16_sus"]

    def hbm_roof(nbytes, ms, traffic=None):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                "frac": round(gbs / pk["hbm"], 4), "traffic": traffic}

    def tc_roof(flops, ms, traffic=None):
        tfs = flops / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(tfs, 1), "peak": tf_peak, "unit": "TFLOP/s",
                "frac": round(tfs / tf_peak, 4), "traffic": traffic}

    roofs = {
        "ce_fwd_f32.row_kernel_and_mean": hbm_roof(ce_b, kms["ce_fwd_f32.row_kernel_and_mean"],
                                                   traffic_of("ce_fwd_f32.row_kernel_and_mean")),
        "ce_fwd_sbv_bf16.row_kernel": hbm_roof(sbv_b, kms["ce_fwd_sbv_bf16.row_kernel"],
                                               traffic_of("ce_fwd_sbv_bf16.row_kernel")),
        "flce.tcgen05_gemm_ce": tc_roof(fl_f, kms["flce.tcgen05_gemm_ce"], traffic_of("flce.tcgen05_gemm_ce")),
        "fljsd.tcgen05_gemm_lse": tc_roof(js_pf, kms["fljsd.tcgen05_gemm_lse"], traffic_of("fljsd.tcgen05_gemm_lse")),
        "fljsd.tcgen05_gemm_jsd": tc_roof(js_pf, kms["fljsd.tcgen05_gemm_jsd"], traffic_of("fljsd.tcgen05_gemm_jsd")),
    }
    dominant = max(roofs, key=lambda k: kms[k])
    small_ops, small_roofs = {}, {}
    if not args.no_small_ce:
        small_ops, small_roofs, _ = small_ce(lmho, torch, dev, args.seed + rank, pk)
    ops = {
        "ce_fwd_f32": {"us": round(call_ms["ce"] * 1e3, 2), "GB/s": round(ce_b / call_ms["ce"] / 1e6, 1),
                       "bytes": ce_b, "loss": float(out["ce"].item())},
        "ce_fwd_sbv_bf16": {"us": round(call_ms["sbv"] * 1e3, 2), "GB/s": round(sbv_b / call_ms["sbv"] / 1e6, 1),
                            "bytes": sbv_b, "loss_mean": float(out["sbv"].double().mean().item())},
        "flce_fwd_bf16": {"us": round(call_ms["fl"] * 1e3, 2), "TFLOP/s": round(fl_f / call_ms["fl"] / 1e9, 1),
                          "flops": fl_f, "loss": float(out["fl"].item())},
        "fljsd_fwd_bf16": {"us": round(call_ms["js"] * 1e3, 2),
                           "TFLOP/s": round(2 * js_pf / call_ms["js"] / 1e9, 1), "flops": 2 * js_pf,
                           "loss": float(out["js"].item())},
    }

    # -------- end to end through host buffers
    e2e = None
    clock_e2e = None
    if not args.no_e2e:
        host_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out.items()}
        h2d = sum(v.numel() * v.element_size() for v in h.values())
        d2h = sum(v.numel() * v.element_size() for v in out.values())

        # The host link's own rate here: a 1 GiB pinned copy by lmho_copy_h2d (the
        # e2e step's transfer path), median of 3 after one untimed.
        # h2d / link_GBps is the floor of an end-to-end step (the copies alone).
        # The same copy by the copy engines is reported beside it.
        probe_h = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
        probe_d = torch.empty(1 << 30, dtype=torch.uint8, device=dev)

        def link_rate(copy):
            r = []
            for _ in range(4):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                copy()
                b.record(stream)
                b.synchronize()
                r.append((1 << 30) / (a.elapsed_time(b) * 1e-3) / 1e9)
            return float(np.median(r[1:]))

        link_gbps = link_rate(lambda: lmho.copy_h2d(probe_d, probe_h))
        engine_gbps = link_rate(lambda: probe_d.copy_(probe_h, non_blocking=True))
        del probe_h, probe_d

        # Each op's inputs are copied on a second stream, in the order below (most
        # compute per copied byte first; of the two CE calls, whose compute per
        # byte is alike, the shorter last, since its kernel is the step's tail),
        # and each op waits only for its own inputs, so copies of later inputs
        # overlap earlier ops' kernels.  A step's
        # copies start after the previous step's kernels (buffers are reused).
        # The copies are lmho_copy_h2d (SM loads from the pinned buffers): on this
        # machine copy-engine transfers stalled in bursts on host page faults.
        copy_stream = torch.cuda.Stream(device=dev)
        order = (("js", ("js_xs", "js_ws", "js_xt", "js_wt")), ("fl", ("fl_x", "fl_w", "fl_t")),
                 ("ce", ("ce_z", "ce_t")), ("sbv", ("sbv_z", "sbv_t")))
        assert sorted(k for _, ks in order for k in ks) == sorted(h)
        landed = {op: torch.cuda.Event() for op, _ in order}

        def e2e_step(marks=None):
            if marks:
                marks[0].record(stream)
            copy_stream.wait_stream(stream)
            with torch.cuda.stream(copy_stream):
                for op, keys in order:
                    for k in keys:
                        lmho.copy_h2d(d[k], h[k])
                    landed[op].record(copy_stream)
            for op, _ in order:
                stream.wait_event(landed[op])
                op_fns[op]()
            if marks:
                marks[1].record(copy_stream)   # last input landed
                marks[2].record(stream)        # last kernel done
            for k, v in out.items():
                host_out[k].copy_(v, non_blocking=True)
            if marks:
                marks[3].record(stream)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        Ke = max(3, min(K, 10))
        marks = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(Ke)]
        with ClockSampler(local_rank if args.e2e_clocks else -1) as ck:
            barrier()
            e0.record(stream)
            for j in range(Ke):
                e2e_step(marks[j])
            e1.record(stream)
            barrier()
        ms_e2e = max_over_ranks(e0.elapsed_time(e1) / Ke)
        clock_e2e = ck.summary()
        copy_ms = float(np.mean([m[0].elapsed_time(m[1]) for m in marks]))
        kern_ms = float(np.mean([m[0].elapsed_time(m[2]) for m in marks]))
        d2h_ms = float(np.mean([m[2].elapsed_time(m[3]) for m in marks]))
        e2e = {"value": round(ms_e2e * 1e3, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": Ke,
               "overlap": "each op's inputs copied on a second stream by lmho_copy_h2d (SM loads of the pinned "
                          "buffers), ops start as their inputs land",
               "phases_us": {"inputs_landed": round(copy_ms * 1e3, 1), "kernels_done": round(kern_ms * 1e3, 1),
                             "d2h": round(d2h_ms * 1e3, 1)},
               "h2d_GBps": round(h2d / (copy_ms * 1e-3) / 1e9, 1),
               "link_GBps": round(link_gbps, 1),
               "copy_engine_GBps": round(engine_gbps, 1),
               "copy_floor_us": round(h2d / (link_gbps * 1e9) * 1e6, 1),
               # per step: the host link is shared with other GPUs' jobs on the same CPU
               "h2d_GBps_per_step": [round(h2d / (m[0].elapsed_time(m[1]) * 1e-3) / 1e9, 1) for m in marks]}

    result = {
        "metric": METRIC, "value": round(ms_step * 1e3, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 (bf16 tensor-core operands)",
        "data": "synthetic (seeded Philox generator, host-made, pinned)",
        "config": {"workload": WORKLOAD, "l2": "inputs larger than L2 (no flush)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "peaks": pk["src"]},
        "ops": ops,
        "kernels_ms": {k: round(v, 4) for k, v in kms.items()},
        "roofline": dict(roofs[dominant], kernel=dominant),
        "rooflines": roofs,
        "small_ce": {"ops": small_ops, "rooflines": small_roofs,
                     "note": "each configuration alone after the step; not part of value"},
        "e2e": e2e,
        "gpu_launches": KERNELS_PER_STEP * K,
        "clocks": clock_dev,
        "clocks_e2e": clock_e2e,
        "input_gen_s": round(t_gen, 1),
    }
    if world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(h=h, seed=args.seed)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return result


# ---------------------------------------------------------------- vocab-parallel arm
def run_tp(args, rank, world, local_rank):
    """Tensor-parallel Megatron cross-entropy over `world` ranks (one GPU each):
    rank r holds the vocab columns shard_vocab(V, r, world) of bf16 logits
    [S, B, V] ~ N(0, 2^2); a step is the rank's partials kernel, one NCCL
    all-gather of the partials (12 bytes per token per rank) and the merge
    kernel.  Total work is fixed as N grows ("strong").  A one-rank NCCL group
    is used at N = 1, so the collective path runs there too."""
    import torch
    import torch.distributed as tdist
    import gen
    import lm_head_online_gb300 as lmho
    from lm_head_online_gb300 import dist as lmdist

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lmho.load()
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ.setdefault("MASTER_PORT", "29533")
    tdist.init_process_group("nccl", rank=rank, world_size=world, device_id=dev)
    S, B, V = SBV["S"], SBV["B"], SBV["V"]
    v0, w = lmdist.shard_vocab(V, rank, world)
    thr = os.cpu_count() or 1
    full = torch.empty((S, B, V), dtype=torch.bfloat16)
    gen.normal_bf16_bits(args.seed, gen.STREAM_LOGITS, (S, B, V), 2.0, out=full.view(torch.int16), threads=thr)
    local = full[:, :, v0:v0 + w].contiguous().to(dev)
    del full
    t = torch.from_numpy(gen.targets(args.seed, gen.STREAM_TARGET, (S, B), V, threads=thr)).to(dev)
    part = torch.empty((3, S, B), device=dev)
    gathered = torch.empty((world, 3, S, B), device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        lmho.ce_partials_sbv_bf16(local, t, v0, partials=part)
        if ev:
            ev[1].record(stream)
        tdist.all_gather_into_tensor(gathered.view(world * 3, S, B), part)
        if ev:
            ev[2].record(stream)
        loss = lmho.ce_merge_partials(gathered, t, V)
        if ev:
            ev[3].record(stream)
        return loss

    for _ in range(args.warmup):
        loss = step()
    torch.cuda.synchronize()
    single = lmho.ce_fwd_sbv_bf16(local, t) if world == 1 else None
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        tdist.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(K):
            loss = step(evs[i])
        e1.record(stream)
        torch.cuda.synchronize()
        tdist.barrier()
    ms = lmdist.max_over_ranks(e0.elapsed_time(e1) / K)
    ph = {name: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)]))
          for j, name in enumerate(("partials", "all_gather", "merge"))}
    local_bytes = 2 * S * B * w + 8 * S * B + 12 * S * B
    pk = peaks()
    gbs = local_bytes / (ph["partials"] * 1e-3) / 1e9
    res = {"metric": "vocab-parallel Megatron CE us/step (partials + all-gather + merge)", "impl": "ours",
           "mode": "vocab-parallel", "value": round(ms * 1e3, 2), "unit": "us/step", "n_gpus": world, "steps": K,
           "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": False, "scaling": "strong",
           "vs_baseline": None, "dtype": "bf16 in, f32 accumulate", "data": "synthetic (seeded Philox generator)",
           "config": {"workload": f"ce_partials_sbv_bf16 + all-gather + ce_merge_partials, bf16[{S},{B},{V}] "
                                  f"vocab-sharded over {world} rank(s)", "parallelism": f"tp{world}",
                      "l2": "local logits larger than L2 (no flush)" if 2 * S * B * w > L2_BYTES else
                            "local logits smaller than L2 (consecutive steps may hit L2)"},
           "phases_us": {k: round(v * 1e3, 2) for k, v in ph.items()},
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                        "frac": round(gbs / pk["hbm"], 4), "traffic": None, "kernel": "ce_partials_sbv_bf16"},
           "gpu_launches": 2 * K, "clocks": clocks.summary(),
           "loss_mean": float(loss.double().mean().item())}
    if single is not None:
        res["max_abs_diff_vs_ce_fwd_sbv_bf16"] = float((loss - single).abs().max().item())
    tdist.destroy_process_group()
    return res


def run_tp_fused(args, rank, world, local_rank):
    """Vocab-parallel fused losses over `world` ranks (one GPU each): rank r
    holds the rows shard_vocab(V, r, world) of W (of both heads for the JSD);
    the inputs x / xs, xt and the targets are on every rank.  One step:
      flce:  flce_partials_bf16, one NCCL all-gather of [3, T], ce_merge_partials,
             rows_mean; its backward flce_shard_bwd_bf16 (the rank's dx share and
             dW rows) and one all-reduce of dx;
      fljsd: fljsd_lse_partials_bf16, all-gather of [2, T], lse_merge_partials,
             fljsd_terms_bf16 with the KL shares, all-gather of [2, T], jsd_merge_terms
             (terms and KL); the student backward fljsd_shard_bwd_bf16 and one
             all-reduce of dxs.
    Total work is fixed as N grows ("strong").  A one-rank NCCL group is used at
    N = 1 (the collectives run there too), where the unsharded calls are timed
    beside it and their results compared."""
    import torch
    import torch.distributed as tdist
    import gen
    import lm_head_online_gb300 as lmho
    from lm_head_online_gb300 import dist as lmdist

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lmho.load()
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ.setdefault("MASTER_PORT", "29534")
    tdist.init_process_group("nccl", rank=rank, world_size=world, device_id=dev)
    thr = os.cpu_count() or 1
    H, V = FLCE["H"], FLCE["V"]
    Tc, Tj = FLCE["T"], FLJSD["T"]
    v0, w = lmdist.shard_vocab(V, rank, world)

    def rows_of(stream_id, sigma):
        full = torch.empty((V, H), dtype=torch.bfloat16)
        gen.normal_bf16_bits(args.seed, stream_id, (V, H), sigma, out=full.view(torch.int16), threads=thr)
        return full[v0:v0 + w].contiguous().to(dev)

    def host_bf16(stream_id, T):
        t = torch.empty((T, H), dtype=torch.bfloat16)
        gen.normal_bf16_bits(args.seed, stream_id, (T, H), 1.0, out=t.view(torch.int16), threads=thr)
        return t.to(dev)

    x = host_bf16(gen.STREAM_X, Tc)
    W = rows_of(gen.STREAM_W, 0.02)
    tgt = torch.from_numpy(gen.targets(args.seed, gen.STREAM_TARGET, (Tc,), V, threads=thr)).to(dev)
    xs, xt = host_bf16(gen.STREAM_X, Tj), host_bf16(gen.STREAM_XT, Tj)
    Ws, Wt = rows_of(gen.STREAM_W, 0.02), rows_of(gen.STREAM_WT, 0.02)
    ws_c = lmho.workspace(lmho.flce_bwd_workspace_bytes(Tc, H, w), dev)
    dx = torch.empty((Tc, H), device=dev)
    dW = torch.empty((w, H), device=dev)
    ws_j = lmho.workspace(lmho.fljsd_bwd_workspace_bytes(Tj, H, w), dev)
    dxs = torch.empty((Tj, H), device=dev)
    dWs = torch.empty((w, H), device=dev)
    part = torch.empty((3, Tc), device=dev)
    g_part = torch.empty((world, 3, Tc), device=dev)
    lse_l = torch.empty((2, Tj), device=dev)
    g_lse = torch.empty((world, 2, Tj), device=dev)
    tk = torch.empty((2, Tj), device=dev)
    g_tk = torch.empty((world, 2, Tj), device=dev)
    stream = torch.cuda.current_stream()
    names = ("flce_pass", "flce_gather", "flce_merge", "flce_bwd", "dx_allreduce", "lse_pass", "lse_gather",
             "lse_merge", "jsd_pass", "jsd_gather", "jsd_merge", "jsd_bwd", "dxs_allreduce")

    def step(ev=None):
        def mark(i):
            if ev:
                ev[i].record(stream)
        mark(0)
        lmho.flce_partials_bf16(x, W, tgt, v0, partials=part, ws=ws_c)
        mark(1)
        tdist.all_gather_into_tensor(g_part.view(world * 3, Tc), part)
        mark(2)
        rows = lmho.ce_merge_partials(g_part.view(world, 3, Tc, 1), tgt.view(Tc, 1), V).view(Tc)
        ce_mean = lmho.rows_mean(rows)
        mark(3)
        lmho.flce_shard_bwd_bf16(x, W, tgt, g_part, v0, V, 1.0, dx=dx, dW=dW, ws=ws_c)
        mark(4)
        tdist.all_reduce(dx, op=tdist.ReduceOp.SUM)
        mark(5)
        lmho.fljsd_lse_partials_bf16(xs, Ws, xt, Wt, 1.0, out=lse_l, ws=ws_j)
        mark(6)
        tdist.all_gather_into_tensor(g_lse.view(world * 2, Tj), lse_l)
        mark(7)
        lse = lmho.lse_merge_partials(g_lse)
        mark(8)
        lmho.fljsd_terms_bf16(xs, Ws, xt, Wt, lse, 0.5, 1.0, out=tk[0], ws=ws_j, kl_local=tk[1])
        mark(9)
        tdist.all_gather_into_tensor(g_tk.view(world * 2, Tj), tk)
        mark(10)
        jsd, _ = lmho.jsd_merge_terms(g_tk[:, 0].contiguous())
        _, kl = lmho.jsd_merge_terms(g_tk[:, 1].contiguous())
        mark(11)
        lmho.fljsd_shard_bwd_bf16(xs, Ws, xt, Wt, lse, kl, 0.5, 1.0, None, 1.0, dx=dxs, dW=dWs, ws=ws_j)
        mark(12)
        tdist.all_reduce(dxs, op=tdist.ReduceOp.SUM)
        mark(13)
        return ce_mean, jsd

    for _ in range(max(1, args.warmup)):
        ce_mean, jsd = step()
    torch.cuda.synchronize()
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(14)] for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        tdist.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(K):
            ce_mean, jsd = step(evs[i])
        e1.record(stream)
        torch.cuda.synchronize()
        tdist.barrier()
    ms = lmdist.max_over_ranks(e0.elapsed_time(e1) / K)
    ph = {name: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)]))
          for j, name in enumerate(names)}
    pk = peaks()
    fl_flops = 2 * Tc * H * w
    js_flops = 4 * Tj * H * w
    tf = js_flops / (ph["jsd_pass"] * 1e-3) / 1e12
    bwd_flops = 2 * fl_flops + fl_flops   # dZ recompute pass, dx and dW products
    jbwd_flops = 2 * js_flops   # both heads' dZ recompute (js_flops), then the dx and dW products (js_flops / 2 each)
    res = {"metric": "vocab-parallel fused linear + CE and + JSD, forward and backward, us/step", "impl": "ours",
           "mode": "vocab-parallel fused", "value": round(ms * 1e3, 1), "unit": "us/step", "n_gpus": world,
           "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": False,
           "scaling": "strong", "vs_baseline": None, "dtype": "bf16 in, f32 accumulate",
           "data": "synthetic (seeded Philox generator)",
           "config": {"workload": f"flce x[{Tc},{H}] + fljsd xs,xt[{Tj},{H}], W rows [{V},{H}] sharded over "
                                  f"{world} rank(s) ({w} rows here)", "parallelism": f"tp{world}",
                      "l2": "inputs larger than L2 (no flush)"},
           "phases_us": {k: round(v * 1e3, 1) for k, v in ph.items()},
           "TFLOP/s": {"flce_pass": round(fl_flops / (ph["flce_pass"] * 1e-3) / 1e12, 1),
                       "flce_bwd": round(bwd_flops / (ph["flce_bwd"] * 1e-3) / 1e12, 1),
                       "lse_pass": round(js_flops / (ph["lse_pass"] * 1e-3) / 1e12, 1),
                       "jsd_pass": round(tf, 1),
                       "jsd_bwd": round(jbwd_flops / (ph["jsd_bwd"] * 1e-3) / 1e12, 1)},
           "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": pk["bf16_sus"],
                        "unit": "TFLOP/s", "frac": round(tf / pk["bf16_sus"], 4), "traffic": None,
                        "kernel": "fljsd_terms_bf16 tensor-core pass"},
           "gpu_launches": 21 * K, "clocks": clocks.summary(),
           "flce_loss": float(ce_mean.item()), "fljsd_loss": float(jsd.item())}
    if world == 1:
        # the unsharded calls on the same inputs, timed the same way
        ws1 = lmho.workspace(lmho.flce_bwd_workspace_bytes(Tc, H, V), dev)
        ws2 = lmho.workspace(lmho.fljsd_bwd_workspace_bytes(Tj, H, V), dev)
        dx1, dW1 = torch.empty_like(dx), torch.empty_like(dW)
        dxs1, dWs1 = torch.empty_like(dxs), torch.empty_like(dWs)
        for _ in range(2):
            a = lmho.flce_fwd_bwd_bf16(x, W, tgt, 1.0, dx=dx1, dW=dW1, ws=ws1)[0]
            b = lmho.fljsd_fwd_bwd_bf16(xs, Ws, xt, Wt, 0.5, 1.0, None, 1.0, dxs=dxs1, dWs=dWs1, ws=ws2)[0]
        torch.cuda.synchronize()
        u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        u0.record(stream)
        for _ in range(K):
            a = lmho.flce_fwd_bwd_bf16(x, W, tgt, 1.0, dx=dx1, dW=dW1, ws=ws1)[0]
            b = lmho.fljsd_fwd_bwd_bf16(xs, Ws, xt, Wt, 0.5, 1.0, None, 1.0, dxs=dxs1, dWs=dWs1, ws=ws2)[0]
        u1.record(stream)
        torch.cuda.synchronize()
        res["unsharded_us_per_step"] = round(u0.elapsed_time(u1) / K * 1e3, 1)
        res["bitwise_equal_to_unsharded"] = bool(torch.equal(a, ce_mean) and torch.equal(b, jsd) and
                                                 torch.equal(dx1, dx) and torch.equal(dW1, dW) and
                                                 torch.equal(dxs1, dxs) and torch.equal(dWs1, dWs))
    tdist.destroy_process_group()
    return res


# ---------------------------------------------------------------- oracle (CPU) arm
def oracle_samples(seed=0, h=None, budget_s=ORACLE_BUDGET_S):
    """Bounded samples of every op's inputs (taken from the bench's own host
    tensors when given, else regenerated by counter offset)."""
    import gen
    cores = os.cpu_count() or 1
    f = budget_s / 12.0
    # sized for ~10 s of host time at budget_s = 12 on 16 cores (CE rows cost
    # ~1.5 ms each per thread, fused tokens ~0.3 s (CE) / 0.6 s (JSD) per thread)
    n_ce = min(CE["T"], max(cores, int(16384 * f)))
    n_sbv = min(SBV["S"] * SBV["B"], max(cores, int(8192 * f)))
    n_fl = max(1, int(8 * cores * f))
    n_js = max(1, int(3 * cores * f))

    def np_bits(t):
        import torch
        return t.view(torch.int16).numpy().view(np.uint16)

    s = {"n": dict(ce=n_ce, sbv=n_sbv, fl=n_fl, js=n_js), "cores": cores}
    if h is not None:
        s["ce"] = (h["ce_z"][:n_ce].numpy(), h["ce_t"][:n_ce].numpy())
        s["sbv"] = (np_bits(h["sbv_z"]).reshape(-1, 1, SBV["V"])[:n_sbv], h["sbv_t"].numpy().reshape(-1, 1)[:n_sbv])
        s["fl"] = (np_bits(h["fl_x"])[:n_fl], np_bits(h["fl_w"]), h["fl_t"][:n_fl].numpy())
        s["js"] = (np_bits(h["js_xs"])[:n_js], np_bits(h["js_ws"]), np_bits(h["js_xt"])[:n_js], np_bits(h["js_wt"]))
        return s
    H, V = FLCE["H"], FLCE["V"]
    s["ce"] = (gen.normal_f32(seed, gen.STREAM_LOGITS, (n_ce, CE["V"])),
               gen.targets(seed, gen.STREAM_TARGET, (n_ce,), CE["V"]))
    s["sbv"] = (gen.normal_bf16_bits(seed, gen.STREAM_LOGITS, (n_sbv, 1, SBV["V"]), 2.0),
                gen.targets(seed, gen.STREAM_TARGET, (n_sbv, 1), SBV["V"]))
    W = gen.normal_bf16_bits(seed, gen.STREAM_W, (V, H), 0.02)
    s["fl"] = (gen.normal_bf16_bits(seed, gen.STREAM_X, (n_fl, H)), W,
               gen.targets(seed, gen.STREAM_TARGET, (n_fl,), V))
    s["js"] = (gen.normal_bf16_bits(seed, gen.STREAM_X, (n_js, H)), W,
               gen.normal_bf16_bits(seed, gen.STREAM_XT, (n_js, H)),
               gen.normal_bf16_bits(seed, gen.STREAM_WT, (V, H), 0.02))
    return s


def time_oracle(s, single_thread=False):
    """The oracle as it stands on the samples; CE rows are split over host
    threads (each oracle call releases the GIL), fused tokens use the
    oracle's own token partition.  Returns the extrapolated us per full step."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    cores, n = s["cores"], s["n"]

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    def rows_parallel(fn, z, t):
        parts = np.array_split(np.arange(len(z)), cores)
        with ThreadPoolExecutor(cores) as ex:
            list(ex.map(lambda idx: fn(z[idx[0]:idx[-1] + 1], t[idx[0]:idx[-1] + 1]) if len(idx) else None, parts))

    t_ce = timed(lambda: rows_parallel(oracle.ce_f32, *s["ce"]))
    t_sbv = timed(lambda: rows_parallel(oracle.ce_sbv_bf16, *s["sbv"]))
    t_fl = timed(lambda: oracle.flce_bf16(*s["fl"], threads=cores))
    t_js = timed(lambda: oracle.fljsd_bf16(*s["js"], 0.5, threads=cores))
    us = 1e6 * (t_ce * CE["T"] / n["ce"] + t_sbv * SBV["S"] * SBV["B"] / n["sbv"] +
                t_fl * FLCE["T"] / n["fl"] + t_js * FLJSD["T"] / n["js"])
    out = {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": (f"ce {n['ce']}/{CE['T']} rows, sbv {n['sbv']}/{SBV['S'] * SBV['B']} tokens, "
                      f"flce {n['fl']}/{FLCE['T']} tokens, fljsd {n['js']}/{FLJSD['T']} tokens of the same "
                      f"workload on {cores} threads; scaled linearly to one full step"),
           "seconds": {"ce": round(t_ce, 2), "sbv": round(t_sbv, 2), "flce": round(t_fl, 2),
                       "fljsd": round(t_js, 2)}}
    if single_thread:
        # one thread on a fixed small subset of the same sample (16 CE rows of each
        # layout, 2 flce tokens, 1 fljsd token), extrapolated to one step
        k_ce, k_sbv = min(16, n["ce"]), min(16, n["sbv"])
        t1_ce = timed(lambda: oracle.ce_f32(s["ce"][0][:k_ce], s["ce"][1][:k_ce]))
        t1_sbv = timed(lambda: oracle.ce_sbv_bf16(s["sbv"][0][:k_sbv], s["sbv"][1][:k_sbv]))
        x, W, t = s["fl"]
        t1_fl = timed(lambda: oracle.flce_bf16(x[:2], W, t[:2], threads=1))
        xs, Ws, xt, Wt = s["js"]
        t1_js = timed(lambda: oracle.fljsd_bf16(xs[:1], Ws, xt[:1], Wt, 0.5, threads=1))
        us1 = 1e6 * (t1_ce * CE["T"] / k_ce + t1_sbv * SBV["S"] * SBV["B"] / k_sbv +
                     t1_fl * FLCE["T"] / 2 + t1_js * FLJSD["T"])
        out["single_thread"] = {"value": round(us1, 1), "unit": UNIT, "cores": 1, "extrapolated": True,
                                "sample": f"ce {k_ce} rows, sbv {k_sbv} tokens, flce 2 tokens, fljsd 1 token "
                                          f"on one thread, scaled linearly to one full step"}
    return out


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(h=None, budget_s=ORACLE_BUDGET_S, seed=0):
    r = time_oracle(oracle_samples(seed, h, budget_s), single_thread=True)
    r["cpu_model"] = cpu_model()
    return r


def run_reference(args):
    import oracle
    oracle.build()
    s = oracle_samples(args.seed, None, budget_s=ORACLE_BUDGET_S)
    vals, r = [], None
    for i in range(args.warmup + args.steps):
        r = time_oracle(s)
        if i >= args.warmup:
            vals.append(r["value"])
    v = float(np.median(vals))
    return {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Philox generator)",
            "config": {"workload": WORKLOAD, "l2": "n/a (host)", "parallelism": "host threads"},
            "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                             "sample": r["sample"], "cpu_model": cpu_model()},
            "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_case(args):
    """One op alone, `warmup` untimed + `steps` timed calls (CUDA events on
    the launching stream).  Used for ncu captures on small cases."""
    import torch
    import gen
    import lm_head_online_gb300 as lmho
    torch.cuda.set_device(0)
    lmho.load()
    lmho.set_ce_variant(args.ce_variant)
    lmho.set_raster_group(args.raster_group)
    thr = os.cpu_count() or 1

    def bf16(seed, stream, shape, sigma):
        t = torch.empty(shape, dtype=torch.bfloat16)
        gen.normal_bf16_bits(seed, stream, shape, sigma, out=t.view(torch.int16), threads=thr)
        return t.cuda()

    def targets(shape, V):
        return torch.from_numpy(gen.targets(args.seed, gen.STREAM_TARGET, shape, V, threads=thr)).cuda()

    c, H = args.case, args.H
    if c == "ce":
        T, V = args.T or CE["T"], args.V or CE["V"]
        z = torch.from_numpy(gen.normal_f32(args.seed, 0, (T, V), threads=thr)).cuda()
        t = targets((T,), V)
        ws = lmho.workspace(lmho.ce_workspace_bytes(T, V))
        fn = lambda: lmho.ce_fwd_f32(z, t, ws=ws)  # noqa: E731
        work, unit = rl.ce_flat_bytes(T, V), "GB/s"
    elif c == "sbv":
        S, V = args.T or SBV["S"], args.V or SBV["V"]
        z = bf16(args.seed, 0, (S, 4, V), 2.0)
        t = targets((S, 4), V)
        fn = lambda: lmho.ce_fwd_sbv_bf16(z, t)  # noqa: E731
        work, unit = rl.ce_sbv_bytes(S, 4, V), "GB/s"
    elif c == "ce_fb":
        T, V = args.T or CE["T"], args.V or CE["V"]
        z = torch.from_numpy(gen.normal_f32(args.seed, 0, (T, V), threads=thr)).cuda()
        t = targets((T,), V)
        ws = lmho.workspace(lmho.ce_workspace_bytes(T, V))
        dz = torch.empty_like(z)
        fn = lambda: lmho.ce_fwd_bwd_f32(z, t, 1.0, ws=ws, dlogits=dz)  # noqa: E731
        work, unit = rl.ce_flat_fwd_bwd_bytes(T, V), "GB/s"
    elif c == "sbv_fb":
        S, V = args.T or SBV["S"], args.V or SBV["V"]
        z = bf16(args.seed, 0, (S, 4, V), 2.0)
        t = targets((S, 4), V)
        dz = torch.empty_like(z)
        fn = lambda: lmho.ce_fwd_bwd_sbv_bf16(z, t, dlogits=dz)  # noqa: E731
        work, unit = rl.ce_sbv_fwd_bwd_bytes(S, 4, V), "GB/s"
    elif c == "cublas":
        # practical ceiling of the fused configs: a library bf16 GEMM of the same
        # shape, logits = x W^T written to memory (run only, timed like the rest)
        T, V = args.T or FLCE["T"], args.V or FLCE["V"]
        x, W = bf16(args.seed, 0, (T, H), 1.0), bf16(args.seed, 2, (V, H), 0.02)
        logits = torch.empty((T, V), dtype=torch.bfloat16, device="cuda")
        fn = lambda: torch.matmul(x, W.t(), out=logits)  # noqa: E731
        work, unit = rl.flce_flops(T, H, V), "TFLOP/s"
    elif c == "flce":
        T, V = args.T or FLCE["T"], args.V or FLCE["V"]
        x, W, t = bf16(args.seed, 0, (T, H), 1.0), bf16(args.seed, 2, (V, H), 0.02), targets((T,), V)
        ws = lmho.workspace(lmho.flce_workspace_bytes(T, H, V))
        fn = lambda: lmho.flce_fwd_bf16(x, W, t, ws=ws)  # noqa: E731
        work, unit = rl.flce_flops(T, H, V), "TFLOP/s"
    elif c in ("cpo", "cpo_fb"):
        # the CPO page's workload: seq 1024 x batch, chosen = first half of the batch
        T, V = args.T or FLCE["T"], args.V or FLCE["V"]
        Bq = max(2, T // 1024 // 2 * 2)
        S = T // Bq
        T = Bq * S
        x, W, t = bf16(args.seed, 0, (Bq, S, H), 1.0), bf16(args.seed, 2, (V, H), 0.02), targets((Bq, S), V)
        if c == "cpo":
            ws = lmho.workspace(lmho.flce_cpo_workspace_bytes(Bq, S, H, V))
            fn = lambda: lmho.flce_cpo_fwd_bf16(x, W, t, 0.1, 1.0, ws=ws)  # noqa: E731
            work = rl.flce_flops(T, H, V)
        else:
            ws = lmho.workspace(lmho.flce_cpo_bwd_workspace_bytes(Bq, S, H, V))
            dx = torch.empty((Bq, S, H), dtype=torch.float32, device="cuda")
            dW = torch.empty((V, H), dtype=torch.float32, device="cuda")
            fn = lambda: lmho.flce_cpo_fwd_bwd_bf16(x, W, t, 0.1, 1.0, ws=ws, dx=dx, dW=dW)  # noqa: E731
            work = rl.flce_fwd_bwd_flops(T, H, V)
        unit = "TFLOP/s"
    elif c == "flce_fb":
        T, V = args.T or FLCE["T"], args.V or FLCE["V"]
        x, W, t = bf16(args.seed, 0, (T, H), 1.0), bf16(args.seed, 2, (V, H), 0.02), targets((T,), V)
        ws = lmho.workspace(lmho.flce_bwd_workspace_bytes(T, H, V))
        dx = torch.empty((T, H), dtype=torch.float32, device="cuda")
        dW = torch.empty((V, H), dtype=torch.float32, device="cuda")
        fn = lambda: lmho.flce_fwd_bwd_bf16(x, W, t, 1.0, ws=ws, dx=dx, dW=dW)  # noqa: E731
        work, unit = rl.flce_fwd_bwd_flops(T, H, V), "TFLOP/s"
    elif c == "fljsd_fb":
        T, V = args.T or FLJSD["T"], args.V or FLJSD["V"]
        xs, Ws = bf16(args.seed, 0, (T, H), 1.0), bf16(args.seed, 2, (V, H), 0.02)
        xt, Wt = bf16(args.seed, 3, (T, H), 1.0), bf16(args.seed, 4, (V, H), 0.02)
        ws = lmho.workspace(lmho.fljsd_bwd_workspace_bytes(T, H, V))
        dxs = torch.empty((T, H), dtype=torch.float32, device="cuda")
        dWs = torch.empty((V, H), dtype=torch.float32, device="cuda")
        fn = lambda: lmho.fljsd_fwd_bwd_bf16(xs, Ws, xt, Wt, 0.5, ws=ws, dxs=dxs, dWs=dWs)  # noqa: E731
        work, unit = rl.fljsd_fwd_bwd_flops(T, H, V), "TFLOP/s"
    else:
        T, V = args.T or FLJSD["T"], args.V or FLJSD["V"]
        xs, Ws = bf16(args.seed, 0, (T, H), 1.0), bf16(args.seed, 2, (V, H), 0.02)
        xt, Wt = bf16(args.seed, 3, (T, H), 1.0), bf16(args.seed, 4, (V, H), 0.02)
        ws = lmho.workspace(lmho.fljsd_workspace_bytes(T, H, V))
        fn = lambda: lmho.fljsd_fwd_bf16(xs, Ws, xt, Wt, 0.5, ws=ws)  # noqa: E731
        work, unit = rl.fljsd_flops(T, H, V), "TFLOP/s"
    b2b = None
    if c in ("ce", "sbv"):
        # the same call back to back over rotating copies of the logits (> 3x L2)
        if c == "ce":
            fns = [lambda zz=zz: lmho.ce_fwd_f32(zz, t, ws=ws) for zz in rotating_copies(z, torch)]
        else:
            fns = [lambda zz=zz: lmho.ce_fwd_sbv_bf16(zz, t) for zz in rotating_copies(z, torch)]
        b2b = time_back_to_back(fns, torch, max(args.warmup, 3), max(args.steps, 20))
        del fns
        torch.cuda.empty_cache()
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    # L2 is flushed before every timed call, outside the events, by READING a
    # 512 MB buffer: small cases would otherwise find their inputs in the
    # 129 MB L2, and a write-based flush would leave ~129 MB of dirty lines
    # whose write-back the timed kernel would pay for.
    flush = torch.ones(128 << 20, dtype=torch.float32, device="cuda")
    nk = {"ce": 1, "sbv": 1, "flce": 2, "fljsd": 4, "ce_fb": 1, "sbv_fb": 1, "flce_fb": 4, "fljsd_fb": 4, "cpo": 2,
          "cpo_fb": 4, "cublas": 1}[c]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    for row in evs:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.sum()
        # events recorded by the library itself around its own launches: no
        # host-side gap between the start event and the first kernel
        if c == "cublas":      # not a library call: bracket it here
            evs[i][0].record()
            fn()
            evs[i][1].record()
            continue
        lmho.set_launch_events(evs[i])
        fn()
        lmho.set_launch_events(None)
    torch.cuda.synchronize()
    ms = [evs[i][0].elapsed_time(evs[i][-1]) for i in range(args.steps)]
    kernel_ms = [[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(nk)] for i in range(args.steps)]
    med = float(np.median(ms))
    rate = work / (med * 1e-3) / (1e9 if unit == "GB/s" else 1e12)
    extra = {}
    if b2b is not None:
        extra = {"us_back_to_back": round(b2b, 2), "GB/s_back_to_back": round(work / (b2b * 1e-6) / 1e9, 1)}
    return {**extra, "case": c, "T": args.T, "V": args.V, "H": H, "ce_variant": args.ce_variant, "raster_group": args.raster_group, "l2": "flushed (512 MB read) before each call",
            "us_median": round(med * 1e3, 2),
            "us_p10": round(float(np.percentile(ms, 10)) * 1e3, 2),
            "us_p90": round(float(np.percentile(ms, 90)) * 1e3, 2),
            "us_all": [round(m * 1e3, 2) for m in ms],
            "kernels_us_median": [round(float(np.median([k[j] for k in kernel_ms])) * 1e3, 2) for j in range(nk)],
            unit: round(rate, 1)}


SWEEP = ([("ce", 16384, V) for V in (4096, 8192, 16384, 32768, 65536, 131072)] +
         [("ce_fb", 16384, V) for V in (4096, 8192, 16384, 32768, 65536, 131072)] +
         [("sbv_fb", 2048, V) for V in (4096, 8192, 16384, 32768, 65536, 131072)] +
         [("sbv", 2048, V) for V in (4096, 8192, 16384, 32768, 65536, 131072)] +
         [("flce", 1024 * b, 128256) for b in (2, 4, 8, 16)] +
         [("flce_fb", 1024 * b, 128256) for b in (2, 16)] +
         [("cpo", 1024 * b, 128256) for b in (2, 4, 8, 16)] +
         [("cpo_fb", 1024 * b, 128256) for b in (2, 16)] +
         [("fljsd_fb", T, 128256) for T in (1024, 8192)] +
         [("fljsd", T, 128256) for T in (1024, 2048, 4096, 8192)] +
         [("cublas", 1024 * b, 128256) for b in (2, 16)])


def run_sweep(args):
    """Every configuration of the workload table, one op alone each time
    (L2 flushed by a read before each call), in this process."""
    import torch
    pk = peaks()
    for case, T, V in SWEEP:
        a = argparse.Namespace(**vars(args))
        a.case, a.T, a.V = case, T, V
        # 5 warm-ups; 50 timed calls for the microsecond CE calls, 20 for the fused ones
        a.steps = 50 if case in ("ce", "sbv", "ce_fb", "sbv_fb") else 20
        a.warmup = 5
        r = run_case(a)
        if "GB/s" in r:
            r["frac_of_measured_hbm"] = round(r["GB/s"] / pk["hbm"], 4)
        else:
            r["frac_of_measured_bf16_sustained"] = round(r["TFLOP/s"] / pk["bf16_sus"], 4)
        r["peaks"] = pk["src"]
        print(json.dumps(r), flush=True)
        torch.cuda.empty_cache()


def main():
    args = parse()
    if args.sweep:
        run_sweep(args)
        return
    if args.case:
        print(json.dumps(run_case(args)), flush=True)
        return
    if args.small_ce_only:
        print(json.dumps(run_small_ce_only(args)), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.tp_fused:
        res = run_tp_fused(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    if args.tp:
        res = run_tp(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
