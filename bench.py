"""Benchmark of the causal short convolution hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the whole hot path over one batch of synthetic input:
  * cconv_fwd  on the production-length workload  B=2 T=8192 D=4096 W=4, no bias,
    bf16 activations, fp32 weights;
  * cconv_bwd  (dx, dw and dbias; stream kernel + deterministic reduction) on the same
    workload, dw / dbias reduced over its 16384 rows;
  * cconv_update, one decode step of the decode workload: pool [512, 4096, 3] bf16,
    256 active rows, W=4, bias.
The reported value is achieved HBM throughput, algorithmic bytes over device time, in
TB/s (fwd: 4 B/element, bwd: 6 B/element, decode: x + state read/write + y per step);
per-part TB/s, fractions of the measured copy peak and decode microseconds per step are
reported beside it.  Inputs are rotated so that no kernel reads data the previous kernel
touched, and every per-launch working set (>= 268 MB) is larger than the 129 MB L2.

Timing: the K steps of the timed region are captured once in a CUDA graph (every kernel of
every step is in it) and replayed between two CUDA events on the launching stream (max over
ranks), so the host's argument checks and ctypes marshalling stay outside the timed region;
the same K steps as eager calls are timed too and reported beside the value.  Each part's
device time per call comes from calls of
that entry point captured in one CUDA graph and replayed between two events, so host-side
time (argument checks, ctypes) cannot leak into it; the eager per-call time is reported
beside it.  The decode update is also timed as 1000 updates replayed from one CUDA graph.
Each part lists the kernels it launches with their registers per thread, local (spill)
bytes, shared memory and resident CTAs per SM (the library's launch descriptions).

Under torchrun (N > 1) every rank runs the same step on its own data (weak scaling, no
collective on the data path); the timed region is bracketed by a barrier and
synchronisation, the max over ranks is taken, and rank 0 prints the JSON line.

``--impl reference`` times the fp64 CPU oracle (the only reference this path has) on the
host cores, on a bounded sample of the same workload per step, and prints the same line
with "impl": "reference".
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

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

from depthwise_causal_short_gb300 import inputs  # noqa: E402

METRIC = "achieved HBM TB/s (fwd, bwd) and % of GB300 peak; decode update µs/step"
UNIT = "TB/s"
FALLBACK_HBM_GBS = 6800.0

FWD = inputs.PROD
DEC = inputs.DECODE_SHAPE
N_ELEM = FWD.B * FWD.T * FWD.D
FWD_BYTES = 4 * N_ELEM                       # x read + y written, bf16
BWD_BYTES = 6 * N_ELEM                       # x, dy read + dx written, bf16
DEC_BYTES = (2 * DEC.N * DEC.D                # x read
             + 2 * 2 * DEC.N * DEC.D * (DEC.W - 1)  # named state rows read + written
             + 2 * DEC.N * DEC.D)             # y written
STEP_BYTES = FWD_BYTES + BWD_BYTES + DEC_BYTES
# Packed sequences at the production row count: 16 mixed lengths, initial states in, final
# states out (forward), initial-state gradient out (backward).
VL_NSEQ = 16
VL_STATE_BYTES = 2 * VL_NSEQ * FWD.D * (FWD.W - 1)
VL_FWD_BYTES = FWD_BYTES + 2 * VL_STATE_BYTES    # + initial states read, final written
VL_BWD_BYTES = BWD_BYTES + 2 * VL_STATE_BYTES    # + initial states read, gradient written
LAUNCHES_PER_STEP = 4                        # fwd, bwd stream, bwd reduce, update

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant call (the
# backward: stream kernel + reduction), averaged over back-to-back launches in one ncu
# capture (profiles/, file named below), together with the hash of the kernel sources it
# was taken on.  `traffic` is reported only while the sources still hash the same.
BWD_TRAFFIC = {"bytes_per_call": 408_681_728, "sources_sha16": "1c5b4950e9e17415",
               "profile": "profiles/cconv_bwd_traffic_b2_t8192_d4096.md"}
TRAFFIC_SOURCES = ("csrc/bwd.cu", "csrc/strip.cuh", "csrc/common.cuh")

# Achieved occupancy (sm__warps_active.avg.pct_of_peak_sustained_active: active warps as a
# share of the SM's warp slots) of each stream and decode kernel, from the section captures
# summarised under profiles/.  Reported beside each kernel's live launch description while
# the sources of that kernel's family hash to the value recorded for the family.
OCCUPANCY_SOURCES = {
    "fwd": ("csrc/fwd.cu", "csrc/strip.cuh", "csrc/common.cuh"),
    "bwd": ("csrc/bwd.cu", "csrc/strip.cuh", "csrc/common.cuh"),
    "update": ("csrc/update.cu", "csrc/common.cuh"),
}
ACHIEVED_OCCUPANCY = {
    "sources_sha16": {"fwd": "7418f927c2fcbdd4", "bwd": "1c5b4950e9e17415", "update": "ec15eacc1c4b0ba6"},
    "pct": {
        "cconv_fwd_kernel<4, 8, 10, 8, 1, true, 0>": 14.21,
        "cconv_bwd_ls_kernel<4, 12, 4, 8, 1, 0>": 13.92,
        "cconv_update_kernel<8, 4, 3, 4, 0, 256>": 11.55,
        "cconv_fwd_kernel<4, 8, 10, 8, 1, true, 1>": 13.77,
        "cconv_bwd_ls_kernel<4, 12, 4, 8, 1, 1>": 13.72,
        "cconv_fwd_multi_kernel<4, 8, 10, 8, 1, true>": 14.00,
        "cconv_bwd_ls_multi_kernel<4, 12, 4, 8>": 14.00,
    },
    "profiles": ["profiles/cconv_fwd_bwd_update_kernels_b2_t8192_d4096.md",
                 "profiles/cconv_varlen_multi_bwd_kernels_b2_t8192_d4096.md"],
}

WORKLOAD = ("fwd+bwd B=2 T=8192 D=4096 W=4 no bias (bf16 x/dy, f32 w) + 1 decode update "
            "S=512 N=256 D=4096 W=4 bias per step")


def sources_sha16(files=TRAFFIC_SOURCES) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(HERE, "depthwise_causal_short_gb300", rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_family(kernel: str):
    """fwd, bwd or update: the source family a kernel name belongs to (None if unknown)."""
    for fam in ("fwd", "bwd", "update"):
        if kernel.startswith(f"cconv_{fam}_"):
            return fam
    return None


def achieved_occupancy(kernel: str):
    """Achieved occupancy (%) of a kernel from the profiles, or None if its family's sources
    changed since they were captured (or the kernel was not captured)."""
    fam = kernel_family(kernel)
    if fam is None or kernel not in ACHIEVED_OCCUPANCY["pct"]:
        return None
    if ACHIEVED_OCCUPANCY["sources_sha16"][fam] != sources_sha16(OCCUPANCY_SOURCES[fam]):
        return None
    return ACHIEVED_OCCUPANCY["pct"][kernel]


def bwd_traffic():
    """Measured DRAM bytes per backward call, or None if the kernels changed since."""
    if BWD_TRAFFIC["bytes_per_call"] is None or BWD_TRAFFIC["sources_sha16"] != sources_sha16():
        return None
    return BWD_TRAFFIC["bytes_per_call"]


def measured_peak():
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (identity on one rank)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(per_rank_units: float, elapsed_max_s: float, world: int) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return per_rank_units * world / elapsed_max_s


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: str):
        self.dev = device
        self.lines: list[str] = []
        self.proc = None
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sm, smax, names = [], [], set()
        labels = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for lab, val in zip(labels, parts[5:9]):
                if val.lower().startswith("active"):
                    names.add(lab)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no parsable samples"],
                    "samples": 0}
        loaded = [v for v in sm if v > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(names), "samples": len(sm)}


def gpu_id(dev) -> str:
    """nvidia-smi's name for a torch device (its UUID), independent of CUDA_VISIBLE_DEVICES."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------

def short_name(name: str) -> str:
    """cconv_bwd_ls_kernel<4, 12, 4, 8, 1, 0> from the demangled signature."""
    n = name.split("(")[0]
    n = n.replace("void ", "").replace("cconv::", "")
    return n.strip()


def kernels_of(cc, fn, max_threads_per_sm: int):
    """The kernels fn() launches, with their resources (launch descriptions, nothing runs)."""
    out = []
    for d in cc.describe(fn):
        out.append({
            "kernel": short_name(d["name"]),
            "registers": d["registers"],
            "local_bytes_per_thread": d["local_bytes"],
            "smem_bytes": d["static_shared_bytes"] + d["dynamic_shared_bytes"],
            "threads": d["threads"],
            "ctas": d["ctas"],
            "ctas_per_sm": d["ctas_per_sm"],
            "theoretical_occupancy": round(d["ctas_per_sm"] * d["threads"] / max_threads_per_sm, 4),
            "achieved_occupancy_pct_profiled": achieved_occupancy(short_name(d["name"])),
        })
    return out


def run_ours(args, world, rank, local):
    import depthwise_causal_short_gb300 as cc
    from depthwise_causal_short_gb300 import _build

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or not _build.up_to_date():
        _build.build()
    barrier(world)
    cc.load()
    props = torch.cuda.get_device_properties(dev)
    max_thr = props.max_threads_per_multi_processor

    # ---- inputs (seeded, synthetic), resident in HBM before the timed region ----------
    x, dy, w, _ = inputs.fwd_bwd_inputs(FWD.B, FWD.T, FWD.D, FWD.W, FWD.bias, seed=rank)
    NSET = 2
    xf = [x.to(dev) for _ in range(NSET)]            # forward inputs
    xb = [x.to(dev) for _ in range(NSET)]            # backward inputs (distinct buffers)
    dyb = [dy.to(dev) for _ in range(NSET)]
    ys = [torch.empty_like(xf[0]) for _ in range(NSET)]
    dxs = [torch.empty_like(xf[0]) for _ in range(NSET)]
    wg = w.to(dev)
    dw = torch.empty_like(wg)
    db = torch.empty(FWD.D, dtype=wg.dtype, device=dev)
    ws = torch.empty(cc.cconv_bwd_workspace_bytes(FWD.B, FWD.T, FWD.D, FWD.W), dtype=torch.uint8,
                     device=dev)
    st, xr, idx, wd, bd = inputs.decode_inputs(DEC.S, DEC.N, DEC.D, DEC.W, DEC.bias, n_x=8,
                                               seed=rank)
    st, xr, idx, wd, bd = (t.to(dev) for t in (st, xr, idx, wd, bd))
    yd = torch.empty(DEC.N, DEC.D, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(2, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    # Every part runs on the current stream (the launching stream, or the capture stream).
    def fwd(i):
        k = i % NSET
        cc.cconv_fwd(xf[k], wg, None, y=ys[k])

    def bwd(i):
        k = i % NSET
        cc.cconv_bwd(xb[k], dyb[k], wg, None, want_dbias=True, dx=dxs[k], dw=dw, dbias=db,
                     workspace=ws)

    def upd(i):
        cc.cconv_update(xr[i % xr.shape[0]], st, wd, bd, idx, y=yd, status=status)

    def step(i):
        fwd(i)
        bwd(i)
        upd(i)

    def loop_us(fn, n):
        """Average time per call of fn over n back-to-back eager calls (CUDA events on the
        stream; includes whatever host time the calls take beyond the device's)."""
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / n

    def graph_us(fn, n):
        """Device time per call of fn: min(n, 50) calls captured in one CUDA graph, the
        graph replayed until about n calls have run, between two CUDA events."""
        per = max(2, min(n, 50))
        reps = max(1, n // per)
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn(0)
            with torch.cuda.graph(g, stream=side):
                for i in range(per):
                    fn(i)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * per)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # ---- the K steps, captured once in a CUDA graph (every kernel of every step runs on each
    # replay; the host's argument checks and marshalling stay outside the timed region) ------
    K = args.steps
    G = min(K, 512)  # steps per graph; 512 keeps the rotation of 2 input sets and 8 tokens
    side = torch.cuda.Stream(device=dev)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    step(i)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g.replay()  # one untimed replay: the graph's first launch uploads it
        torch.cuda.synchronize()
        return g

    graphs = [capture(G)] * (K // G) + ([capture(K % G)] if K % G else [])

    # ---- timed region: exactly K steps --------------------------------------------------
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_id(dev)) as clk:
        t0 = time.perf_counter()
        start.record(stream)
        for g in graphs:  # exactly K steps
            g.replay()
        end.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier(world)
    elapsed = start.elapsed_time(end) / 1e3
    elapsed_max = max_over_ranks(elapsed, world, dev)
    assert status.tolist() == [0, 0]
    del graphs

    # ---- the same K steps as eager calls (reported beside the value) -----------------------
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for i in range(K):
        step(i)
    eb.record(stream)
    torch.cuda.synchronize()
    eager_step_ms = max_over_ranks(ea.elapsed_time(eb) / K, world, dev)

    # ---- per-part device time (graph replay) and eager time per call ---------------------
    for fn in (fwd, bwd):
        for i in range(3):
            fn(i)
    f_us, b_us, u_us = graph_us(fwd, K), graph_us(bwd, K), graph_us(upd, K)
    f_eager, b_eager, u_eager = loop_us(fwd, K), loop_us(bwd, K), loop_us(upd, K)

    # ---- decode: 1000 steps replayed from one CUDA graph --------------------------------
    def decode_graph_us(n_rows):
        """us per decode step of the first n_rows rows (and slots), from one CUDA graph."""
        g = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream(device=dev)
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            cc.cconv_update(xr[0][:n_rows], st, wd, bd, idx[:n_rows], y=yd[:n_rows],
                            status=status)
            with torch.cuda.graph(g, stream=s2):
                for j in range(DEC.steps):
                    cc.cconv_update(xr[j % xr.shape[0]][:n_rows], st, wd, bd, idx[:n_rows],
                                    y=yd[:n_rows], status=status)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        ga.record(stream)
        for _ in range(reps):
            g.replay()
        gb.record(stream)
        torch.cuda.synchronize()
        return ga.elapsed_time(gb) * 1e3 / (reps * DEC.steps)

    dec_graph_us = decode_graph_us(DEC.N)
    dec_small_us = {n: decode_graph_us(n) for n in (1, 16, 64)}
    assert status.tolist() == [0, 0]

    # ---- packed sequences: same rows, 16 mixed lengths, with states ------------------------
    lens = inputs.seqlen_mix(FWD.B * FWD.T, VL_NSEQ, seed=rank)
    vx, vdy, vcu, vw, _, vinit = inputs.varlen_inputs(lens, FWD.D, FWD.W, bias=False, seed=rank)
    vxs = [vx.to(dev) for _ in range(NSET)]
    vdys = [vdy.to(dev) for _ in range(NSET)]
    vinits = [vinit.to(dev) for _ in range(NSET)]
    vcu, vw = vcu.to(dev), vw.to(dev)
    vfin = torch.empty_like(vinits[0])
    vdinit = torch.empty_like(vinits[0])
    vws = torch.empty(cc.cconv_bwd_varlen_workspace_bytes(FWD.B * FWD.T, FWD.D, FWD.W),
                      dtype=torch.uint8, device=dev)

    def vfwd(i):
        k = i % NSET
        cc.cconv_fwd_varlen(vxs[k], vcu, vw, None, initial_state=vinits[k], final_state=vfin,
                            y=ys[k].view(-1, FWD.D))

    def vbwd(i):
        k = i % NSET
        cc.cconv_bwd_varlen(vxs[k], vdys[k], vcu, vw, None, initial_state=vinits[k],
                            want_dbias=True, dx=dxs[k].view(-1, FWD.D), dw=dw, dbias=db,
                            d_initial_state=vdinit, workspace=vws)

    for fn in (vfwd, vbwd):
        for i in range(3):
            fn(i)
    vf_us, vb_us = graph_us(vfwd, K), graph_us(vbwd, K)

    # ---- q, k, v of a layer in one launch: D = 1024, 1024, 2048 (same rows and bytes) -------
    qkv_D = [FWD.D // 4, FWD.D // 4, FWD.D // 2]
    qsets = []
    for k in range(NSET):
        pr = [inputs.fwd_bwd_inputs(FWD.B, FWD.T, D, FWD.W, False, seed=rank * 100 + 10 * k + j)
              for j, D in enumerate(qkv_D)]
        qsets.append(([t[0].to(dev) for t in pr], [t[1].to(dev) for t in pr]))
    qw = [inputs.fwd_bwd_inputs(1, 1, D, FWD.W, False, seed=j)[2].to(dev)
          for j, D in enumerate(qkv_D)]
    qys = [[torch.empty(FWD.B, FWD.T, D, dtype=torch.bfloat16, device=dev) for D in qkv_D]
           for _ in range(NSET)]
    qdxs = [[torch.empty(FWD.B, FWD.T, D, dtype=torch.bfloat16, device=dev) for D in qkv_D]
            for _ in range(NSET)]
    qdws = [torch.empty(D, FWD.W, device=dev) for D in qkv_D]
    qdbs = [torch.empty(D, device=dev) for D in qkv_D]
    qws = torch.empty(cc.cconv_bwd_multi_workspace_bytes(qkv_D, FWD.B, FWD.T, FWD.W),
                      dtype=torch.uint8, device=dev)
    qws1 = [torch.empty(cc.cconv_bwd_workspace_bytes(FWD.B, FWD.T, D, FWD.W), dtype=torch.uint8,
                        device=dev) for D in qkv_D]

    def qfwd(i):
        k = i % NSET
        cc.cconv_fwd_multi(qsets[k][0], qw, ys=qys[k])

    def qbwd(i):
        k = i % NSET
        cc.cconv_bwd_multi(qsets[k][0], qsets[k][1], qw, want_dbias=True, dxs=qdxs[k], dws=qdws,
                           dbiases=qdbs, workspace=qws)

    def qfwd3(i):
        k = i % NSET
        for j in range(3):
            cc.cconv_fwd(qsets[k][0][j], qw[j], None, y=qys[k][j])

    def qbwd3(i):
        k = i % NSET
        for j in range(3):
            cc.cconv_bwd(qsets[k][0][j], qsets[k][1][j], qw[j], None, want_dbias=True,
                         dx=qdxs[k][j], dw=qdws[j], dbias=qdbs[j], workspace=qws1[j])

    for fn in (qfwd, qbwd, qfwd3, qbwd3):
        for i in range(3):
            fn(i)
    qf_us, qb_us = graph_us(qfwd, K), graph_us(qbwd, K)
    qf3_us, qb3_us = graph_us(qfwd3, K), graph_us(qbwd3, K)

    # ---- what each part launches (launch descriptions: nothing runs) -----------------------
    kern = {name: kernels_of(cc, lambda f=f: f(0), max_thr)
            for name, f in (("fwd", fwd), ("bwd", bwd), ("decode_update", upd),
                            ("fwd_varlen", vfwd), ("bwd_varlen", vbwd),
                            ("fwd_qkv_one_launch", qfwd), ("bwd_qkv_one_launch", qbwd))}
    del qsets

    # ---- end to end through the public API with host buffers ------------------------------
    e2e = run_e2e(cc, dev, stream, args, x, dy, w, wg, ws, xr, st, wd, bd, idx, world)

    cpu = cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)
        cpu_all = cpu_baseline_all_cores(args.cpu_seconds, cpu)

    if rank != 0:
        return None
    peak_gbs, peak_kind = measured_peak()

    def tb(nbytes, us):
        return nbytes / (us * 1e-6) / 1e12

    def part(nbytes, us, eager=None, **extra):
        row = {"us": round(us, 3), "tbps": round(tb(nbytes, us), 4),
               "frac_of_peak": round(tb(nbytes, us) * 1e3 / peak_gbs, 4),
               "algorithmic_bytes": nbytes}
        if eager is not None:
            row["us_eager"] = round(eager, 3)
        row.update(extra)
        return row

    bwd_tbps = tb(BWD_BYTES, b_us)
    value = aggregate(STEP_BYTES * K, elapsed_max, world) / 1e12
    out = {
        "metric": METRIC,
        "value": round(value, 4),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed_max * 1e3 / K, 5),
        "ms_per_step_eager": round(eager_step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD,
            "storage": "bf16 activations and state, f32 weights",
            "l2": "inputs larger than L2 and rotated: each launch reads buffers the previous "
                  "launch did not touch (per-launch working set >= 268 MB > 129 MB L2)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "parts": {
            "fwd": part(FWD_BYTES, f_us, f_eager, kernels=kern["fwd"]),
            "bwd": part(BWD_BYTES, b_us, b_eager, kernels=kern["bwd"],
                        note="stream kernel + deterministic reduction kernel; dx, dw, dbias"),
            "decode_update": {"us_per_step_graph_1000": round(dec_graph_us, 3),
                              "us_per_call_graph": round(u_us, 3),
                              "us_per_call_eager": round(u_eager, 3),
                              "bytes_per_step": DEC_BYTES, "kernels": kern["decode_update"]},
            "decode_update_small_batches": {
                "us_per_step_graph": {str(n): round(v, 3) for n, v in dec_small_us.items()},
                "note": "the same pool, weights and tokens, first N rows and slots only"},
            "fwd_varlen": part(VL_FWD_BYTES, vf_us, kernels=kern["fwd_varlen"],
                               note=f"{VL_NSEQ} packed sequences of mixed lengths, same rows; "
                                    "initial states in, final states out (one stream kernel; "
                                    "final states from its register ring)"),
            "bwd_varlen": part(VL_BWD_BYTES, vb_us, kernels=kern["bwd_varlen"],
                               note="same packing; initial states in, dx, dw, dbias and the "
                                    "initial-state gradient out (stream + reduction kernel)"),
            "fwd_qkv_one_launch": part(FWD_BYTES, qf_us, kernels=kern["fwd_qkv_one_launch"],
                                       three_calls_us=round(qf3_us, 3),
                                       note="q, k, v convolutions of a layer (D = 1024, 1024, "
                                            "2048, same B, T) in one launch vs three cconv_fwd "
                                            "calls"),
            "bwd_qkv_one_launch": part(BWD_BYTES, qb_us, kernels=kern["bwd_qkv_one_launch"],
                                       three_calls_us=round(qb3_us, 3)),
        },
        "roofline": {
            "kernel": "cconv_bwd (stream + reduction)",
            "bound": "hbm",
            "achieved": round(bwd_tbps * 1e3, 1),
            "peak": peak_gbs,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(bwd_tbps * 1e3 / peak_gbs, 4),
            "traffic": bwd_traffic(),
            "traffic_profile": BWD_TRAFFIC["profile"],
            "algorithmic_bytes_per_launch": BWD_BYTES,
        },
        "e2e": e2e,
        "gpu_launches": LAUNCHES_PER_STEP * K,
        "timing": "value: K whole steps (every kernel of every step) captured once in a CUDA "
                  "graph and replayed between two CUDA events on the launching stream "
                  "(ms_per_step_eager: the same K steps as eager calls); parts: device time per "
                  "call from calls captured in one CUDA graph and replayed between two events "
                  "(us_eager: K back-to-back eager calls); decode: 1000 updates replayed from "
                  "one CUDA graph",
        "clocks": clk.summary(),
        "wall_s_timed": round(wall, 4),
    }
    if cpu is not None:
        out["cpu_baseline"] = cpu
    if cpu_all is not None:
        out["cpu_baseline_all_cores"] = cpu_all
    return out


def run_e2e(cc, dev, stream, args, x, dy, w, wg, ws, xr, st, wd, bd, idx, world):
    """The same step through the public API, inputs copied in from pinned host memory and
    results (y, dx, dw, decode y) copied back, copies inside the timed region.

    Steps are pipelined the way a data loader feeds a device: step i+1's inputs go up on
    one stream while step i computes on the launching stream and step i-1's results come
    down on a third (the two copy directions run on separate copy engines).  Device
    buffers are double-buffered and every reuse waits on the event that frees it."""
    NB = 2
    hx = [x.pin_memory() for _ in range(NB)]
    hdy = [dy.pin_memory() for _ in range(NB)]
    hxd = [xr[0].cpu().pin_memory() for _ in range(NB)]
    hy = [torch.empty_like(hx[0]).pin_memory() for _ in range(NB)]
    hdx = [torch.empty_like(hx[0]).pin_memory() for _ in range(NB)]
    hdw = [torch.empty(wg.shape, dtype=wg.dtype).pin_memory() for _ in range(NB)]
    hdb = [torch.empty(wg.shape[0], dtype=wg.dtype).pin_memory() for _ in range(NB)]
    hyd = [torch.empty(DEC.N, DEC.D, dtype=torch.bfloat16).pin_memory() for _ in range(NB)]
    x_ = [torch.empty(x.shape, dtype=torch.bfloat16, device=dev) for _ in range(NB)]
    dy_ = [torch.empty_like(x_[0]) for _ in range(NB)]
    y_ = [torch.empty_like(x_[0]) for _ in range(NB)]
    dx_ = [torch.empty_like(x_[0]) for _ in range(NB)]
    dw_ = [torch.empty_like(wg) for _ in range(NB)]
    db_ = [torch.empty(wg.shape[0], dtype=wg.dtype, device=dev) for _ in range(NB)]
    xd_ = [torch.empty(DEC.N, DEC.D, dtype=torch.bfloat16, device=dev) for _ in range(NB)]
    yd_ = [torch.empty_like(xd_[0]) for _ in range(NB)]
    status = torch.zeros(2, dtype=torch.int32, device=dev)
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    uploaded = [torch.cuda.Event() for _ in range(NB)]
    computed = [torch.cuda.Event() for _ in range(NB)]
    downloaded = [torch.cuda.Event() for _ in range(NB)]
    for k in range(NB):   # every buffer starts free
        computed[k].record(stream)
        downloaded[k].record(stream)

    def upload(i):
        k = i % NB
        up.wait_event(computed[k])          # step i-NB has finished reading these inputs
        with torch.cuda.stream(up):
            x_[k].copy_(hx[k], non_blocking=True)
            dy_[k].copy_(hdy[k], non_blocking=True)
            xd_[k].copy_(hxd[k], non_blocking=True)
        uploaded[k].record(up)

    def compute(i):
        k = i % NB
        stream.wait_event(uploaded[k])
        stream.wait_event(downloaded[k])    # step i-NB's results have been copied out
        cc.cconv_fwd(x_[k], wg, None, y=y_[k], stream=stream)
        cc.cconv_bwd(x_[k], dy_[k], wg, None, want_dbias=True, dx=dx_[k], dw=dw_[k],
                     dbias=db_[k], workspace=ws, stream=stream)
        cc.cconv_update(xd_[k], st, wd, bd, idx, y=yd_[k], status=status, stream=stream)
        computed[k].record(stream)

    def download(i):
        k = i % NB
        down.wait_event(computed[k])
        with torch.cuda.stream(down):
            hy[k].copy_(y_[k], non_blocking=True)
            hdx[k].copy_(dx_[k], non_blocking=True)
            hdw[k].copy_(dw_[k], non_blocking=True)
            hdb[k].copy_(db_[k], non_blocking=True)
            hyd[k].copy_(yd_[k], non_blocking=True)
        downloaded[k].record(down)

    def run(n):
        """n pipelined steps: uploads run one step ahead, downloads one step behind."""
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute(i)
            if i > 0:
                download(i - 1)
        download(n - 1)

    run(3)
    torch.cuda.synchronize()
    n = args.e2e_steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    a.record(up)
    run(n)
    stream.wait_stream(down)
    stream.wait_stream(up)
    b.record(stream)
    torch.cuda.synchronize()
    el = max_over_ranks(a.elapsed_time(b) / 1e3, world, dev)
    h2d = (hx[0].numel() + hdy[0].numel() + hxd[0].numel()) * 2
    d2h = ((hy[0].numel() + hdx[0].numel() + hyd[0].numel()) * 2
           + (hdw[0].numel() + hdb[0].numel()) * hdw[0].element_size())
    return {"value": round(aggregate(STEP_BYTES * n, el, world) / 1e12, 4), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(el * 1e3 / n, 4), "steps": n,
            "pipelined": "step i+1's upload, step i's kernels and step i-1's download overlap "
                         "on three streams; every step's copies are inside the timed region"}


# ---------------------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------------------

def _oracle_sample(B: int, rows: int):
    """Inputs for a bounded sample of the workload: B sequences' first `rows` rows at the
    production width, plus the decode workload's pool and two token rows."""
    import oracle
    x, dy, w, _ = inputs.fwd_bwd_inputs(B, rows, FWD.D, FWD.W, False)
    xd, dyd, wdd = (t.double().numpy() for t in (x, dy, w))
    st, xr, idx, wdec, bdec = inputs.decode_inputs(DEC.S, DEC.N, DEC.D, DEC.W, DEC.bias, n_x=2)
    stb = st.view(torch.int16).numpy().view(np.uint16).copy()
    xrb = xr.view(torch.int16).numpy().view(np.uint16)
    return oracle, (xd, dyd, wdd), (stb, xrb, idx.numpy(), wdec.double().numpy(),
                                    bdec.double().numpy())


def _oracle_step(o, fb, dec):
    """One step of the workload's composition on the oracle: fwd + bwd of the sample, then
    one decode update.  Returns the algorithmic bytes it stands for."""
    xd, dyd, wdd = fb
    o.fwd(xd, wdd, None)
    o.bwd(xd, dyd, wdd, None, want_dbias=True)
    stb, xrb, idx, wdec, bdec = dec
    rc, _, new = o.update(xrb[0], stb, idx, wdec, bdec)
    assert rc == 0
    dec[0][...] = new
    return xd.size * (FWD_BYTES + BWD_BYTES) / N_ELEM + DEC_BYTES


def cpu_baseline(seconds: float):
    """The oracle, as it stands, on whole steps of the workload (B=2 T=8192 D=4096 fwd+bwd
    + one decode update each), repeated while the total stays near `seconds`."""
    o, fb, dec = _oracle_sample(FWD.B, FWD.T)
    t0 = time.perf_counter()
    nbytes = _oracle_step(o, fb, dec)
    steps = 1
    while True:
        dt = time.perf_counter() - t0
        if dt * (steps + 1) / steps > seconds:
            break
        nbytes += _oracle_step(o, fb, dec)
        steps += 1
    dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e12, 8), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"fp64 C oracle, one thread: {steps} whole workload step(s) (fwd+bwd "
                      f"B={FWD.B} T={FWD.T} D={FWD.D} W={FWD.W} + 1 decode update), "
                      f"{dt:.2f} s"}


def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _slice_worker(k: int, n: int, steps: int, ready, go, done):
    """One process of the all-cores oracle run: channels of slice k of n (the convolution is
    depthwise, so channel slices are independent problems) of the whole workload step."""
    import oracle
    d = FWD.D // n + (1 if k < FWD.D % n else 0)
    x, dy, w, _ = inputs.fwd_bwd_inputs(FWD.B, FWD.T, d, FWD.W, False, seed=k)
    xd, dyd, wdd = (t.double().numpy() for t in (x, dy, w))
    st, xr, idx, wdec, bdec = inputs.decode_inputs(DEC.S, DEC.N, d, DEC.W, DEC.bias, n_x=1,
                                                   seed=k)
    stb = st.view(torch.int16).numpy().view(np.uint16).copy()
    xrb = xr[0].view(torch.int16).numpy().view(np.uint16)
    idxn, wdn, bdn = idx.numpy(), wdec.double().numpy(), bdec.double().numpy()
    ready.put(k)
    go.wait()
    t0 = time.perf_counter()
    for _ in range(steps):
        o_fwd = oracle.fwd(xd, wdd, None)
        oracle.bwd(xd, dyd, wdd, None, want_dbias=True)
        rc, _, new = oracle.update(xrb, stb, idxn, wdn, bdn)
        assert rc == 0 and o_fwd.shape == xd.shape
        stb[...] = new
    done.put((k, time.perf_counter() - t0))


def cpu_baseline_all_cores(seconds: float, single: dict | None):
    """The same oracle on every host core at once: one process per core, each running whole
    workload steps on its slice of the channels; whole-job throughput over the wall time of
    the slowest process.  Processes are spawned (never forked after CUDA is initialised)."""
    import multiprocessing as mp
    n = _cores()
    per_step_1 = None
    if single is not None and single.get("value"):
        per_step_1 = (FWD_BYTES + BWD_BYTES + DEC_BYTES) / (single["value"] * 1e12)
    steps = max(1, int(seconds * n / per_step_1 / 1.3)) if per_step_1 else 2
    ctx = mp.get_context("spawn")
    ready, done, go = ctx.Queue(), ctx.Queue(), ctx.Event()
    procs = [ctx.Process(target=_slice_worker, args=(k, n, steps, ready, go, done), daemon=True)
             for k in range(n)]
    for pr in procs:
        pr.start()
    try:
        for _ in range(n):
            ready.get(timeout=600)
        t0 = time.perf_counter()
        go.set()
        times = [done.get(timeout=max(600, 20 * seconds))[1] for _ in range(n)]
        wall = time.perf_counter() - t0
    finally:
        for pr in procs:
            pr.join(timeout=60)
    nbytes = steps * (FWD_BYTES + BWD_BYTES + DEC_BYTES)
    return {"value": round(nbytes / wall / 1e12, 8), "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"fp64 C oracle (unchanged), one process per core, each running {steps} "
                      f"whole workload step(s) (fwd+bwd B={FWD.B} T={FWD.T} W={FWD.W} + 1 "
                      f"decode update) on its 1/{n} of the D={FWD.D} channels; wall {wall:.2f} s, "
                      f"slowest process {max(times):.2f} s"}


def run_reference(args, world, rank):
    """The oracle timed as the reference arm: each step is a bounded sample of the workload
    (the first `rows` rows of one sequence, fwd + bwd, plus one decode update), sized so the
    whole run takes about `--reference-seconds`."""
    if rank != 0:
        return None
    o, fb, dec = _oracle_sample(1, 64)
    t0 = time.perf_counter()
    _oracle_step(o, fb, dec)
    t_small = time.perf_counter() - t0
    o, fb, dec = _oracle_sample(1, 128)
    t0 = time.perf_counter()
    _oracle_step(o, fb, dec)
    per_row = max(1e-7, (time.perf_counter() - t0 - t_small) / 64)
    fixed = max(0.0, t_small - 64 * per_row)
    total = max(1, args.steps + args.warmup)
    rows = int((args.reference_seconds / total - fixed) / per_row)
    rows = max(8, min(FWD.T, rows))
    o, fb, dec = _oracle_sample(1, rows)
    for _ in range(args.warmup):
        _oracle_step(o, fb, dec)
    t0 = time.perf_counter()
    nbytes = 0.0
    for _ in range(args.steps):
        nbytes += _oracle_step(o, fb, dec)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e12
    sample = (f"fp64 C oracle, one thread; per step: fwd+bwd of one sequence's first {rows} "
              f"rows at D={FWD.D} W={FWD.W} + 1 decode update (S={DEC.S} N={DEC.N} D={DEC.D})")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 8),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_per_step": sample},
        "cpu_baseline": {"value": round(value, 8), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 8), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the (untimed) oracle baseline leg")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" and torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)

    if args.impl == "reference":
        out = run_reference(args, world, rank)
    else:
        out = run_ours(args, world, rank, local)
    if out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
