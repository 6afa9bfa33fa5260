"""Benchmark of the S4 layer forward pass (kernel generation + fused FFT
convolution) on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one s4_layer_fwd over one batch of the largest workload, N=256,
r=1, H=1024, L=65536, batch 2 (synthetic inputs resident in HBM); --workload
picks one of the smaller seeded workloads instead.  Input/output buffer sets
rotate so that the bytes touched between two uses of the same buffer exceed
twice the L2 size.  `value` is channel-samples per second (batch*H*L per step,
summed over ranks / max time over ranks).  `e2e` times the same call with the
input copied from pinned host memory and the output copied back every step.
Each step replays a CUDA graph holding one captured s4_layer_fwd call (one
graph per buffer set), so host launch overhead does not enter the timing.
Per-kernel durations come from the library's launch events (CUDA events on
the launch stream around every kernel) over eager C-ABI calls.  The CPU
baseline is the float64 oracle on the host cores, on a stated sample of the
workload's channels.  `--impl reference` times that oracle alone.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "S4 layer fwd channel-samples/s (B·H·L/s); Cauchy terms/s; % FP32 / HBM roofline"
UNIT = "channel-samples/s"
# The layer's bench line is the largest workload (index 4), the one that fits
# one GPU with the most work; --workload selects another of the seeded
# workloads.  The auxiliary paths (--path) default to workload 1.  Spawned
# oracle workers read the choice from the environment.
LAYER_WORKLOAD = 4
PATH_WORKLOAD = 1
WORKLOAD_INDEX = int(os.environ.get("S4_BENCH_WORKLOAD", str(LAYER_WORKLOAD)))
FP32_LANES_PER_SM = 128


def cauchy_flop(r):
    """Algorithmic flop per (channel, root, pole) term of the direct root-value
    sums: 8 (r+1)^2 for the complex multiply-adds of the (r+1)^2 weighted
    reciprocals, plus 10 for the denominator s - lambda_j and its reciprocal
    (42 at rank 1, 82 at rank 2)."""
    return 8 * (r + 1) ** 2 + 10


FAR_TERMS = 42  # the far-root series' largest number of terms (the library's kFarTerms)


def cauchy_work(p, w, sms):
    """The root-value kernel's algorithmic flop for one call, as it splits the
    roots: a warp's 32 RPT consecutive roots (RPT roots per thread) with any root
    near the channel's poles (|s - c| < 1.5 R) sum directly over the N poles
    (cauchy_flop per pole and root, for every root of the warp); the other roots
    evaluate the series, (r+1)^2 (P - 1) complex multiply-adds of 8 flop plus ~24
    flop of set-up each, P the terms their warp takes.  With the series' second
    level (rank 1, large grids, 128 <= N <= 512) a near warp instead sums directly over
    the poles of each of the 4 groups (equal widths in imaginary part) it is near
    and takes the group series of the others.  The split is replayed here in
    float64 from the parameters (the kernel decides in fp32; the two can differ
    only at a warp on the boundary).  Returns (flop, fraction of root-pole terms
    summed directly)."""
    import numpy as np
    H, N, r, M = w.H, w.N, w.r, w.M
    nw = (r + 1) ** 2
    if M < 8192 or N < 48:  # the library takes the series only on rows of M >= 8192 roots, N >= 48 poles
        return H * M * N * cauchy_flop(r), 1.0
    big = H * M >= 512 * 5 * 2 * sms
    cta = 32 * (4 if (big and r <= 2) else (2 if r <= 2 else 1))  # roots per warp
    grouped = r == 1 and big and 128 <= N <= 512
    G = 4
    k = np.arange(M)
    t = np.tan(np.pi * k / M)
    direct_roots = 0
    far_terms = 0
    grp_flop = 0.0  # near warps of grouped channels: direct over near groups, series for the others
    grp_terms = 0   # (root, pole) terms those warps sum directly
    far_roots = 0
    for h in range(H):
        lam = p["Lambda"][h].astype(np.complex128)
        c = 0.5 * (lam.real.min() + lam.real.max()) + 0.5j * (lam.imag.min() + lam.imag.max())
        R = np.abs(lam - c).max() or 1.0
        a = 2.0 / float(p["dt"][h])
        u = 1j * a * t - c
        far = np.abs(u) ** 2 >= 2.25 * R * R
        if M >= 2:
            far[M // 2] = True
        nb = -(-M // cta)
        pad = np.ones(nb * cta, bool)
        pad[:M] = far
        blk_far = pad.reshape(nb, cta).all(axis=1)
        if grouped:
            lo, hi = lam.imag.min(), lam.imag.max()
            gid = np.minimum(np.where(hi > lo, (lam.imag - lo) * G / max(hi - lo, 1e-300), 0).astype(int), G - 1)
            gsets = [lam[gid == g] for g in range(G)]
            gpar = []
            for gl in gsets:
                if len(gl) == 0:
                    gpar.append((0j, 1.0, 0))
                    continue
                cg = 0.5 * (gl.real.min() + gl.real.max()) + 0.5j * (gl.imag.min() + gl.imag.max())
                gpar.append((cg, np.abs(gl - cg).max() or 1.0, len(gl)))
            padu = np.full(nb * cta, 1e300 + 0j)
            padu[:M] = 1j * a * t
            for wi in np.where(~blk_far)[0]:
                sw = padu[wi * cta:(wi + 1) * cta]
                sw = sw[np.abs(sw) < 1e299]
                for cg, Rg, ng in gpar:
                    ug = sw - cg
                    if np.all(np.abs(ug) >= 1.5 * Rg):
                        axg = np.abs(Rg / ug).max()
                        P = int(np.clip(23 / -np.log2(max(axg, 1e-300)) + 2, 1, FAR_TERMS))
                        grp_flop += cta * (nw * 8 * (P - 1) + 24)
                    else:
                        grp_flop += cta * ng * cauchy_flop(r)
                        grp_terms += cta * ng
            # the warps' roots are counted by grp_flop instead of the full direct sum
        else:
            direct_roots += int((~blk_far).sum()) * cta
        # terms of the series per root, as the kernel takes them (the warp's largest)
        with np.errstate(divide="ignore", invalid="ignore"):
            ax = np.abs(R / u)
            need = np.where((ax > 0) & np.isfinite(ax), 23 / -np.log2(ax), 1) + 2
        need = np.clip(np.nan_to_num(need, nan=1.0), 1, FAR_TERMS).astype(int)
        padn = np.ones(nb * cta, int)
        padn[:M] = need
        warp = padn.reshape(nb, cta).max(axis=1, keepdims=True).repeat(cta, axis=1)
        far_terms += int(warp[blk_far].sum())
        far_roots += int(blk_far.sum()) * cta
    # far_terms counts, per far root, the terms P its warp takes: P - 1 Horner steps each
    flop = (direct_roots * N * cauchy_flop(r) + grp_flop + nw * 8 * max(far_terms - far_roots, 0)
            + 24 * far_roots)
    return flop, (direct_roots * N + grp_terms) / (H * M * N)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def dist_env():
    from structured_state_space_gb300.multi import dist_env as _d
    return _d()


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU is busy."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.err = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception as e:  # no nvidia-smi
            self.err = str(e)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"error": self.err or "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"error": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "structured_state_space_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


_FFT_FILES = ["fft_rows.cu", "fft_fourstep.cu", "s4_fft.cuh", "s4_kspec.cuh", "s4_dev.cuh", "s4_plan.cuh",
              "../gen_twiddles.py"]
KERNEL_FILES = {
    "conv": _FFT_FILES,
    "cauchy": ["cauchy.cu", "s4_dev.cuh", "s4_internal.h", "../gen_twiddles.py"],
    "spectrum": _FFT_FILES,
    "kspec": _FFT_FILES,
    "ifft": _FFT_FILES,
}


def profiled_traffic(kernel, workload):
    """DRAM bytes per step of a part (the sum over its launches) on `workload`
    from the committed ncu summary, if they were taken on the current source of
    that part's kernels; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
        e = d[workload][kernel]
        if e.get("source_hash") != kernel_source_hash(KERNEL_FILES[kernel]):
            return None
        return e["dram_bytes_per_launch"]
    except Exception:
        return None


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm) -- run in spawned worker processes
# ---------------------------------------------------------------------------

def _oracle_init():
    os.environ["OMP_NUM_THREADS"] = "1"
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["MKL_NUM_THREADS"] = "1"


def _oracle_channel(args):
    """Oracle on one channel: its kernel and the convolution of each of the
    channel's input rows.  `args` carries the channel's parameters and rows
    (sent by the parent, so workers never build the whole workload).
    Returns the channel-samples produced."""
    lam, P, Q, B, Ct, dt, D, rows, L = args
    import oracle.s4_oracle as O
    K = O.s4_kernel(lam, P, Q, B, Ct, dt, L)
    for row in rows:
        O.causal_conv(K, row, D)
    return len(rows) * L


def channel_units(p, u, chans, L):
    """Work items of _oracle_channel for the listed channels (all batch rows)."""
    import numpy as np
    return [(p["Lambda"][h], p["P"][h], p["Q"][h], p["B"][h], p["Ctilde"][h], float(p["dt"][h]),
             float(p["D"][h]), np.ascontiguousarray(u[:, h, :]), L) for h in chans]


def baseline_channels(w):
    """Channels of the CPU baseline's sample: every channel of the small
    workloads, the stated 8-channel sample (first two, middle two, last, four
    seeded) of the large ones."""
    from structured_state_space_gb300 import workloads as W
    return list(range(w.H)) if w.batch * w.H * w.L <= (1 << 24) else W.sample_channels(w)


_DATA = None


def _oracle_data():
    global _DATA
    if _DATA is None:
        from structured_state_space_gb300 import workloads as W
        w = W.WORKLOADS[WORKLOAD_INDEX]
        p = W.make_params(w)
        _DATA = (p, W.make_u(w, p))
    return _DATA


def _warm_unit():
    """A tiny oracle work item: imports and first-call costs out of the timing."""
    import numpy as np
    N, L = 4, 64
    lam = (-0.5 + 1j * np.pi * np.arange(N)).astype(np.complex64)
    v = np.full(N, 0.1, np.complex64)
    return (lam, v.reshape(N, 1), v.reshape(N, 1), v, v, 0.01, 0.5, np.ones((1, L), np.float32), L)


def make_pool(procs):
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(procs, initializer=_oracle_init)
    pool.map(_oracle_channel, [_warm_unit()] * procs)
    return pool


CPU_BASELINE_CPU_S = 12.0  # whole passes until about this much CPU time is spent


def timed_passes(pool, procs, fn, items, max_passes=50):
    """Whole passes of pool.map(fn, items), repeated until the pool has spent
    about CPU_BASELINE_CPU_S seconds of CPU time (wall x procs).  Returns the
    units done (sum of fn's results), the wall seconds and the passes."""
    t0 = time.perf_counter()
    done, passes = 0, 0
    while True:
        done += sum(pool.map(fn, items))
        passes += 1
        dt = time.perf_counter() - t0
        if dt * procs >= CPU_BASELINE_CPU_S or passes >= max_passes:
            return done, dt, passes


def oracle_rate(pool, procs, units):
    samples, dt, passes = timed_passes(pool, procs, _oracle_channel, units)
    return samples / dt, dt, samples, passes


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def fp32_probe(dev, fp32_peak, iters=4096, reps=5):
    """FP32 issue rate the SMs sustain (the library's FFMA probe, 8 CTAs of 256
    threads per SM), beside the peak derived from unit counts and clocks."""
    import torch
    import structured_state_space_gb300 as s4
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks = sms * 8
    out = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    for _ in range(3):
        s4.s4_fp32_probe(out, blocks, iters)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    flop = sum(s4.s4_fp32_probe(out, blocks, iters) for _ in range(reps))
    e1.record()
    torch.cuda.synchronize()
    tf = flop / (e0.elapsed_time(e1) / 1e3) / 1e12
    return {"achieved": tf, "unit": "TFLOP/s", "frac_of_derived_peak": tf / fp32_peak,
            "how": f"s4_fp32_probe: {blocks} CTAs x 256 threads x {iters} iterations of 8 independent FFMA "
                   f"chains, {reps} launches timed with CUDA events"}


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import structured_state_space_gb300 as s4
    from structured_state_space_gb300 import build as s4build
    from structured_state_space_gb300 import multi
    from structured_state_space_gb300 import workloads as W

    rank, local_rank, world = dist_env()
    w = W.WORKLOADS[WORKLOAD_INDEX]
    if args.channels:  # a reduced-channel copy for profiling (same N, r, L, batch and distributions)
        w = dataclasses.replace(w, H=args.channels, name=f"{w.name} with H={args.channels} (profiling copy)")
    # CPU baseline pool first: spawned before any GPU work, one process per
    # sampled channel up to the host's cores
    pool, procs = None, 0
    base_chans = baseline_channels(w)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        procs = max(1, min(os.cpu_count() or 1, len(base_chans)))
        pool = make_pool(procs)

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0:
        s4build.build()
    if world > 1:
        dist.barrier()
    s4.load()

    H, N, r, L, Bsz, M = w.H, w.N, w.r, w.L, w.batch, w.M
    p = W.make_params(w)
    u_host = W.make_u(w, p)
    dev = torch.device("cuda", local_rank)
    prm = {k: torch.from_numpy(np.ascontiguousarray(p[k])).to(dev) for k in ["Lambda", "P", "Q", "B", "Ctilde", "dt", "D"]}
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    set_bytes = Bsz * H * L * (4 + 8)
    # enough rotating sets to exceed twice the L2, at most 16: a workload whose
    # 16 sets still fit in L2 is timed L2-resident and says so in its line
    nsets = min(16, max(3, math.ceil(2 * l2 / set_bytes) + 1))
    l2_note = (f"{nsets} rotating input/output sets of {set_bytes / 2**20:.0f} MiB (> 2x L2 {l2 / 2**20:.0f} MiB)"
               if nsets * set_bytes > 2 * l2 else
               f"{nsets} rotating sets of {set_bytes} B: inputs L2-resident (workload far smaller than L2)")
    u_d = [torch.from_numpy(u_host).to(dev) for _ in range(nsets)]
    y_d = [torch.empty((Bsz, H, L), dtype=torch.complex64, device=dev) for _ in range(nsets)]
    K_d = torch.empty((H, L), dtype=torch.complex64, device=dev)
    ws = s4.workspace(H, N, r, L, Bsz, dev)
    stream = torch.cuda.Stream(dev)

    def layer(i):
        # one pass of the whole path on the current stream (the graph capture stream)
        s4.s4_layer_fwd(prm["Lambda"], prm["P"], prm["Q"], prm["B"], prm["Ctilde"], prm["dt"], prm["D"],
                        u_d[i % nsets], K=K_d, y=y_d[i % nsets], ws=ws)

    with torch.cuda.stream(stream):
        for i in range(3):           # eager warm-up: module load, kernel attributes
            layer(i)
    stream.synchronize()
    st = s4.s4_get_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {s4.s4_status_str(st)}")
    # captured graphs: G consecutive steps (cycling through the buffer sets)
    # in one graph, plus one single-step graph per buffer set for remainders
    G = nsets * 4
    gbig = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gbig, stream=stream):
        for i in range(G):
            layer(i)
    graphs = []
    for j in range(nsets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            layer(j)
        graphs.append(g)

    def timed(body, k):
        # barrier + sync on both sides; the job time is the max over ranks
        multi.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        body(k)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = multi.max_over_ranks(e0.elapsed_time(e1), device=dev)
        multi.barrier()
        return ms

    def replay_steps(k):
        # exactly k steps: k // G replays of the G-step graph, then single steps
        with torch.cuda.stream(stream):
            for _ in range(k // G):
                gbig.replay()
            for j in range(k % G):
                graphs[j % nsets].replay()

    sampler = ClockSampler(local_rank)
    sampler.start()
    replay_steps(args.warmup)
    K = args.steps
    ms_total = timed(replay_steps, K)
    clocks = sampler.stop()

    # per-kernel durations: the library's launch events (CUDA events recorded
    # on the launch stream around every kernel) over S eager steps, issued by
    # direct C-ABI calls while a graph replay keeps the GPU busy, so that the
    # device never waits for the host between a kernel and its events
    S = max(1, min(K, 200))
    lib = s4.load()
    vp = ctypes.c_void_p
    arg_sets = []
    for j in range(nsets):
        arg_sets.append([vp(prm[k].data_ptr()) for k in ["Lambda", "P", "Q", "B", "Ctilde", "dt", "D"]]
                        + [vp(u_d[j].data_ptr()), Bsz, H, N, r, L, vp(K_d.data_ptr()), vp(y_d[j].data_ptr()),
                           vp(ws.data_ptr()), ws.numel(), vp(stream.cuda_stream)])
    s4.timing.reset()
    s4.timing.enable(True)
    for i in range(S):               # create the event pool
        lib.s4_layer_fwd(*arg_sets[i % nsets])
    torch.cuda.synchronize()
    s4.timing.reset()

    def head_start(_k=0):
        with torch.cuda.stream(stream):
            for _ in range(4):
                gbig.replay()

    def prof_steps(k):
        head_start()
        for i in range(k):
            rc = lib.s4_layer_fwd(*arg_sets[i % nsets])
            if rc != 0:
                raise RuntimeError(f"s4_layer_fwd: {s4.s4_status_str(rc)}")

    ms_prof = timed(prof_steps, S)
    s4.timing.enable(False)
    ms_prof -= timed(head_start, 0)
    fams = ["moments", "cauchy", "ifft", "kspec_cross", "spectrum", "spec_fwd", "kspec", "conv", "conv_fwd",
            "conv_col", "conv_inv"]
    raw = {}
    for name in fams:
        n, t = s4.timing.read(name)
        raw[name] = {"launches": n, "avg_us": 1e3 * t / max(n, 1)}
    s4.timing.reset()
    launches_per_step = int(round(sum(v["launches"] for v in raw.values()) / S))
    # the step's parts: the root values, the kernel spectrum (one launch on short
    # rows; on long rows the column inverse transforms, the cross step that writes
    # K, and the column spectra) and the convolution (one launch on short rows;
    # on long rows the across-column step, the column transforms and the inverse
    # across-column step); a part's time is the sum of its launches per step
    groups = {"cauchy": ["cauchy", "moments"], "kspec": ["kspec", "ifft", "kspec_cross", "spectrum", "spec_fwd"],
              "conv": ["conv", "conv_fwd", "conv_col", "conv_inv"]}
    kern = {}
    for g, members in groups.items():
        used = [k for k in members if raw[k]["launches"]]
        if not used:
            continue
        kern[g] = {"launches": max(raw[k]["launches"] for k in used),
                   "avg_us": sum(raw[k]["avg_us"] * raw[k]["launches"] / S for k in used), "share": 0.0}
        if len(used) > 1:
            kern[g]["parts"] = {k: raw[k] for k in used}
    tot = sum(v["avg_us"] for v in kern.values())
    for v in kern.values():
        v["share"] = v["avg_us"] / tot if tot > 0 else 0.0

    # end to end through the public call: every step copies its input from
    # pinned host memory and its output back, pipelined over three streams
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    u_pin = torch.from_numpy(u_host).pin_memory()
    slots = 3
    y_pin = [torch.empty((Bsz, H, L), dtype=torch.complex64).pin_memory() for _ in range(slots)]
    ev_in = [torch.cuda.Event() for _ in range(slots)]
    ev_cp = [torch.cuda.Event() for _ in range(slots)]
    ev_out = [torch.cuda.Event() for _ in range(slots)]

    def e2e_steps(k):
        start = torch.cuda.Event()
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for i in range(k):
            j = i % slots
            if i >= slots:
                s_in.wait_event(ev_out[j])
                stream.wait_event(ev_out[j])
            with torch.cuda.stream(s_in):
                u_d[j].copy_(u_pin, non_blocking=True)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            with torch.cuda.stream(stream):
                graphs[j].replay()
                ev_cp[j].record(stream)
            s_out.wait_event(ev_cp[j])
            with torch.cuda.stream(s_out):
                y_pin[j].copy_(y_d[j], non_blocking=True)
                ev_out[j].record(s_out)
        done = torch.cuda.Event()
        done.record(s_out)
        stream.wait_event(done)

    e2e_n = max(3, min(K, 500))
    e2e_steps(6)
    ms_e2e = timed(e2e_steps, e2e_n)
    e2e_steps_done = e2e_n

    samples_step = Bsz * H * L
    value = multi.job_throughput(samples_step, K, world, ms_total)
    e2e_value = multi.job_throughput(samples_step, e2e_steps_done, world, ms_e2e)

    peaks, peak_src = read_peaks()
    sms = props.multi_processor_count
    fp32_peak = sms * FP32_LANES_PER_SM * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    peak_source = f"{sms} SMs (queried) x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x max SM clock"
    lg2m = (2 * M).bit_length() - 1
    # algorithmic work per launch of each kernel family: (bound, amount, description)
    cflop, direct_frac = cauchy_work(p, w, sms)
    work = {
        "cauchy": ("alu", cflop,
                   f"{cauchy_flop(r)} flop per (channel, root, pole) on the {100 * direct_frac:.2f} % of root-pole terms summed "
                   f"directly, 8 (r+1)^2 (P - 1) + 24 flop per far root (series of P <= {FAR_TERMS} terms)"),
        "conv": ("hbm", Bsz * H * L * (4 + 8) + H * 2 * M * 8,
                 "u 4 B + y 8 B per channel-sample, kernel spectrum 16 B per channel-root once"),
        "spectrum": ("hbm", H * L * 8 + H * 2 * M * 8, "K 8 B per tap in, spectrum 8 B per 2M bin out"),
        "kspec": ("hbm", H * M * 8 + H * L * 8 + H * 2 * M * 8,
                  "root values 8 B in, K 8 B out, spectrum 8 B per 2M bin out"),
        "ifft": ("hbm", H * M * 8 + H * L * 8, "root values 8 B in, K 8 B out"),
    }

    def roof_of(name):
        bound, amount, desc = work[name]
        t = kern[name]["avg_us"] * 1e-6
        if bound == "alu":
            ach = amount / t / 1e12
            e = {"kernel": f"{name}_kernel", "bound": "alu", "achieved": ach, "peak": fp32_peak,
                 "unit": "TFLOP/s", "frac": ach / fp32_peak, "peak_source": peak_source}
        else:
            ach = amount / t / 1e9
            e = {"kernel": f"{name}_kernel", "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                 "unit": "GB/s", "frac": ach / peaks["hbm_gbs"]}
        e["traffic"] = profiled_traffic(name, w.name)
        e["algorithmic"] = desc
        e["avg_us"] = kern[name]["avg_us"]
        if name == "conv":
            # the transforms' arithmetic (about 15 flop per byte moved) is above the FP32/HBM
            # ridge (about 12 flop per byte), so the FP32 side is reported as well
            cflops = Bsz * H * (15 * M * lg2m + 16 * M)
            cach = cflops / t / 1e12
            e["fp32"] = {"achieved": cach, "peak": fp32_peak, "unit": "TFLOP/s", "frac": cach / fp32_peak,
                         "algorithmic": "15 M log2(2M) + 16 M flop per batch row (real-input forward, "
                                        "complex inverse, 5 n log2 n per transform)"}
        return e

    # roofline of the dominant kernel, the other kernels of the step beside it
    dom = max(kern, key=lambda k: kern[k]["avg_us"])
    roof = roof_of(dom)
    roof["peak_kind"] = f"of {peak_src}"
    roof["fp32_probe"] = fp32_probe(dev, fp32_peak)
    roof["others"] = {k: roof_of(k) for k in kern if k != dom and kern[k]["launches"]}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_total / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": w.name, "N": N, "r": r, "H": H, "L": L, "M": M, "batch": Bsz,
                   "parallelism": f"replica x{world} (channels independent, no collective)",
                   "l2": l2_note},
        "cauchy_terms_per_s_direct_equivalent": H * M * N * (r + 1) ** 2 * world * K / (ms_total / 1e3),
        "gpu_launches": launches_per_step * K,
        "kernels": kern,
        "profiled_pass": {"steps": S, "ms_per_step": ms_prof / S,
                          "how": "eager C-ABI calls with the library's launch events around each kernel"},
        "launch": f"captured CUDA graph of {G} consecutive s4_layer_fwd calls (a status-block memset and {launches_per_step} kernels each: captured calls reset the block), replayed; remainder steps from single-call graphs",
        "roofline": roof,
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(u_host.nbytes),
                "d2h_bytes_per_step": int(Bsz * H * L * 8), "steps": e2e_steps_done,
                "how": "per step: H2D of u from pinned memory, the layer graph, D2H of y to pinned memory; three streams pipeline consecutive steps"},
    }
    if pool is not None:
        # bounded sample: the sampled channels (every channel of a small
        # workload), each with its kernel and all of its batch rows
        units = channel_units(p, u_host, base_chans, L)
        rate, secs, samples, passes = oracle_rate(pool, procs, units)
        what = ("the whole workload" if len(base_chans) == H else
                f"channels {base_chans} of {H}")
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": procs, "kind": "oracle",
                                "sample": f"{passes} passes over {what}: {len(base_chans)} channels x {Bsz} rows "
                                          f"x L={L} ({samples} channel-samples, {secs:.1f} s wall, ~{secs * procs:.0f} CPU-s)"}
        pool.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


PATHS = {
    # path: (unit of the rate, timing families of the library, dominant family)
    "kernel_gen": ("channel-roots/s", ["moments", "cauchy", "ifft"], "cauchy"),
    "conv": ("channel-samples/s", ["spec_fwd", "spectrum", "conv", "conv_fwd", "conv_col", "conv_inv"], "conv"),
    "conv_real": ("channel-samples/s", ["spectrum", "conv_real"], "conv_real"),
    "recurrent": ("channel-samples/s", ["recurrent", "bordered"], "recurrent"),
    "ctilde": ("channel-steps/s", ["ctilde", "bordered"], "ctilde"),
}


def _oracle_path_unit(args):
    """Oracle work of one unit of an auxiliary path (see run_path)."""
    path, h, b = args
    import numpy as np
    import oracle.s4_oracle as O
    from structured_state_space_gb300 import workloads as W
    w = W.WORKLOADS[WORKLOAD_INDEX]
    p, u = _oracle_data()
    if path in ("conv", "conv_real"):
        K = _path_kernel(w)[h].astype(np.complex128)
        O.causal_conv(K.real if path == "conv_real" else K, u[b, h], p["D"][h])
        return w.L
    if path == "kernel_gen":
        O.s4_kernel(p["Lambda"][h], p["P"][h], p["Q"][h], p["B"][h], p["Ctilde"][h], p["dt"][h], w.L)
        return w.M
    _, Abar, Bbar = O.bilinear(p["Lambda"][h], p["P"][h], p["Q"][h], p["B"][h], p["dt"][h])
    if path == "recurrent":
        O.recurrence(Abar, Bbar, p["Ctilde"][h], p["D"][h], u[b, h])
        return w.L
    O.ctilde_from_c(Abar, p["Ctilde"][h], w.M)
    return w.M


_PATH_K = None


def _path_kernel(w):
    """Seeded complex kernel [H][L] (complex64) fed to the convolution paths by
    both the GPU run and its CPU baseline (made once per process)."""
    global _PATH_K
    if _PATH_K is None:
        import numpy as np
        rng = np.random.default_rng(7000 + w.L)
        _PATH_K = ((rng.standard_normal((w.H, w.L)) + 1j * rng.standard_normal((w.H, w.L))) * 0.05).astype(np.complex64)
    return _PATH_K


def run_path(args):
    """One of the entry points beside the layer, timed like the layer: conv
    (s4_conv_fwd with a given kernel), conv_real (s4_conv_fwd_real), recurrent
    (s4_recurrent_fwd over the L steps of every row, state carried from call
    to call) or ctilde (s4_ctilde).  A step is one call over the whole workload."""
    import numpy as np
    import torch

    import structured_state_space_gb300 as s4
    from structured_state_space_gb300 import build as s4build
    from structured_state_space_gb300 import workloads as W

    unit, families, dom = PATHS[args.path]
    pool, procs = None, 0
    if not args.no_cpu_baseline:
        procs = max(1, os.cpu_count() or 1)
        pool = make_pool(procs)
    torch.cuda.set_device(0)
    s4build.build()
    s4.load()
    w = W.WORKLOADS[WORKLOAD_INDEX]
    H, N, r, L, Bsz, M = w.H, w.N, w.r, w.L, w.batch, w.M
    p = W.make_params(w)
    u_host = W.make_u(w, p)
    dev = torch.device("cuda", 0)
    prm = {k: torch.from_numpy(np.ascontiguousarray(p[k])).to(dev) for k in ["Lambda", "P", "Q", "B", "Ctilde", "dt", "D"]}
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    stream = torch.cuda.Stream(dev)
    ws = s4.workspace(H, N, r, L, Bsz, dev)
    if args.path == "ctilde":
        set_bytes = H * N * 8 * 2
        in_host, out_shape, out_dtype = None, (H, N), torch.complex64
    elif args.path == "kernel_gen":
        set_bytes = H * L * 8
        in_host, out_shape, out_dtype = None, (H, L), torch.complex64
    else:
        out_dtype = torch.float32 if args.path == "conv_real" else torch.complex64
        set_bytes = Bsz * H * L * (4 + (4 if args.path == "conv_real" else 8))
        in_host, out_shape = u_host, (Bsz, H, L)
    nsets = min(16, max(3, math.ceil(2 * l2 / set_bytes) + 1))
    ins = [torch.from_numpy(in_host).to(dev) for _ in range(nsets)] if in_host is not None else [None] * nsets
    outs = [torch.empty(out_shape, dtype=out_dtype, device=dev) for _ in range(nsets)]
    Kd = torch.from_numpy(_path_kernel(w)).to(dev) if args.path in ("conv", "conv_real") else None
    xs = torch.zeros((Bsz, H, N), dtype=torch.complex64, device=dev)

    def call(i):
        j = i % nsets
        if args.path == "kernel_gen":
            s4.s4_kernel_gen(prm["Lambda"], prm["P"], prm["Q"], prm["B"], prm["Ctilde"], prm["dt"], L, K=outs[j], ws=ws)
        elif args.path == "conv":
            s4.s4_conv_fwd(ins[j], Kd, prm["D"], y=outs[j], ws=ws)
        elif args.path == "conv_real":
            s4.s4_conv_fwd_real(ins[j], Kd, prm["D"], y=outs[j], ws=ws)
        elif args.path == "recurrent":
            s4.s4_recurrent_fwd(prm["Lambda"], prm["P"], prm["Q"], prm["B"], prm["Ctilde"], prm["dt"], prm["D"],
                                ins[j], x=xs, y=outs[j], ws=ws)
        else:
            s4.s4_ctilde(prm["Lambda"], prm["P"], prm["Q"], prm["dt"], prm["Ctilde"], L, Ctilde=outs[j], ws=ws)

    with torch.cuda.stream(stream):
        for i in range(3):
            call(i)
    stream.synchronize()
    if s4.s4_get_status(ws, stream) != 0:
        raise RuntimeError("device status after warm-up")
    G = nsets * 2
    gbig = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gbig, stream=stream):
        for i in range(G):
            call(i)

    def timed(body, k):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        body(k)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def replay(k):  # k rounded up to whole graphs
        with torch.cuda.stream(stream):
            for _ in range(max(1, -(-k // G))):
                gbig.replay()

    K = max(G, -(-args.steps // G) * G)
    sampler = ClockSampler(0)
    sampler.start()
    replay(max(args.warmup, G))
    ms_total = timed(replay, K)
    clocks = sampler.stop()
    # per-kernel event times over S eager calls behind a graph head start
    S = max(1, min(K, 200))
    s4.timing.reset()
    s4.timing.enable(True)
    with torch.cuda.stream(stream):
        for i in range(S):
            call(i)
    torch.cuda.synchronize()
    s4.timing.reset()

    def prof(k):
        with torch.cuda.stream(stream):
            gbig.replay()
            for i in range(k):
                call(i)

    timed(prof, S)
    s4.timing.enable(False)
    raw = {}
    for name in families:
        n, t = s4.timing.read(name)
        raw[name] = {"launches": n, "avg_us": 1e3 * t / max(n, 1)}
    s4.timing.reset()
    launches_per_call = int(round(sum(v["launches"] for v in raw.values()) / S))
    # long rows: the convolution's three launches count as one part, the
    # spectrum's two likewise (per-call time = the sum)
    groups = {"conv": ["conv", "conv_fwd", "conv_col", "conv_inv"], "spectrum": ["spectrum", "spec_fwd"],
              "cauchy": ["cauchy", "moments"]}
    kern = {}
    for name in families:
        g = next((k for k, v in groups.items() if name in v), name)
        if g in kern or not (raw[name]["launches"] or name == g):
            continue
        used = [k for k in groups.get(g, [g]) if k in raw and raw[k]["launches"]] or [name]
        kern[g] = {"launches": max(raw[k]["launches"] for k in used),
                   "avg_us": sum(raw[k]["avg_us"] * raw[k]["launches"] / S for k in used)}
        if len(used) > 1:
            kern[g]["parts"] = {k: raw[k] for k in used}
    per_call = H * M if args.path in ("ctilde", "kernel_gen") else Bsz * H * L
    value = per_call * K / (ms_total / 1e3)
    peaks, peak_src = read_peaks()
    sms = props.multi_processor_count
    fp32_peak = sms * FP32_LANES_PER_SM * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    peak_source = f"{sms} SMs (queried) x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x max SM clock"
    if args.path in ("conv", "conv_real"):
        yb = 4 if args.path == "conv_real" else 8
        byts = Bsz * H * L * (4 + yb) + H * 2 * M * 8
        ach = byts / (kern[dom]["avg_us"] * 1e-6) / 1e9
        roof = {"kernel": "conv_real_pair_kernel" if args.path == "conv_real" else "conv_pair_kernel", "bound": "hbm",
                "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                "traffic": None,
                "algorithmic": f"u 4 B + y {yb} B per channel-sample, kernel spectrum 16 B per channel-root once"}
    elif args.path == "kernel_gen":
        flops = H * M * N * cauchy_flop(r)
        ach = flops / (kern[dom]["avg_us"] * 1e-6) / 1e12
        roof = {"kernel": "cauchy_kernel", "bound": "alu", "achieved": ach, "peak": fp32_peak, "unit": "TFLOP/s",
                "frac": ach / fp32_peak, "traffic": None,
                "algorithmic": f"{cauchy_flop(r)} flop per (channel, root, pole)",
                "peak_source": peak_source}
    else:
        steps = Bsz * H * L if args.path == "recurrent" else H * M
        flops = steps * N * (20 + 16 * r)
        ach = flops / (kern[dom]["avg_us"] * 1e-6) / 1e12
        roof = {"kernel": f"{dom}_kernel", "bound": "alu", "achieved": ach, "peak": fp32_peak, "unit": "TFLOP/s",
                "frac": ach / fp32_peak, "traffic": None,
                "algorithmic": f"{20 + 16 * r} flop per (row or channel, step, state element)",
                "peak_source": peak_source}
    roof["peak_kind"] = f"of {peak_src}"
    # end to end: input from pinned host memory, the call, output back, one stream
    e2e = None
    if in_host is not None:
        in_pin = torch.from_numpy(in_host).pin_memory()
        out_pin = torch.empty(out_shape, dtype=out_dtype).pin_memory()

        def e2e_steps(k):
            with torch.cuda.stream(stream):
                for i in range(k):
                    ins[i % nsets].copy_(in_pin, non_blocking=True)
                    call(i)
                    out_pin.copy_(outs[i % nsets], non_blocking=True)

        n_e2e = max(3, min(K, 200))
        e2e_steps(3)
        ms_e2e = timed(e2e_steps, n_e2e)
        e2e = {"value": per_call * n_e2e / (ms_e2e / 1e3), "unit": unit, "h2d_bytes_per_step": int(in_pin.numel() * 4),
               "d2h_bytes_per_step": int(out_pin.numel() * out_pin.element_size()), "steps": n_e2e,
               "how": "per step on one stream: H2D of u from pinned memory, the call, D2H of the output"}
    line = {"metric": f"S4 {args.path} {unit}", "path": args.path, "value": value, "unit": unit, "n_gpus": 1,
            "steps": K, "warmup": max(args.warmup, G), "ms_per_step": ms_total / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": {"workload": w.name, "N": N, "r": r, "H": H, "L": L, "M": M, "batch": Bsz},
            "gpu_launches": launches_per_call * K,
            "kernels": kern, "roofline": roof, "clocks": clocks, "e2e": e2e}
    if pool is not None:
        if args.path in ("ctilde", "kernel_gen"):
            units = [(args.path, h, 0) for h in range(H)]
            what = f"{len(units)} channels x M={M} " + ("steps" if args.path == "ctilde" else "roots")
        else:
            units = [(args.path, h, b) for h in range(H) for b in range(Bsz)]
            what = f"{len(units)} rows x L={L}"
        done, secs, passes = timed_passes(pool, procs, _oracle_path_unit, units)
        line["cpu_baseline"] = {"value": done / secs, "unit": unit, "cores": procs, "kind": "oracle",
                                "sample": f"{passes} passes over {what} ({done} units, {secs:.1f} s wall, "
                                          f"~{secs * procs:.0f} CPU-s)"}
        pool.close()
    print(json.dumps(line), flush=True)


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    from structured_state_space_gb300 import workloads as W
    w = W.WORKLOADS[WORKLOAD_INDEX]
    procs = max(1, min(os.cpu_count() or 1, w.H))
    pool = make_pool(procs)
    p = W.make_params(w)
    u = W.make_u(w, p)

    # one step = one channel per worker process (its kernel and every batch
    # row), channels taken in turn through the workload
    def step(i):
        chans = [((i * procs) + j) % w.H for j in range(procs)]
        return sum(pool.map(_oracle_channel, channel_units(p, u, chans, w.L)))
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    samples = 0
    for i in range(args.steps):
        samples += step(args.warmup + i)
    secs = time.perf_counter() - t0
    pool.close()
    value = samples / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": w.name, "N": w.N, "r": w.r, "H": w.H, "L": w.L, "M": w.M, "batch": w.batch},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": procs, "kind": "oracle",
                         "sample": f"per step {procs} channels (taken in turn) x {w.batch} rows x L={w.L}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=["layer"] + sorted(PATHS), default="layer",
                    help="layer (the bench line) or a step either side of it")
    ap.add_argument("--channels", type=int, default=None,
                    help="layer only: run the workload with this many channels instead (a smaller copy "
                         "for ncu captures; its line is not a bench line)")
    ap.add_argument("--workload", type=int, default=None,
                    help=f"seeded workload index (default {LAYER_WORKLOAD} for the layer and the reference arm, "
                         f"{PATH_WORKLOAD} for --path)")
    args = ap.parse_args()
    global WORKLOAD_INDEX
    if args.workload is None:
        args.workload = PATH_WORKLOAD if args.path != "layer" and args.impl != "reference" else LAYER_WORKLOAD
    WORKLOAD_INDEX = args.workload
    os.environ["S4_BENCH_WORKLOAD"] = str(args.workload)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.path != "layer":
        run_path(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
