#!/usr/bin/env python3
"""Benchmark: S6 selective-scan forward + backward on one GB300 (per rank).

A step is one pass of the whole training hot path on one batch of the
Mamba-1.4B-shaped workload (B=4, L=4096, d_inner=4096, N=16, bf16 activations,
f32 parameters and state): ssm_scan_fwd (with chunk-state saves) followed by
ssm_scan_bwd (backward scan + fixed-order reductions), all through the C ABI.

Printed (rank 0, one JSON line): the metric in G(B*L*D*N)/s over fwd+bwd,
device-timed with CUDA events on the launching stream (inputs resident in
HBM, larger than L2), the same metric end to end from pinned host buffers
(e2e), the HBM roofline of the dominant kernel, and the oracle timed on the
host cores on a bounded sample (cpu_baseline).

--impl reference times the oracle (plain f64 C, all host cores) instead, on
a bounded sample of the same workload, and prints the same kind of line.

Multi-GPU (torchrun, N > 1): every rank runs an independent replica on its
own batch (weak scaling, no collective on the data path); the step time is
the max over ranks and value = all ranks' cells / that time.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from selective_state_space_s6_gb300 import inputs  # noqa: E402

WORKLOAD = "mamba1p4b"
METRIC = "fwd+bwd selective-scan G(B*L*D*N)/s"
UNIT = "G(B*L*D*N)/s"
ARGS = ("u", "delta_raw", "z", "Bm", "Cm", "A_log", "Dp", "delta_bias")
# FP32 pipe: 152 SMs x 128 lanes x 2 flops (FMA) x 2.07 GHz (maximum SM clock)
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
# Algorithmic f32 flops per cell (b, t, d, n) of the method as the oracle
# computes it (FMA = 2, exp on the special-function unit not counted):
#   fwd: delta*A, (delta*u)*B, h = Abar*h + b, y += C*h                      -> 6
#   bwd: the forward recurrence again (4) + g = dy*C + carry (2), a*g (1),
#        (a*g)*h_prev (1), sum_n A*p (2), sum_t delta*p (2), sum_n g*B (2),
#        sum_n C*h (2), dBm term g*delta*u and its sum over d (2), dCm term
#        dy*h and its sum over d (2)                                          -> 20
FLOPS_PER_CELL = {"fwd": 6, "bwd": 20}


def launches_per_step(fwd_segments, bwd_segments):
    """Kernels one step launches: the forward scan (or segment aggregates,
    carries and the segmented scan), the backward scan (likewise), then the
    two fixed-order reduction kernels of the finalize."""
    return (1 if fwd_segments == 1 else 3) + (1 if bwd_segments == 1 else 3) + 2


def load_peaks(key="hbm_gbs"):
    """A measured peak from MEASURED_PEAKS.json (HBM copy GB/s by default, or
    bf16_tflops), else the fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk[key]), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}[key], "fallback"


# The method's own checkpoint spacing for the algorithmic byte count: one
# saved state per 256 steps (the chunked scan's chunk).  The kernels save one
# state per chunk_len steps; the extra states are counted as overhead, not as
# algorithmic bytes.
ALGO_STATE_SPACING = 256


def algorithmic_bytes(B, L, D, N, e, chunk=ALGO_STATE_SPACING):
    """Bytes each kernel must move at minimum (inputs read once, outputs written once).

    fwd: u, delta_raw, z read + out write (4*BLD*e); Bm, Cm read (2*BLN*e);
         chunk states written (4*B*nc*D*N); A_log, Dp, delta_bias read.
    bwd: u, delta_raw, z, dout read + du, d_delta_raw, dz write (7*BLD*e);
         Bm, Cm read + dBm, dCm written (4*BLN*e); chunk states read;
         A_log, Dp, delta_bias read + dA_log, dDp, d_delta_bias written.
    nc = ceil(L / chunk) states per sequence.
    """
    nc = -(-L // chunk)
    bld, bln = B * L * D, B * L * N
    params = 4 * (D * N + 2 * D)
    fwd = 4 * bld * e + 2 * bln * e + 4 * B * nc * D * N + params
    bwd = 7 * bld * e + 4 * bln * e + 4 * B * nc * D * N + 2 * params
    return fwd, bwd


def time_step(dev, reps=50, rounds=5):
    """The decode step (ssm_step) on the decode workload's shape (B=256,
    D=1536, N=16, f32), each step on a cold L2: CUDA graphs of `reps` x
    (256 MB read + step) and of `reps` x (256 MB read) are replayed and the
    step time is their difference (a read leaves L2 full of clean lines, so
    the step pays for its own misses and no write-backs).  Also the
    L2-resident time (graph of chained steps only; h is 25 MB, smaller than
    L2)."""
    from selective_state_space_s6_gb300 import s6

    w = inputs.WORKLOADS["decode"]
    B, D, N = w.batch, w.dim, w.dstate
    e = 2 if w.act == "bf16" else 4
    x = inputs.make_inputs(B, 1, D, N, w.act, seed=0, h0_std=0.5)
    x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    sl = {k: x[k][:, 0].contiguous() for k in ("u", "delta_raw", "z", "Bm", "Cm")}
    h = x["h0"].clone()
    out = torch.empty_like(sl["u"])
    scratch = torch.ones((256 << 20) // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def step():
        s6.ssm_step(sl["u"], sl["delta_raw"], sl["z"], sl["Bm"], sl["Cm"], x["A_log"], x["Dp"],
                    x["delta_bias"], h, out=out)

    def flush():
        torch.sum(scratch, dim=0, out=sink)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(3):
            flush()
            step()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)

    def capture(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                body()
        return g

    g_fs = capture(lambda: (flush(), step()))
    g_f = capture(flush)
    g_s = capture(step)

    def replay_ms(g):
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(rounds):
            g.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / (rounds * reps)

    t_fs, t_f, t_s = replay_ms(g_fs), replay_ms(g_f), replay_ms(g_s)
    us_cold = (t_fs - t_f) * 1e3
    nbytes = B * D * N * 4 * 2 + 4 * B * D * e + 2 * B * N * e + D * N * 4 + 2 * D * 4
    peak, kind = load_peaks()
    gbs = nbytes / (us_cold * 1e-6) / 1e9
    return {"workload": f"decode: {w.description}", "us_per_step": round(us_cold, 2),
            "us_per_step_l2_resident": round(t_s * 1e3, 2), "algorithmic_bytes": nbytes,
            "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peak, 4),
            "timing": f"CUDA graphs of {reps} steps; cold L2 = (read 256 MB + step) - (read 256 MB)"}


def time_conv1d(dev, B, L, D, act, K=4, reps=10):
    """The causal conv1d + SiLU in front of the scan, on the workload's [B,L,D]
    shape (K = 4 taps), forward and backward, CUDA events over `reps` calls;
    inputs are larger than L2.  HBM roofline: x read + out written (forward);
    x, dout read + dx written (backward)."""
    from selective_state_space_s6_gb300 import s6

    g = torch.Generator().manual_seed(0)
    dt = torch.bfloat16 if act == "bf16" else torch.float32
    e = 2 if act == "bf16" else 4
    x = torch.randn(B, L, D, generator=g).to(dt).to(dev)
    dout = torch.randn(B, L, D, generator=g).to(dt).to(dev)
    w = (torch.randn(D, K, generator=g) * 0.5).to(dev)
    bias = (torch.randn(D, generator=g) * 0.2).to(dev)
    s0 = torch.zeros(B, D, K - 1, dtype=dt, device=dev)
    out = torch.empty_like(x)
    s_last = torch.empty_like(s0)
    ws = torch.empty((s6.conv1d_bwd_workspace_bytes(B, L, D, K, s6.SSM_BF16 if act == "bf16" else s6.SSM_F32) + 256,),
                     dtype=torch.uint8, device=dev)

    def fwd():
        s6.conv1d_fwd(x, w, bias, s0, out=out, state_last=s_last)

    def bwd():
        s6.conv1d_bwd(x, w, bias, s0, dout, ws=ws)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    peak, _ = load_peaks()
    bld = B * L * D
    res = {"workload": f"B={B} L={L} D={D} K={K} {act}", "timing": f"CUDA events over {reps} calls"}
    for name, fn, nbytes in (("fwd", fwd, 2 * bld * e), ("bwd", bwd, 3 * bld * e)):
        ms = timed(fn)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": round(ms, 4), "algorithmic_bytes": nbytes, "hbm_gbs": round(gbs, 1),
                     "hbm_frac": round(gbs / peak, 4)}
    return res


def ssd_algorithmic(w):
    """Algorithmic bytes and tensor flops of one SSD forward: x, dt, Bm, Cm read
    and y written once, the final state written once; per (b, t, h) the four
    chunk products at 64-step chunks: C B^T (2 Q N), its product with delta x
    (2 Q P), C S_in (2 N P) and the state update B^T x' (2 N P)."""
    B, L, H, P, G, N = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate
    e = 2 if w.act == "bf16" else 4
    nbytes = 2 * B * L * H * P * e + 2 * B * L * G * N * e + B * L * H * e + B * H * N * P * 4
    flops = B * L * H * (2 * 64 * N + 2 * 64 * P + 4 * N * P)
    return nbytes, flops


def ssd_bwd_algorithmic(w):
    """Algorithmic bytes and tensor flops of one SSD backward: x, dy, dt, Bm,
    Cm and the saved chunk states (bf16, one per 64 steps) read, dx, ddt_raw,
    dBm, dCm written once; per 64-step chunk the ten products G = C B^T,
    Z = dy x^T, dx's (L o G)^T dy, dB's (L o Z)^T C and dC's (L o Z) B
    (2 Q^2 N or 2 Q^2 P each) and C S_in, B dS, the state-gradient update,
    x'' dS^T, dy' S_in^T (2 Q N P each)."""
    B, L, H, P, G, N = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate
    e = 2 if w.act == "bf16" else 4
    nch = -(-L // 64)
    nbytes = 3 * B * L * H * P * e + 4 * B * L * G * N * e + 2 * B * L * H * e + B * H * nch * N * P * 2
    flops = B * L * H * (2 * 64 * (3 * N + 2 * P) + 10 * N * P)
    return nbytes, flops


def time_ssd(dev, reps=10, workload="mamba2_1p3b", with_wide=True):
    """The Mamba-2 SSD forward (plain and with state saves) and backward on the
    1.3B block's shape, CUDA events over `reps` calls each (inputs larger than
    L2); and (`wide`) the same on the same width in heads of 128 columns."""
    from selective_state_space_s6_gb300 import s6

    w = inputs.SSD_WORKLOADS[workload]
    x = inputs.make_ssd_inputs(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.act, seed=0)
    xd = {k: (v.to(dev) if v is not None else None) for k, v in x.items()}
    gen = torch.Generator(device=dev).manual_seed(1)
    dy = torch.randn(xd["x"].shape, device=dev, generator=gen).to(torch.bfloat16)
    keys = ("x", "dt_raw", "dt_bias", "A_log", "Bm", "Cm", "Dp")
    y = torch.empty_like(xd["x"])
    hl = torch.empty((w.batch, w.nheads, w.dstate, w.headdim), dtype=torch.float32, device=dev)
    _, _, cs = s6.ssd_fwd(*[xd[k] for k in keys], None, save=True)
    grads = s6.ssd_bwd(*[xd[k] for k in keys], cs, dy, None, want_dh0=False)
    ws = torch.empty((s6.ssd_bwd_workspace_bytes(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate)
                      + 256,), dtype=torch.uint8, device=dev)

    def fwd():
        s6.ssd_fwd(*[xd[k] for k in keys], None, y=y, h_last=hl)

    def fwd_save():
        s6.ssd_fwd(*[xd[k] for k in keys], None, y=y, h_last=hl, save=True, chunk_states=cs)

    def bwd():
        s6.ssd_bwd(*[xd[k] for k in keys], cs, dy, None, want_dh0=False, ws=ws, grads=grads)

    def timed(run):
        for _ in range(3):
            run()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            run()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    peak, _ = load_peaks()
    tpeak = load_peaks("bf16_tflops")[0]

    def line(ms, nbytes, flops):
        gbs = nbytes / (ms * 1e-3) / 1e9
        tfl = flops / (ms * 1e-3) / 1e12
        return {"ms": round(ms, 4), "gcells_s": round(w.cells / (ms * 1e-3) / 1e9, 1), "algorithmic_bytes": nbytes,
                "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peak, 4), "algorithmic_flops": flops,
                "tensor_tflops": round(tfl, 1), "tensor_frac": round(tfl / tpeak, 4)}

    fb, ff = ssd_algorithmic(w)
    bb, bf = ssd_bwd_algorithmic(w)
    res = line(timed(fwd), fb, ff)
    res.update({"workload": w.description,
                "fwd_save": line(timed(fwd_save), fb + w.batch * w.nheads * (-(-w.seqlen // 64)) * w.dstate
                                 * w.headdim * 2, ff),
                "bwd": line(timed(bwd), bb, bf),
                "peaks": "measured hbm_gbs (copy) and bf16_tflops (cuBLAS, burst)",
                "timing": f"CUDA events over {reps} calls each"})
    if with_wide:
        wide = time_ssd(dev, reps, "mamba2_1p3b_p128", with_wide=False)
        res["wide"] = {"workload": wide["workload"], "fwd": {k: wide[k] for k in ("ms", "tensor_frac", "hbm_frac")},
                       "bwd": {k: wide["bwd"][k] for k in ("ms", "tensor_frac", "hbm_frac")}}
    return res


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Samples nvidia-smi clocks/throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle (CPU baseline)

def oracle_sample(w, cells_target, rank=0, threads=None):
    """A bounded sample of the workload for the oracle, about ``cells_target``
    cells: whole sequences first, then more channels, then more batch rows
    (the full workload if that is smaller); same distributions as the full
    workload."""
    import oracle
    threads = threads or oracle.default_threads()
    B, L, D, N = w.batch, w.seqlen, w.dim, w.dstate
    ch0 = min(D, 64 * threads)  # at least one 64-channel block per thread
    nl = max(1, min(L, cells_target // (ch0 * N)))
    nd = max(ch0, min(D, cells_target // (nl * N)))
    nb = max(1, min(B, cells_target // (nl * nd * N)))
    x = inputs.make_inputs(nb, nl, nd, N, w.act, seed=rank, delta_lo=w.delta_lo, delta_hi=w.delta_hi)
    x64 = {k: (oracle._f64(v) if v is not None else None) for k, v in x.items()}
    cells = nb * nl * nd * N
    desc = (f"batch rows 0..{nb - 1} of {B}, channels 0..{nd - 1} of {D}, "
            f"steps 0..{nl - 1} of {L}")
    return x64, cells, desc, threads


def oracle_step(x64, threads):
    import oracle
    oracle.fwd(*[x64[k] for k in ARGS], None, threads=threads)
    oracle.bwd(*[x64[k] for k in ARGS], None, x64["dout"], None, threads=threads)


def time_oracle(w, steps, warmup, target_s, rank=0, min_total_s=0.0):
    """Oracle fwd+bwd throughput on a sample sized so that one step takes about
    ``target_s`` seconds (calibrated on a small sample first); with
    ``min_total_s``, enough steps are timed to cover at least that much work."""
    x64, cells, _, threads = oracle_sample(w, 64 * 128 * w.dstate * 16, rank)
    t0 = time.perf_counter()
    oracle_step(x64, threads)
    per_cell = (time.perf_counter() - t0) / cells
    x64, cells, desc, threads = oracle_sample(w, int(target_s / max(per_cell, 1e-15)), rank, threads)
    for _ in range(warmup):
        oracle_step(x64, threads)
    est = cells * per_cell
    steps = max(steps, int(-(-min_total_s // max(est, 1e-9))))
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(x64, threads)
    dt = (time.perf_counter() - t0) / max(steps, 1)
    return cells / dt / 1e9, desc, threads, dt, steps


# ------------------------------------------------------------------ our arm

def run_ours(args, world, rank, local):
    from selective_state_space_s6_gb300 import s6

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = inputs.WORKLOADS[args.workload]
    B, L, D, N = w.batch, w.seqlen, w.dim, w.dstate
    e = 2 if w.act == "bf16" else 4
    act = s6.SSM_BF16 if w.act == "bf16" else s6.SSM_F32
    x_cpu = inputs.make_workload(args.workload, seed=rank)
    x = {k: (v.to(dev) if v is not None else None) for k, v in x_cpu.items()}
    stream = torch.cuda.current_stream(dev)

    out = torch.empty_like(x["u"])
    h_last = torch.empty((B, D, N), dtype=torch.float32, device=dev)
    cs = torch.empty((B, s6.num_chunks(L), D, N), dtype=torch.float32, device=dev)
    g = {"du": torch.empty_like(x["u"]), "d_delta_raw": torch.empty_like(x["u"]),
         "dz": torch.empty_like(x["u"]), "dBm": torch.empty_like(x["Bm"]),
         "dCm": torch.empty_like(x["Cm"]), "dA_log": torch.empty_like(x["A_log"]),
         "dD": torch.empty_like(x["Dp"]), "d_delta_bias": torch.empty_like(x["delta_bias"]),
         "dh0": None}
    ws_bytes = max(s6.bwd_workspace_bytes(B, L, D, N, act), s6.fwd_workspace_bytes(B, L, D, N, act))
    ws = torch.empty((ws_bytes + 256,), dtype=torch.uint8, device=dev)

    def fwd():
        s6.ssm_scan_fwd(*[x[k] for k in ARGS], None, out=out, h_last=h_last, chunk_states=cs,
                        ws=ws, stream=stream)

    def bwd_partials():
        s6.bwd_partials(*[x[k] for k in ARGS], cs, x["dout"], None, g, ws, stream)

    def bwd_finalize():
        s6.bwd_finalize(B, L, D, N, act, g, ws, stream)

    fallbacks0 = s6.plan_fallbacks()
    for _ in range(args.warmup):
        fwd(); bwd_partials(); bwd_finalize()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    barrier(world)
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(K):
        ev[k][0].record(stream)
        fwd()
        ev[k][1].record(stream)
        bwd_partials()
        ev[k][2].record(stream)
        bwd_finalize()
        ev[k][3].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    total_ms = start.elapsed_time(end)
    clk = clocks.stop()
    t_fwd = sum(ev[k][0].elapsed_time(ev[k][1]) for k in range(K)) / K
    t_bwd = sum(ev[k][1].elapsed_time(ev[k][2]) for k in range(K)) / K
    t_fin = sum(ev[k][2].elapsed_time(ev[k][3]) for k in range(K)) / K

    ms_step = max_over_ranks(total_ms / K, world)
    cells = w.cells
    value = world * cells / (ms_step * 1e-3) / 1e9

    fallbacks_timed = s6.plan_fallbacks() - fallbacks0
    # ---- e2e: pinned host inputs -> device -> fwd + bwd -> every output back
    # to pinned host memory, every step (out and all gradients: 538 MB per
    # step on the 1.4B shape).  A side figure reads back only the parameter
    # gradients (dA_log, dDp, d_delta_bias: what an optimizer reads), the
    # activation gradients staying on the device.  Serial: one stream, copy
    # in, compute, copy out.  Pipelined: three streams and two device buffer
    # sets, so that the copy-in of step k+1 and the copy-out of step k-1 run
    # on the copy engines while step k computes.
    in_keys = ["u", "delta_raw", "z", "Bm", "Cm", "A_log", "Dp", "delta_bias", "dout"]
    out_keys = ["du", "d_delta_raw", "dz", "dBm", "dCm", "dA_log", "dD", "d_delta_bias"]
    result_keys = ["dA_log", "dD", "d_delta_bias"]
    readback = {"keys": result_keys, "out": False}
    h_in = {k: x_cpu[k].pin_memory() for k in in_keys}

    def host_outputs():
        h = {k: torch.empty(g[k].shape, dtype=g[k].dtype, pin_memory=True) for k in out_keys}
        h["out"] = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        return h

    h_out = [host_outputs(), host_outputs()]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h_full = sum(t.numel() * t.element_size() for t in h_out[0].values())
    d2h = sum(h_out[0][k].numel() * h_out[0][k].element_size() for k in result_keys)

    def device_set(first):
        if first:
            return {"x": x, "g": g, "out": out, "cs": cs, "ws": ws, "h_last": h_last}
        return {"x": {k: (torch.empty_like(v) if isinstance(v, torch.Tensor) else v) for k, v in x.items()},
                "g": {k: (torch.empty_like(v) if isinstance(v, torch.Tensor) else v) for k, v in g.items()},
                "out": torch.empty_like(out), "cs": torch.empty_like(cs), "ws": torch.empty_like(ws),
                "h_last": torch.empty_like(h_last)}

    sets = [device_set(True), device_set(False)]

    def compute(S, st):
        xs = S["x"]
        s6.ssm_scan_fwd(*[xs[k] for k in ARGS], None, out=S["out"], h_last=S["h_last"],
                        chunk_states=S["cs"], ws=S["ws"], stream=st)
        s6.bwd_partials(*[xs[k] for k in ARGS], S["cs"], xs["dout"], None, S["g"], S["ws"], st)
        s6.bwd_finalize(B, L, D, N, act, S["g"], S["ws"], st)

    def copy_in(S):
        for k in in_keys:
            S["x"][k].copy_(h_in[k], non_blocking=True)

    def copy_out(S, H):
        if readback["out"]:
            H["out"].copy_(S["out"], non_blocking=True)
        for k in readback["keys"]:
            H[k].copy_(S["g"][k], non_blocking=True)

    def serial_step():
        copy_in(sets[0])
        compute(sets[0], stream)
        copy_out(sets[0], h_out[0])

    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def pipelined_step(k):
        i = k % 2
        S = sets[i]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_cmp[i])  # step k-2 has finished reading set i
            copy_in(S)
            ev_in[i].record(s_in)
        s_cmp.wait_event(ev_in[i])
        if k >= 2:
            s_cmp.wait_event(ev_out[i])  # step k-2's results have left set i
        compute(S, s_cmp)
        ev_cmp[i].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[i])
            copy_out(S, h_out[i])
            ev_out[i].record(s_out)

    def timed(run, nsteps, first_stream, last_stream):
        torch.cuda.synchronize(dev)
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(first_stream)
        for k in range(nsteps):
            run(k)
        e1.record(last_stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(e0.elapsed_time(e1) / nsteps, world)

    for k in range(max(2, min(args.warmup, 4))):
        serial_step()
    torch.cuda.synchronize(dev)
    s_in.wait_stream(stream)
    for k in range(max(2, min(args.warmup, 4))):
        pipelined_step(k)
    torch.cuda.synchronize(dev)
    ke = max(2, args.e2e_steps)
    # three runs of each, the median reported: the host link's rate moves
    # between runs (other work on the host's memory), the kernels' does not
    serial_runs, e2e_runs = [], []
    for _ in range(3):
        serial_runs.append(timed(lambda k: serial_step(), ke, stream, stream))
        s_in.wait_stream(stream)
        e2e_runs.append(timed(pipelined_step, ke, s_in, s_out))
    serial_ms = sorted(serial_runs)[1]
    e2e_ms = sorted(e2e_runs)[1]
    e2e_value = world * cells / (e2e_ms * 1e-3) / 1e9
    serial_value = world * cells / (serial_ms * 1e-3) / 1e9
    # every output read back
    readback.update(keys=out_keys, out=True)
    full_runs = []
    for _ in range(3):
        s_in.wait_stream(stream)
        full_runs.append(timed(pipelined_step, ke, s_in, s_out))
    full_ms = sorted(full_runs)[1]
    # the host link alone: the same copies with no compute, each direction by
    # itself and both at once (the floor under the pipelined e2e step)
    in_ms = timed(lambda k: copy_in(sets[k % 2]), ke, stream, stream)
    out_ms = timed(lambda k: copy_out(sets[k % 2], h_out[k % 2]), ke, stream, stream)

    def both(k):
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        with torch.cuda.stream(s_in):
            copy_in(sets[k % 2])
        with torch.cuda.stream(s_out):
            copy_out(sets[(k + 1) % 2], h_out[k % 2])
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    both_ms = timed(both, ke, stream, stream)
    torch.cuda.synchronize(dev)
    link = {"h2d_gbs": round(h2d / (in_ms * 1e-3) / 1e9, 1), "d2h_gbs": round(d2h_full / (out_ms * 1e-3) / 1e9, 1),
            "both_ms_per_step": round(both_ms, 4),
            "note": "pinned-host copies of one step's inputs and of every output alone, no compute"}

    # ---- roofline of the dominant kernel (the backward scan), live event timing.
    # The metric is achieved HBM bandwidth against the measured copy peak:
    # algorithmic bytes (states counted at one per 256 steps) / event time.
    # The scans are in fact bound by instruction issue on the FP32 pipe; the
    # FP32 fraction (algorithmic flops / event time / derived peak) is given
    # beside it.
    peak, peak_kind = load_peaks()
    fwd_bytes, bwd_bytes = algorithmic_bytes(B, L, D, N, e)
    kern = {
        "s6_fwd": {"ms": t_fwd, "bytes": fwd_bytes, "flops": FLOPS_PER_CELL["fwd"] * cells},
        "s6_bwd": {"ms": t_bwd, "bytes": bwd_bytes, "flops": FLOPS_PER_CELL["bwd"] * cells},
    }
    dom = max(kern, key=lambda k: kern[k]["ms"])
    secs = kern[dom]["ms"] * 1e-3
    tflops = kern[dom]["flops"] / secs / 1e12
    gbs_dom = kern[dom]["bytes"] / secs / 1e9
    roofline = {"bound": "hbm", "kernel": dom + " (all of its launches in the step)",
                "achieved": round(gbs_dom, 1), "peak": peak, "unit": "GB/s",
                "frac": round(gbs_dom / peak, 4), "traffic": load_traffic(dom),
                "peak_source": f"{peak_kind} hbm_gbs (copy)",
                "algorithmic_bytes_per_launch": kern[dom]["bytes"],
                "bytes_formula": ("bwd: 7*B*L*D*e + 4*B*L*N*e + 4*B*ceil(L/256)*D*N + 2*params; "
                                  "fwd: 4*B*L*D*e + 2*B*L*N*e + 4*B*ceil(L/256)*D*N + params "
                                  f"(e = {e} bytes; the kernels save a state every {s6.CHUNK_LEN} steps, "
                                  "the extra states are overhead)"),
                "fp32": {"achieved": round(tflops, 2), "peak": round(FP32_PEAK_TFLOPS, 2), "unit": "TFLOP/s",
                         "frac": round(tflops / FP32_PEAK_TFLOPS, 4),
                         "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 (FMA) x 2.07 GHz",
                         "algorithmic_flops_per_launch": kern[dom]["flops"]}}
    per_kernel = {}
    for k in kern:
        s_k = kern[k]["ms"] * 1e-3
        gbs = kern[k]["bytes"] / s_k / 1e9
        per_kernel[k] = {"ms": round(kern[k]["ms"], 4), "gcells_s": round(cells / s_k / 1e9, 1),
                         "tflops": round(kern[k]["flops"] / s_k / 1e12, 2),
                         "fp32_frac": round(kern[k]["flops"] / s_k / 1e12 / FP32_PEAK_TFLOPS, 4),
                         "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peak, 4)}
    per_kernel["s6_bwd_finalize (reduce_dbc + reduce_params)"] = {"ms": round(t_fin, 4)}
    fwd_seg, bwd_seg = s6.plan_segments(B, L, D, N, act)

    step_line = time_step(dev) if not args.no_step else None
    conv_line = time_conv1d(dev, B, L, D, w.act) if not args.no_step else None
    ssd_line = time_ssd(dev) if not args.no_step else None

    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, threads, dt, n = time_oracle(w, steps=1, warmup=0, target_s=15.0, min_total_s=10.0)
        cpu_base = {"value": round(v, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                    "sample": desc + f" ({dt:.1f} s per fwd+bwd, {n} timed)"}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) activations, Mamba dt/A/D initialisation)",
        "config": {"workload": f"{args.workload}: {w.description}", "B": B, "L": L, "D": D,
                   "N": N, "act_dtype": w.act, "state_dtype": "f32",
                   "l2": f"no flush; each step reads {(4 * B * L * D * e) / 1e6:.0f} MB of "
                         f"[B,L,D] inputs, larger than the 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "e2e": {"value": round(world * cells / (full_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h_full,
                "ms_per_step": round(full_ms, 4), "steps": ke,
                "result_read_back": "out and every gradient (du, d_delta_raw, dz, dBm, dCm, dA_log, dDp, "
                                    "d_delta_bias)",
                "overlap": "copy-in of step k+1 and copy-out of step k-1 overlap step k "
                           "(three streams, two device buffer sets)",
                "runs_ms_per_step": [round(v, 4) for v in full_runs], "reported": "median of 3 runs",
                "params_read_back": {"value": round(e2e_value, 2), "ms_per_step": round(e2e_ms, 4),
                                     "d2h_bytes_per_step": d2h,
                                     "runs_ms_per_step": [round(v, 4) for v in e2e_runs],
                                     "note": "only dA_log, dDp, d_delta_bias copied back, pipelined"},
                "serial": {"value": round(serial_value, 2), "ms_per_step": round(serial_ms, 4),
                           "runs_ms_per_step": [round(v, 4) for v in serial_runs],
                           "note": "one stream, parameter gradients read back"},
                "host_link": link},
        "gpu_launches": launches_per_step(fwd_seg, bwd_seg) * K,
        "segments": {"fwd": fwd_seg, "bwd": bwd_seg},
        "plan": {"sms": torch.cuda.get_device_properties(dev).multi_processor_count, "planned_for_sms": 152,
                 "cooperative_fallbacks": fallbacks_timed,
                 "note": ("over the warm-up and timed steps; 0: the forward's stream mode and the backward's hand-over mode ran as planned; "
                          "else that many calls ran their non-cooperative form (same results, slower)")},
        "roofline": roofline,
        "kernels": per_kernel,
        "step": step_line,
        "conv1d": conv_line,
        "ssd": ssd_line,
        "cpu_baseline": cpu_base,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def load_traffic(kernel):
    """dram bytes per launch from the committed ncu summary, if it matches the
    current build of that kernel (else null)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except Exception:
        return None
    ent = t.get(kernel)
    if not ent:
        return None
    try:
        from selective_state_space_s6_gb300 import build as _b
        src = _b.kernel_source_digest(ent.get("sources"))
    except Exception:
        return None
    return ent.get("bytes_per_launch") if ent.get("source_digest") == src else None


# ------------------------------------------------------------------ reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return
    w = inputs.WORKLOADS[args.workload]
    # whole run within a few minutes: about 150 s of oracle work over all steps
    target = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    v, desc, threads, dt, _ = time_oracle(w, steps=args.steps, warmup=args.warmup, target_s=target)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {w.description}", "B": w.batch, "L": w.seqlen,
                   "D": w.dim, "N": w.dstate, "act_dtype": w.act,
                   "sample_per_step": desc},
        "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_kernel(args):
    """One kernel family alone, a few calls on its own workload, for a
    profiler's capture (`--kernel`): the decode step (four calls, each after
    a 256 MB read that empties L2), conv1d + SiLU on the 1.4B block's shape
    (three forward and three backward calls), the SSD forward on the
    Mamba-2-1.3B shape (three calls) or its backward (one saving forward,
    three backward calls).  Prints one JSON line."""
    from selective_state_space_s6_gb300 import s6

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    res = {"kernel": args.kernel}
    if args.kernel == "step":
        w = inputs.WORKLOADS["decode"]
        x = inputs.make_inputs(w.batch, 1, w.dim, w.dstate, w.act, seed=0, h0_std=w.h0_std)
        xd = {k: (v.to(dev) if v is not None else None) for k, v in x.items()}
        a = [xd[k][:, 0].contiguous() if k in ("u", "delta_raw", "z", "Bm", "Cm") else xd[k] for k in ARGS]
        h = xd["h0"].clone()
        scratch = torch.ones((256 << 20) // 4, dtype=torch.float32, device=dev)
        sink = torch.empty((), dtype=torch.float32, device=dev)
        for _ in range(4):
            torch.sum(scratch, dim=0, out=sink)
            s6.ssm_step(*a, h)
        res["workload"] = w.description
    elif args.kernel == "conv1d":
        B, L, D, K = 4, 4096, 4096, 4
        g = torch.Generator(device=dev).manual_seed(0)
        x = torch.randn(B, L, D, device=dev, generator=g).to(torch.bfloat16)
        dout = torch.randn(B, L, D, device=dev, generator=g).to(torch.bfloat16)
        wt = torch.randn(D, K, device=dev, generator=g) * 0.5
        bias = torch.randn(D, device=dev, generator=g) * 0.2
        for _ in range(3):
            s6.conv1d_fwd(x, wt, bias, None, want_state=False)
            s6.conv1d_bwd(x, wt, bias, None, dout, want_dstate0=False)
        res["workload"] = f"B={B} L={L} D={D} K={K} bf16"
        res["path"] = s6.conv1d_path(x, wt)
    elif args.kernel in ("ssd", "ssd_bwd"):
        w = inputs.SSD_WORKLOADS["mamba2_1p3b"]
        x = inputs.make_ssd_inputs(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.act, seed=0)
        xd = {k: (v.to(dev) if v is not None else None) for k, v in x.items()}
        keys = ("x", "dt_raw", "dt_bias", "A_log", "Bm", "Cm", "Dp")
        if args.kernel == "ssd":
            for _ in range(3):
                s6.ssd_fwd(*[xd[k] for k in keys], None)
        else:
            dy = torch.randn(xd["x"].shape, device=dev).to(torch.bfloat16)
            _, _, cs = s6.ssd_fwd(*[xd[k] for k in keys], None, save=True)
            for _ in range(3):
                s6.ssd_bwd(*[xd[k] for k in keys], cs, dy, None, want_dh0=False)
        res["workload"] = w.description
    torch.cuda.synchronize(dev)
    s6.check_device_status()
    print(json.dumps(res), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-step", action="store_true", help="skip the decode-step, conv1d and SSD measurements")
    ap.add_argument("--kernel", choices=["step", "conv1d", "ssd", "ssd_bwd"],
                    help="run only this kernel family a few times (for a profiler) and exit")
    args = ap.parse_args(argv)
    if args.kernel:
        run_kernel(args)
        return
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
