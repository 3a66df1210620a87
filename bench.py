#!/usr/bin/env python
"""Benchmark of the log-linear attention hot path on GB300; prints ONE JSON line.

A step is one pass of the whole hot path on synthetic seeded inputs resident in HBM:
the chunked forward on B1 H16 T16384 dk=dv=128 C64 L15 (bf16 q/k/v/out, fp32 log a and
lambda) followed by one decode step of B128 H16 d128 L15 fp32 states at t = 12345.
``value`` is forward tokens/s (B*T per forward); decode tokens/s is reported beside it.
L2 is flushed (a 512 MiB write) between timed steps, outside the timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs the same per-GPU workload (weak scaling, no collective on
the data path); the max step time over ranks is used and rank 0 prints the line.
``--impl reference`` times the CPU oracle (the only reference this method has) on a
bounded sample of the same forward workload on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "fwd tokens/s at T=16K,H=16,d=128 bf16 + % of roofline; decode tokens/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="target CPU time of the oracle sample")
    p.add_argument("--fwd-only", action="store_true",
                   help="profiling aid: time only the forward (no decode state, no e2e, no "
                        "CPU baseline) and print its own short JSON line")
    p.add_argument("--bwd-only", action="store_true",
                   help="profiling aid: time only the backward, like --fwd-only")
    p.add_argument("--workload", default=None,
                   help="forward workload of --fwd-only / --bwd-only (default: the headline)")
    p.add_argument("--decode-only", choices=["mamba2", "gdn"], default=None,
                   help="profiling aid: time only the decode step (Mamba-2 or Gated DeltaNet) "
                        "on the decode workload, or on --decode-batch rows of it")
    p.add_argument("--decode-batch", type=int, default=None,
                   help="batch of --decode-only (default: the decode workload's 128)")
    p.add_argument("--sweep-t", action="store_true",
                   help="profiling aid: the pages' benchmark shape (B2, 48 heads sharing one "
                        "q/k, d_v 64, d_k 128, C64) over T = 1K..128K: forward, backward and "
                        "training step, one JSON line")
    return p.parse_args()


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return dict(hbm=pk["hbm_gbs"], bf16=pk["bf16_tflops"],
                    bf16_sus=pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def load_traffic(kernel):
    """DRAM bytes per launch (read + write) of `kernel` from the committed ncu record in
    profiles/, or None if there is none or the kernel's source changed since it was taken."""
    import glob
    import hashlib
    for path in glob.glob(os.path.join(ROOT, "profiles", "traffic_*.json")):
        try:
            with open(path) as f:
                rec = json.load(f)
            if rec.get("kernel") != kernel:
                continue
            h = hashlib.sha256()
            for src in rec["source_files"]:
                with open(os.path.join(ROOT, src), "rb") as f:
                    h.update(f.read())
            if h.hexdigest() == rec["source_sha256"]:
                return rec["dram_bytes_read"] + rec["dram_bytes_write"]
        except Exception:
            continue
    return None


# ---------------------------------------------------------------- algorithmic work


def fwd_algorithmic(cfg):
    """Bytes the forward must move (inputs once, output once) and the FLOPs it must do
    (causal half of each chunk's C x C products, per-chunk states, one readout GEMM per
    non-empty inter-chunk level)."""
    e = 2 if cfg.dtype == "bf16" else 4
    BH = cfg.B * cfg.H
    tok = cfg.B * cfg.T * cfg.H
    tok_qk = cfg.B * cfg.T * cfg.qk_heads     # q/k are shared by groups of heads
    bytes_ = tok_qk * 2 * cfg.dk * e + tok * cfg.dv * e + tok * 4 + tok * cfg.L * 4 + tok * cfg.dv * e
    C = cfg.C
    N = cfg.T // C
    intra = C * (C + 1) / 2 * 2 * (cfg.dk + cfg.dv) * N
    states = 2 * C * cfg.dk * cfg.dv * N
    readout = 2 * C * cfg.dk * cfg.dv * sum(bin(j).count("1") for j in range(N))
    flops = BH * (intra + states + readout)
    return bytes_, flops


def bwd_algorithmic(cfg):
    """Bytes and FLOPs of the backward in the chunked form at C = 64: per causal pair
    inside a chunk q.k, dO.v and the dQ, dK, dV updates; per chunk the recomputed chunk
    state; per (chunk, inter level) the dQ readout (dO Tot^T) with its dlambda dot, the
    chunk's part of the mirrored state (q dO^T), and the dK, dV readouts (R v, R^T k).
    Bytes: q, k, v, dO, log a, lambda read once; dq, dk, dv, dlog a, dlambda written once."""
    e = 2 if cfg.dtype == "bf16" else 4
    BH, dk, dv = cfg.B * cfg.H, cfg.dk, cfg.dv
    tok, tok_qk = cfg.B * cfg.T * cfg.H, cfg.B * cfg.T * cfg.qk_heads
    bytes_ = 2 * (tok_qk * 2 * dk * e + tok * 2 * dv * e + tok * 4 + tok * cfg.L * 4)
    C = 64
    N = -(-cfg.T // C)
    pairs = C * (C + 1) / 2 * N
    inter = sum(bin(j).count("1") for j in range(N))
    flops = BH * (pairs * 2 * (3 * dk + 2 * dv) + N * 2 * C * dk * dv
                  + inter * (4 * 2 * C * dk * dv + 2 * C * dk))
    return bytes_, flops


def fp32_alu_peak():
    """FP32 FMA peak: 152 SMs x 128 lanes x 2 FLOPs x 2.07 GHz (maximum SM clock)."""
    return 152 * 128 * 2 * 2.07e9 / 1e12


def decode_levels_written(cfg):
    """Levels the step changes: every level that held data (decayed, merged or cleared)
    and the level lssb(t)+1 that receives the merge."""
    t = cfg.t
    pre = W.nonempty_levels_before(t, cfg.L)
    l = (t & -t).bit_length() - 1
    return len(set(pre) | {l + 1})


def decode_algorithmic(cfg):
    """Bytes of the levels the step must read (non-empty after t-1) and write (every
    level that changes), fp32."""
    lvl_bytes = cfg.dk * cfg.dv * 4
    pre = W.nonempty_levels_before(cfg.t, cfg.L)
    return cfg.B * cfg.H * lvl_bytes * (len(pre) + decode_levels_written(cfg))


# ---------------------------------------------------------------- ranks


def max_over_ranks(values, world, device):
    """Per-rank step times -> their maximum over all ranks (the job is as slow as its
    slowest rank).  One all-reduce of a small tensor; a no-op at world size 1."""
    if world <= 1:
        return list(values)
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world, units_per_rank, seconds):
    """Units all ranks processed (each rank runs the same per-GPU workload: weak
    scaling) divided by the slowest rank's time."""
    return world * units_per_rank / seconds


# ---------------------------------------------------------------- clocks


class NvmlClocks:
    """SM clock, maximum SM clock, power and clock-event reasons of one GPU through NVML
    (ctypes on libnvidia-ml, which the driver installs); the device is found by the UUID
    torch reports for it, so CUDA_VISIBLE_DEVICES does not matter.  Raises if NVML cannot
    be loaded."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index):
        import ctypes
        self.c = ctypes
        self.nv = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
        if not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
        self.h = ctypes.c_void_p()
        if self.nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML device with UUID " + uuid)
        self.reasons_fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        m = ctypes.c_uint()
        self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(m))   # 1: the SM clock
        self.max_mhz = float(m.value)

    def read(self):
        c = self.c
        clk, pw, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, c.byref(clk))
        self.nv.nvmlDeviceGetPowerUsage(self.h, c.byref(pw))
        self.reasons_fn(self.h, c.byref(rs))
        return float(clk.value), pw.value / 1000.0, int(rs.value)


class ClockSampler:
    """SM clocks and throttle reasons sampled during the run, with a marked window.

    With NVML a background thread reads the clock every half millisecond, so that a timed
    region of 10-30 ms holds a few dozen samples; without it, nvidia-smi samples every 20 ms.
    mark_start()/mark_end() bracket the timed region; stop() reports the median SM clock
    and the reasons seen over the samples inside it (and the sample counts)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.thread = None
        self.samples = []          # (host time, sm MHz, power W, reason names)
        self.t0 = self.t1 = None
        self.source = None
        out_dir = os.environ.get("LL_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            self.nvml = NvmlClocks(self.idx)
            self.source = "nvml, every 0.5 ms"
            import threading
            self.stop_flag = threading.Event()

            def loop():
                while not self.stop_flag.is_set():
                    mhz, w, rs = self.nvml.read()
                    names = [n for bit, n in NvmlClocks.REASONS.items() if rs & bit]
                    self.samples.append((time.perf_counter(), mhz, w, names))
                    time.sleep(0.0005)

            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            while not self.samples:
                time.sleep(0.001)
            return
        except Exception:
            self.thread = None
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi, every 20 ms"
            t0 = time.time()  # wait for the first sample so the window really starts here
            while time.time() - t0 < 3.0 and os.path.getsize(self.path) == 0:
                time.sleep(0.02)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join(timeout=2)
            inside = [x for x in self.samples
                      if self.t0 is not None and self.t0 <= x[0] <= (self.t1 or x[0])]
            sm = [x[1] for x in inside]
            reasons = sorted({n for x in inside for n in x[3]})
            return {"sm_mhz": statistics.median(sm) if sm else None,
                    "sm_max_mhz": self.nvml.max_mhz, "reasons": reasons,
                    "samples": len(inside), "samples_whole_run": len(self.samples),
                    "power_w_max": max((x[2] for x in inside), default=None),
                    "window": "the timed region (marked on the host)", "source": self.source}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm), "window": "warm-up + timed region, every 20 ms",
                "source": self.source}


# ---------------------------------------------------------------- CPU oracle sample


def oracle_sample(cfg, seconds, seed=0):
    """Times the oracle's direct forward on sampled query rows of one head, until about
    `seconds` of CPU time; returns (tokens/s extrapolated to the whole workload, sample
    description, threads used)."""
    import oracle
    T = cfg.T
    # one head drawn with the workload's recipe
    x = W.make_fwd_inputs(cfg.with_(B=1, H=1))
    rng = np.random.default_rng(seed)
    rows_done, pairs_done, t0 = 0, 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        rows = np.sort(rng.choice(T, 64, replace=False))
        oracle.forward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"], rows=rows,
                              heads=[(0, 0)])
        rows_done += len(rows)
        pairs_done += int((rows + 1).sum())
    el = time.perf_counter() - t0
    pairs_total = cfg.B * cfg.H * T * (T + 1) / 2
    t_total = el * pairs_total / pairs_done
    tok_s = cfg.B * T / t_total
    threads = _blas_threads()
    desc = (f"oracle forward_direct (fp64 NumPy) on {rows_done} random query rows of one head "
            f"of {cfg.name} in {el:.1f} s, extrapolated by (query, source) pair count to "
            f"B{cfg.B} H{cfg.H} T{T}")
    return tok_s, desc, threads


def oracle_decode_sample(dcfg, seconds):
    """Times the oracle's lssb decode step (fp64 NumPy) on a few (b, h) of the decode
    workload until about `seconds` of CPU time; returns (tokens/s extrapolated to all
    B x H, sample description, threads used)."""
    import oracle
    inp = W.make_decode_step_inputs(dcfg)
    nb = 2                                    # batch rows per call: 2 x H (b, h) pairs
    sub = dataclasses.replace(dcfg, B=nb)
    S = W.make_random_state(sub, dcfg.t, seed=3, scale=0.05).double().numpy()
    x = {k: (None if v is None else v[:nb]) for k, v in inp.items()}
    calls, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds or calls == 0:
        oracle.decode_step(S, x["q"], x["k"], x["v"], x["log_a"], x["lam"], dcfg.t)
        calls += 1
    el = time.perf_counter() - t0
    per_pair = el / (calls * nb * dcfg.H)
    t_step = per_pair * dcfg.B * dcfg.H
    desc = (f"oracle decode_step (fp64 NumPy) on {nb} x {dcfg.H} (b, h) pairs at t={dcfg.t}, "
            f"{calls} calls in {el:.1f} s, extrapolated by pair count to B{dcfg.B} H{dcfg.H}")
    return dcfg.B / t_step, desc, _blas_threads()


def oracle_gdn_decode_sample(dcfg, seconds):
    """Times the oracle's Log-Linear Gated DeltaNet decode step (fp64 NumPy) on a few (b, h)
    of the decode workload; returns (tokens/s extrapolated to all B x H, description,
    threads used)."""
    import oracle
    inp = W.make_gdn_decode_step_inputs(dcfg)
    nb = 2
    sub = dataclasses.replace(dcfg, B=nb)
    S = W.make_random_state(sub, dcfg.t, seed=3, scale=0.05).double().numpy()
    x = {k: (None if v is None else v[:nb]) for k, v in inp.items()}
    calls, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds or calls == 0:
        oracle.gdn_decode_step(S, x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"], dcfg.t)
        calls += 1
    el = time.perf_counter() - t0
    t_step = el / (calls * nb * dcfg.H) * dcfg.B * dcfg.H
    desc = (f"oracle gdn_decode_step (fp64 NumPy) on {nb} x {dcfg.H} (b, h) pairs at "
            f"t={dcfg.t}, {calls} calls in {el:.1f} s, extrapolated by pair count to "
            f"B{dcfg.B} H{dcfg.H}")
    return dcfg.B / t_step, desc, _blas_threads()


def _blas_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max([i.get("num_threads", 1) for i in info] + [1])
    except Exception:
        return os.cpu_count()


# ---------------------------------------------------------------- our implementation


def run_ours(args, rank, world, local_rank):
    import log_linear_attention_fwd_gb300 as LL
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = W.FWD_CONFIGS[W.HEADLINE_FWD]
    dcfg = W.DECODE_CONFIG
    peaks = load_peaks()
    x = W.make_fwd_inputs(cfg)
    d = {k: (None if v is None else v.to(dev)) for k, v in x.items()}
    out = torch.empty(cfg.B, cfg.T, cfg.H, cfg.dv, device=dev, dtype=d["q"].dtype)
    in_code = 1 if cfg.dtype == "bf16" else 0
    path = LL.resolve_path(cfg.dk, cfg.dv, cfg.C, in_code)
    ws = torch.empty(LL.fwd_workspace_size(cfg.B, cfg.T, cfg.H, cfg.dk, cfg.dv, cfg.C, in_code),
                     device=dev, dtype=torch.uint8)
    # decode inputs: state generated on the device from a seeded generator (timing only);
    # every timed step starts from this same state (restored outside the events), so each
    # step is the t = 12345 step on the state after position 12344
    gen = torch.Generator(device=dev).manual_seed(1234)
    state0 = torch.zeros(dcfg.B, dcfg.H, dcfg.L, dcfg.dk, dcfg.dv, device=dev)
    for lv in W.nonempty_levels_before(dcfg.t, dcfg.L):
        state0[:, :, lv].normal_(0.0, 0.05, generator=gen)
    state = torch.empty_like(state0)
    dinp = {k: (None if v is None else v.to(dev)) for k, v in W.make_decode_step_inputs(dcfg).items()}
    dout = torch.empty(dcfg.B, dcfg.H, dcfg.dv, device=dev, dtype=torch.float32)
    flush = torch.empty(512 << 20, device=dev, dtype=torch.uint8)
    n_ev = 5
    stream = torch.cuda.current_stream()

    def one_step(ev_f, ev_d):
        state.copy_(state0)  # restore the decode state (before the L2 flush and the events)
        flush.zero_()
        n_k = LL.loglinear_fwd_with_events(d["q"], d["k"], d["v"], d["log_a"], d["lam"], cfg.C,
                                           ev_f, out, ws)
        ev_d[0].record(stream)
        LL.loglinear_decode_step(state, dinp["q"], dinp["k"], dinp["v"], dinp["log_a"],
                                 dinp["lam"], dcfg.t, out=dout)
        ev_d[1].record(stream)
        return n_k

    mk = lambda n: [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    evs = [(mk(n_ev), mk(2)) for _ in range(args.steps)]
    # clocks are sampled from the start of the warm-up to the end of the timed region
    clocks = ClockSampler(local_rank)
    clocks.start()
    for _ in range(args.warmup):
        one_step(mk(n_ev), mk(2))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    clocks.mark_start()
    n_kernels = 0
    for ef, ed in evs:
        n_kernels = one_step(ef, ed)
    torch.cuda.synchronize()
    clocks.mark_end()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    t_fwd = [ef[0].elapsed_time(ef[n_kernels]) * 1e-3 for ef, _ in evs]
    t_stage = [[ef[i].elapsed_time(ef[i + 1]) * 1e-3 for ef, _ in evs] for i in range(n_kernels)]
    t_dec = [ed[0].elapsed_time(ed[1]) * 1e-3 for _, ed in evs]
    fwd_mean, dec_mean = sum(t_fwd) / len(t_fwd), sum(t_dec) / len(t_dec)
    stage_mean = [sum(s) / len(s) for s in t_stage]
    fwd_mean, dec_mean = max_over_ranks([fwd_mean, dec_mean], world, dev)
    fwd_tok_s = whole_job_rate(world, cfg.B * cfg.T, fwd_mean)
    dec_tok_s = whole_job_rate(world, dcfg.B, dec_mean)
    fbytes, fflops = fwd_algorithmic(cfg)
    dbytes = decode_algorithmic(dcfg)
    t_hbm = fbytes / (peaks["hbm"] * 1e9)
    t_tc = fflops / (peaks["bf16"] * 1e12)
    stage_names = {"simt": ["simt_chunk_state", "simt_level_scan", "simt_intra_readout"],
                   "tc": ["tc_forward"]}[path][-n_kernels:]
    dom = int(np.argmax(stage_mean))
    # achieved numbers for the forward pass as a whole and for its dominant kernel
    roofline_fwd = {"bound": "hbm" if t_hbm >= t_tc else "tensor",
                    "achieved": fbytes / fwd_mean / 1e9, "peak": peaks["hbm"], "unit": "GB/s",
                    "frac": (fbytes / fwd_mean / 1e9) / peaks["hbm"],
                    "frac_of_binding_roofline": max(t_hbm, t_tc) / fwd_mean,
                    "tensor_frac": (fflops / fwd_mean / 1e12) / peaks["bf16"],
                    "algorithmic_bytes": fbytes, "algorithmic_flops": fflops,
                    "peak_source": peaks["src"], "traffic": None}
    dom_bytes = stage_bytes(cfg, path, stage_names[dom])
    traffic = load_traffic(stage_names[dom] + "_kernel")
    roofline = {"kernel": stage_names[dom], "bound": "hbm",
                "achieved": dom_bytes / stage_mean[dom] / 1e9, "peak": peaks["hbm"],
                "unit": "GB/s", "frac": dom_bytes / stage_mean[dom] / 1e9 / peaks["hbm"],
                "traffic": traffic, "algorithmic_bytes": dom_bytes, "peak_source": peaks["src"],
                "us_per_launch": stage_mean[dom] * 1e6}
    decode = {"tokens_per_s": dec_tok_s, "us_per_step": dec_mean * 1e6,
              "roofline": {"kernel": "decode_step_kernel", "bound": "hbm",
                           "achieved": dbytes / dec_mean / 1e9, "peak": peaks["hbm"],
                           "unit": "GB/s", "frac": dbytes / dec_mean / 1e9 / peaks["hbm"],
                           "algorithmic_bytes": dbytes, "peak_source": peaks["src"],
                           "traffic": None},
              "config": {"workload": dcfg.name, "B": dcfg.B, "H": dcfg.H, "dk": dcfg.dk,
                         "dv": dcfg.dv, "L": dcfg.L, "t": dcfg.t, "state": "fp32",
                         "levels_read": len(W.nonempty_levels_before(dcfg.t, dcfg.L)),
                         "levels_written": decode_levels_written(dcfg),
                         "state_restored": "every timed step starts from the same state "
                                           "after t-1 (device copy outside the events)"}}
    gdn = measure_gdn_decode(LL, dcfg, state0, state, flush, peaks)
    gdn_fwd = measure_gdn_fwd(LL, cfg, dev, flush, peaks)
    e2e = measure_e2e(LL, cfg, x, dev, ws, args)
    prefill = measure_prefill(LL, cfg, d, out, ws, flush, peaks)
    del ws
    backward = measure_backward(LL, cfg, d, dev, flush, peaks)
    bench_shape = measure_benchmark_shape(LL, W.FWD_CONFIGS["mva_B2H48_T16384"], dev, flush, peaks)
    res = {"metric": METRIC, "value": fwd_tok_s, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": (fwd_mean + dec_mean) * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": f"{cfg.name}: loglinear_fwd B{cfg.B} H{cfg.H} T{cfg.T} "
                                  f"dk=dv={cfg.dk} C{cfg.C} L{cfg.L} bf16, + decode "
                                  f"B{dcfg.B} H{dcfg.H} d{dcfg.dk} L{dcfg.L} t={dcfg.t}",
                      "B": cfg.B, "H": cfg.H, "T": cfg.T, "dk": cfg.dk, "dv": cfg.dv,
                      "chunk": cfg.C, "L": cfg.L, "path": path,
                      "l2": "flushed (512 MiB write) between timed steps",
                      "parallelism": f"replicas x{world} (independent (b,h) work, no collective)"},
           "fwd_ms": fwd_mean * 1e3, "fwd_stage_us": dict(zip(stage_names, [s * 1e6 for s in stage_mean])),
           "roofline": roofline, "roofline_fwd": roofline_fwd, "decode": decode, "e2e": e2e,
           "prefill": prefill, "backward": backward, "benchmark_shape": bench_shape,
           "gdn_decode": gdn, "gdn_fwd": gdn_fwd,
           "gpu_launches": args.steps * (n_kernels + 1), "clocks": clk,
           "wall_s_timed_region": wall}
    return res


def stage_bytes(cfg, path, name):
    """Bytes each forward kernel of this design must move (its inputs and outputs)."""
    e = 2 if cfg.dtype == "bf16" else 4
    tok = cfg.B * cfg.T * cfg.H
    tile = 128 if path == "tc" else cfg.C
    N = -(-cfg.T // tile)
    st = cfg.B * cfg.H * N * cfg.dk * cfg.dv
    node_e = 2 if path == "tc" else 4
    qkv = cfg.B * cfg.T * cfg.qk_heads * 2 * cfg.dk * e + tok * cfg.dv * e
    if name == "tc_forward":  # one kernel: q, k, v, log a, lambda in, out out
        return qkv + tok * 4 + tok * cfg.L * 4 + tok * cfg.dv * e
    if name.endswith("chunk_state"):
        return cfg.B * cfg.T * cfg.qk_heads * cfg.dk * e + tok * cfg.dv * e + tok * 4 + st * 4
    if name.endswith("level_scan"):
        return st * 4 + st * node_e
    return qkv + tok * 4 + tok * cfg.L * 4 + st * node_e + tok * cfg.dv * e


def measure_gdn_decode(LL, dcfg, state0, state, flush, peaks, reps=20):
    """The Log-Linear Gated DeltaNet decode step on the decode workload's shape (B128 H16
    d128 L15 fp32 states, bf16 tokens, t = 12345): median of `reps` steps, each from the
    same state after t-1 (restored by a device copy, then L2 flushed, both outside the
    events).  With the delta rule every level that holds data changes, so the bytes are the
    decode step's: the non-empty levels read and the changed levels written."""
    dev = state.device
    inp = {k: (None if v is None else v.to(dev)) for k, v in W.make_gdn_decode_step_inputs(dcfg).items()}
    out = torch.empty(dcfg.B, dcfg.H, dcfg.dv, device=dev, dtype=torch.float32)
    ts = []
    for i in range(reps + 3):
        state.copy_(state0)
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        LL.loglinear_gdn_decode_step(state, inp["q"], inp["k"], inp["v"], inp["log_a"],
                                     inp["beta"], inp["lam"], dcfg.t, out=out)
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            ts.append(e0.elapsed_time(e1) * 1e-3)
    t = statistics.median(ts)
    dbytes = decode_algorithmic(dcfg)
    return {"workload": f"{dcfg.name}: loglinear_gdn_decode_step B{dcfg.B} H{dcfg.H} "
                        f"dk=dv={dcfg.dk} L{dcfg.L} t={dcfg.t}, fp32 states, bf16 tokens",
            "tokens_per_s": dcfg.B / t, "us_per_step": t * 1e6,
            "roofline": {"kernel": "gdn_decode_kernel", "bound": "hbm",
                         "achieved": dbytes / t / 1e9, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": dbytes / t / 1e9 / peaks["hbm"], "algorithmic_bytes": dbytes,
                         "peak_source": peaks["src"], "traffic": None}}


def gdn_fwd_algorithmic(cfg):
    """Bytes the Gated DeltaNet forward must move: q, k, v, log a, beta and lambda in, out
    out (the states stay on chip)."""
    e = 2 if cfg.dtype == "bf16" else 4
    tok = cfg.B * cfg.T * cfg.H
    return (cfg.B * cfg.T * cfg.qk_heads * 2 * cfg.dk * e + tok * cfg.dv * e + tok * 4 * 2 +
            tok * cfg.L * 4 + tok * cfg.dv * e)


def gdn_chunk_flops(cfg, C=64):
    """FLOPs of the chunked Gated DeltaNet forward as built (fp32 on CUDA cores): per chunk
    Q K^T and K K^T, the triangular inverse, W = Aqk T, (W ⊙ M^H) V, X = T K, Qt, the
    transition P = K^T X and the chunk state U = K^T T V; per (chunk, chunk level) the
    readout Qt Z and the carry P Z."""
    BH, dk, dv = cfg.B * cfg.H, cfg.dk, cfg.dv
    N = -(-cfg.T // C)
    per_chunk = 2 * (2 * C * C * dk + C ** 3 / 3 + C ** 3 + C * C * dv + C * C * dk * 2
                     + dk * C * dk + C * C * dv + dk * C * dv)
    levels = sum(bin(j).count("1") for j in range(N))
    per_level = 2 * (C * dk * dv + dk * dk * dv)
    return BH * (N * per_chunk + levels * per_level)


def measure_gdn_fwd(LL, cfg, dev, flush, peaks, reps=3):
    """The Log-Linear Gated DeltaNet forward on the headline shape, chunked (64-token chunks,
    fp32 on CUDA cores) and recurrent: median of `reps` calls after one warm-up, L2 flushed
    before each (outside the events).  The chunked form is bound by its fp32 arithmetic;
    its roofline is the FP32 FMA peak."""
    x = {k: (None if v is None else v.to(dev)) for k, v in W.make_gdn_inputs(cfg).items()}
    out = torch.empty(cfg.B, cfg.T, cfg.H, cfg.dv, device=dev, dtype=torch.bfloat16)
    ws = torch.empty(LL.gdn_fwd_chunked_workspace_size(cfg.B, cfg.T, cfg.H, cfg.dk, cfg.dv),
                     device=dev, dtype=torch.uint8)
    chunked = lambda: LL.loglinear_gdn_fwd_chunked(x["q"], x["k"], x["v"], x["log_a"], x["beta"],
                                                   x["lam"], out=out, workspace=ws)
    recurrent = lambda: LL.loglinear_gdn_fwd(x["q"], x["k"], x["v"], x["log_a"], x["beta"],
                                             x["lam"], out=out)
    chunked()
    t = _median_us(chunked, flush, reps)
    recurrent()
    t_rec = _median_us(recurrent, flush, 1)
    gbytes = gdn_fwd_algorithmic(cfg)
    gflops = gdn_chunk_flops(cfg)
    alu = fp32_alu_peak()
    return {"workload": f"{cfg.name}: loglinear_gdn_fwd_chunked B{cfg.B} H{cfg.H} T{cfg.T} "
                        f"dk=dv={cfg.dk} L{cfg.L} bf16 in/out, fp32 arithmetic",
            "tokens_per_s": cfg.B * cfg.T * cfg.H / t, "ms": t * 1e3,
            "roofline": {"kernel": "gdn_chunk_kernel + gdn_chunk_scan_kernel", "bound": "alu",
                         "achieved": gflops / t / 1e12, "peak": alu, "unit": "TFLOP/s",
                         "frac": gflops / t / 1e12 / alu, "algorithmic_flops": gflops,
                         "hbm_frac": gbytes / t / 1e9 / peaks["hbm"], "algorithmic_bytes": gbytes,
                         "peak_source": "fp32 FMA peak from unit counts and clock",
                         "traffic": None},
            "workspace_bytes": ws.numel(),
            "recurrent": {"ms": t_rec * 1e3, "tokens_per_s": cfg.B * cfg.T * cfg.H / t_rec,
                          "kernel": "gdn_fwd_kernel"}}


def oracle_gdn_fwd_sample(cfg, seconds):
    """Times the oracle's Gated DeltaNet recurrence (fp64 NumPy) on one (b, h) of the
    headline shape for a prefix of the sequence; returns (tokens/s, description, threads)."""
    import oracle
    sub = dataclasses.replace(cfg, B=1, H=1, T=256, L=9)
    x = W.make_gdn_inputs(sub)
    calls, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds or calls == 0:
        oracle.gdn_recurrence(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"])
        calls += 1
    el = time.perf_counter() - t0
    desc = (f"oracle gdn_recurrence (fp64 NumPy) on one (b, h), T={sub.T}, dk=dv={sub.dk}: "
            f"{calls} calls in {el:.1f} s; tokens of that sample per second")
    return calls * sub.T / el, desc, _blas_threads()


def measure_prefill(LL, cfg, d, out, ws, flush, peaks, reps=10):
    """The prefill -> decode handoff on the headline prompt: loglinear_prefill (forward
    plus the per-level decode state at T-1), medians of `reps` calls (L2 flushed before
    every call, outside the events), with events between its kernels so that the state
    kernel is timed by its own events.  Its bytes are the fp32 state it writes plus the
    block states it reads."""
    state = torch.empty(cfg.B, cfg.H, cfg.L, cfg.dk, cfg.dv, device=out.device,
                        dtype=torch.float32)

    t_pre, t_k = [], []
    for i in range(reps + 2):
        flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        nk = LL.loglinear_prefill_with_events(d["q"], d["k"], d["v"], d["log_a"], d["lam"], cfg.C,
                                              ev, out, state, ws)
        torch.cuda.synchronize()
        if i >= 2:
            t_pre.append(ev[0].elapsed_time(ev[nk]) * 1e-3)
            t_k.append(ev[nk - 1].elapsed_time(ev[nk]) * 1e-3)   # the state kernel, last
    t = cfg.T - 1
    j = t >> 7
    state_bytes = cfg.B * cfg.H * cfg.L * cfg.dk * cfg.dv * 4
    read_bytes = cfg.B * cfg.H * bin(j).count("1") * cfg.dk * cfg.dv * 2
    t_state = statistics.median(t_k)
    return {"prefill_us": statistics.median(t_pre) * 1e6, "kernels": nk,
            "state_kernel_us": t_state * 1e6, "state_bytes": state_bytes + read_bytes,
            "state_kernel_gbs": (state_bytes + read_bytes) / t_state / 1e9,
            "state_kernel_frac_of_hbm": (state_bytes + read_bytes) / t_state / 1e9 / peaks["hbm"],
            "note": "state kernel timed by its own events inside loglinear_prefill_with_events; "
                    "bytes = fp32 state written + bf16 block states read"}


def _median_us(fn, flush, reps):
    ts = []
    for i in range(reps + 2):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        if i >= 2:
            ts.append(e0.elapsed_time(e1) * 1e-3)
    return statistics.median(ts)


def _bwd_report(cfg, t, peaks, path):
    """The backward's time and roofline.  The tensor-core path is bound by HBM or the bf16
    tensor peak, whichever takes longer for its algorithmic bytes and FLOPs; the CUDA-core
    path by the FP32 FMA peak."""
    bbytes, bflops = bwd_algorithmic(cfg)
    if path == "tc":
        t_hbm = bbytes / (peaks["hbm"] * 1e9)
        t_tc = bflops / (peaks["bf16"] * 1e12)
        if t_hbm >= t_tc:
            roof = {"bound": "hbm", "achieved": bbytes / t / 1e9, "peak": peaks["hbm"],
                    "unit": "GB/s", "frac": bbytes / t / 1e9 / peaks["hbm"]}
        else:
            roof = {"bound": "tensor", "achieved": bflops / t / 1e12, "peak": peaks["bf16"],
                    "unit": "TFLOP/s", "frac": bflops / t / 1e12 / peaks["bf16"]}
        roof.update({"tensor_frac": bflops / t / 1e12 / peaks["bf16"],
                     "peak_source": peaks["src"]})
    else:
        roof = {"bound": "alu", "achieved": bflops / t / 1e12, "peak": fp32_alu_peak(),
                "unit": "TFLOP/s", "frac": bflops / t / 1e12 / fp32_alu_peak(),
                "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz",
                "hbm_frac": bbytes / t / 1e9 / peaks["hbm"]}
    roof.update({"algorithmic_flops": bflops, "algorithmic_bytes": bbytes})
    return {"bwd_us": t * 1e6, "tokens_per_s": cfg.B * cfg.T / t, "path": path, "roofline": roof}


def _bwd_path(LL, cfg):
    return "tc" if (cfg.dtype == "bf16" and cfg.dk == 128 and cfg.dv in (64, 128)) else "simt"


def measure_backward(LL, cfg, d, dev, flush, peaks, reps=5):
    """The backward (CUDA cores, fp32) on the headline shape: median of `reps` calls,
    L2 flushed before each, outside the events; dO drawn on the device (timing only)."""
    g = torch.Generator(device=dev).manual_seed(7)
    dout = torch.randn(cfg.B, cfg.T, cfg.H, cfg.dv, device=dev, generator=g).to(d["q"].dtype)
    ws = torch.empty(LL.bwd_workspace_size(cfg.B, cfg.T, cfg.H, cfg.qk_heads, cfg.dk, cfg.dv,
                                           cfg.L, 1, 1), device=dev, dtype=torch.uint8)
    t = _median_us(lambda: LL.loglinear_bwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], dout,
                                            workspace=ws), flush, reps)
    path = _bwd_path(LL, cfg)
    rep = _bwd_report(cfg, t, peaks, path)
    rep["workload"] = f"{cfg.name}: loglinear_bwd, bf16 inputs and gradients"
    if path == "tc":  # the training step: the forward's workspace kept for the backward
        fws = torch.empty(LL.fwd_workspace_size(cfg.B, cfg.T, cfg.H, cfg.dk, cfg.dv, cfg.C, 1),
                          device=dev, dtype=torch.uint8)
        LL.loglinear_fwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], cfg.C, workspace=fws)
        tg = _median_us(lambda: LL.loglinear_bwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"],
                                                 dout, workspace=ws, fwd_workspace=fws),
                        flush, reps)
        rep["bwd_given_fwd_us"] = tg * 1e6
        rep["note"] = ("bwd_us recomputes the forward's block states; bwd_given_fwd_us reads "
                       "them from the forward's workspace")
    return rep


def measure_benchmark_shape(LL, cfg, dev, flush, peaks, reps=10):
    """The forward on the pages' kernel-benchmark shape (B2, 48 heads, d_v 64, d_k 128,
    one q/k shared by all heads): median of `reps` calls, L2 flushed before each call
    outside the events; tokens/s counts B*T tokens (all heads)."""
    x = W.make_fwd_inputs(cfg)
    d = {k: (None if v is None else v.to(dev)) for k, v in x.items()}
    out = torch.empty(cfg.B, cfg.T, cfg.H, cfg.dv, device=dev, dtype=d["q"].dtype)
    ws = torch.empty(LL.fwd_workspace_size(cfg.B, cfg.T, cfg.H, cfg.dk, cfg.dv, cfg.C, 1),
                     device=dev, dtype=torch.uint8)
    ts = []
    for i in range(reps + 3):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        LL.loglinear_fwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], cfg.C, out=out,
                         workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            ts.append(e0.elapsed_time(e1) * 1e-3)
    if LL.device_error() != 0:
        raise RuntimeError("tensor-core forward reported a device error")
    t = statistics.median(ts)
    fbytes, fflops = fwd_algorithmic(cfg)
    g = torch.Generator(device=dev).manual_seed(7)
    dout = torch.randn(cfg.B, cfg.T, cfg.H, cfg.dv, device=dev, generator=g).to(d["q"].dtype)
    bws = torch.empty(LL.bwd_workspace_size(cfg.B, cfg.T, cfg.H, cfg.qk_heads, cfg.dk, cfg.dv,
                                            cfg.L, 1, 1), device=dev, dtype=torch.uint8)
    tb = _median_us(lambda: LL.loglinear_bwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], dout,
                                             workspace=bws), flush, 3)
    bwd = _bwd_report(cfg, tb, peaks, _bwd_path(LL, cfg))
    # the training step: a forward that keeps its workspace, then the backward reading it
    fws = ws

    def step():
        LL.loglinear_fwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], cfg.C, out=out,
                         workspace=fws)
        LL.loglinear_bwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], dout, workspace=bws,
                         fwd_workspace=fws)

    t_step = _median_us(step, flush, 3)
    return {"workload": f"{cfg.name}: loglinear_fwd B{cfg.B} H{cfg.H} (q/k heads "
                        f"{cfg.qk_heads}) T{cfg.T} dk={cfg.dk} dv={cfg.dv} C{cfg.C} L{cfg.L} bf16",
            "path": LL.resolve_path(cfg.dk, cfg.dv, cfg.C, 1), "fwd_us": t * 1e6,
            "fwd_bwd_us": t_step * 1e6, "backward": bwd,
            "fwd_bwd_note": "one forward keeping its workspace, then the backward reading it "
                            "(the training step); backward.bwd_us alone recomputes the states",
            "tokens_per_s": cfg.B * cfg.T / t,
            "roofline": {"bound": "hbm", "achieved": fbytes / t / 1e9, "peak": peaks["hbm"],
                         "unit": "GB/s", "frac": fbytes / t / 1e9 / peaks["hbm"],
                         "algorithmic_bytes": fbytes, "peak_source": peaks["src"],
                         "tensor_frac": fflops / t / 1e12 / peaks["bf16"],
                         "algorithmic_flops": fflops}}


def run_sweep():
    """The benchmark shape's forward, backward (with its recompute) and training step
    (forward keeping its workspace, then the backward reading it) over the sequence lengths
    of the pages' kernel benchmark, L = bit_length(T - 1) + 1; medians of a few calls, L2
    flushed before each."""
    import log_linear_attention_fwd_gb300 as LL
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    flush = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev)
    base = W.FWD_CONFIGS["mva_B2H48_T16384"]
    rows = []
    for T in (1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072):
        cfg = base.with_(name=f"mva_B2H48_T{T}", T=T, L=(T - 1).bit_length() + 1)
        r = measure_benchmark_shape(LL, cfg, dev, flush, peaks, reps=5)
        rows.append({"T": T, "L": cfg.L, "fwd_us": r["fwd_us"], "bwd_us": r["backward"]["bwd_us"],
                     "fwd_bwd_us": r["fwd_bwd_us"], "fwd_hbm_frac": r["roofline"]["frac"],
                     "fwd_tensor_frac": r["roofline"]["tensor_frac"],
                     "bwd_tensor_frac": r["backward"]["roofline"]["tensor_frac"]})
        torch.cuda.empty_cache()
    print(json.dumps({"mode": "sweep-t", "workload": "B2 H48 (q/k heads 1) dk=128 dv=64 C64 bf16, "
                      "Mamba-2 decay, synthetic", "peak_source": peaks["src"], "rows": rows}))


def measure_e2e(LL, cfg, x, dev, ws, args):
    """Forward through the public API with inputs in pinned host memory: every step copies
    its inputs to the device, runs loglinear_fwd and copies the output back.

    Two forms: serial (copy in, forward, copy out, all on one stream) and pipelined over a
    stream of steps (step i+1's inputs copied in and step i-1's output copied out while
    step i computes; device inputs and outputs double-buffered, ordered by events).  The
    pipelined form is the reported value; both include every step's copies."""
    host = {k: (None if v is None else v.pin_memory()) for k, v in x.items()}
    dbufs = [{k: (None if v is None else torch.empty_like(v, device=dev)) for k, v in x.items()}
             for _ in range(2)]
    outs_h = [torch.empty(cfg.B, cfg.T, cfg.H, cfg.dv, dtype=x["q"].dtype).pin_memory()
              for _ in range(2)]
    outs_d = [torch.empty(cfg.B, cfg.T, cfg.H, cfg.dv, dtype=x["q"].dtype, device=dev)
              for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    n = max(4, args.steps // 2)

    def serial_step():
        for k, v in host.items():
            if v is not None:
                dbufs[0][k].copy_(v, non_blocking=True)
        d = dbufs[0]
        LL.loglinear_fwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], cfg.C, out=outs_d[0],
                         workspace=ws)
        outs_h[0].copy_(outs_d[0], non_blocking=True)

    for _ in range(max(2, args.warmup)):
        serial_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        serial_step()
    e1.record()
    torch.cuda.synchronize()
    t_serial = e0.elapsed_time(e1) * 1e-3 / n

    s_in, s_fwd, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    mk = lambda: [torch.cuda.Event(), torch.cuda.Event()]

    def pipelined(steps):
        ev_in, ev_done, ev_read = mk(), mk(), mk()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s_in)
        for i in range(steps):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[b])      # forward i-2 has read buffer b
                for k, v in host.items():
                    if v is not None:
                        dbufs[b][k].copy_(v, non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_fwd):
                s_fwd.wait_event(ev_in[b])
                if i >= 2:
                    s_fwd.wait_event(ev_read[b])     # output i-2 has been copied out
                d = dbufs[b]
                LL.loglinear_fwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], cfg.C,
                                 out=outs_d[b], workspace=ws, stream=s_fwd)
                ev_done[b].record(s_fwd)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                outs_h[b].copy_(outs_d[b], non_blocking=True)
                ev_read[b].record(s_out)
        end.record(s_out)
        torch.cuda.synchronize()
        return start.elapsed_time(end) * 1e-3 / steps

    pipelined(max(2, args.warmup))
    t_pipe = pipelined(n)
    return {"value": cfg.B * cfg.T / t_pipe, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": t_pipe * 1e3, "pipelined": True,
            "serial": {"value": cfg.B * cfg.T / t_serial, "ms_per_step": t_serial * 1e3}}


def run_one_pass(args, backward):
    """The forward (or the backward) alone on one workload (the headline by default), K
    timed calls after W warm-ups, L2 flushed between calls; for profilers, which should not
    see the 2 GiB decode state."""
    import log_linear_attention_fwd_gb300 as LL
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cfg = W.FWD_CONFIGS[args.workload or W.HEADLINE_FWD]
    x = W.make_fwd_inputs(cfg)
    d = {k: (None if v is None else v.to(dev)) for k, v in x.items()}
    in_code = 1 if cfg.dtype == "bf16" else 0
    if backward:
        g = torch.Generator(device=dev).manual_seed(7)
        dout = torch.randn(cfg.B, cfg.T, cfg.H, cfg.dv, device=dev, generator=g).to(d["q"].dtype)
        ws = torch.empty(LL.bwd_workspace_size(cfg.B, cfg.T, cfg.H, cfg.qk_heads, cfg.dk, cfg.dv,
                                               cfg.L, in_code, in_code), device=dev,
                         dtype=torch.uint8)
        call = lambda: LL.loglinear_bwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], dout,
                                        workspace=ws)
    else:
        out = torch.empty(cfg.B, cfg.T, cfg.H, cfg.dv, device=dev, dtype=d["q"].dtype)
        ws = torch.empty(LL.fwd_workspace_size(cfg.B, cfg.T, cfg.H, cfg.dk, cfg.dv, cfg.C,
                                               in_code), device=dev, dtype=torch.uint8)
        call = lambda: LL.loglinear_fwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], cfg.C,
                                        out=out, workspace=ws)
    flush = torch.empty(512 << 20, device=dev, dtype=torch.uint8)
    times = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1) * 1e3)
    assert LL.device_error() == 0
    name = "bwd" if backward else "fwd"
    print(json.dumps({"mode": f"{name}-only", "workload": cfg.name, "steps": args.steps,
                      "warmup": args.warmup, f"{name}_us_mean": sum(times) / len(times),
                      f"{name}_us_min": min(times)}), flush=True)


def run_decode_only(args):
    """The decode step alone (K timed steps after W warm-ups, each from the same state after
    t-1, L2 flushed between steps), for profilers."""
    import log_linear_attention_fwd_gb300 as LL
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dcfg = W.DECODE_CONFIG
    if args.decode_batch:
        dcfg = dataclasses.replace(dcfg, B=args.decode_batch)
    gen = torch.Generator(device=dev).manual_seed(1234)
    state0 = torch.zeros(dcfg.B, dcfg.H, dcfg.L, dcfg.dk, dcfg.dv, device=dev)
    for lv in W.nonempty_levels_before(dcfg.t, dcfg.L):
        state0[:, :, lv].normal_(0.0, 0.05, generator=gen)
    state = torch.empty_like(state0)
    gdn = args.decode_only == "gdn"
    make = W.make_gdn_decode_step_inputs if gdn else W.make_decode_step_inputs
    inp = {k: (None if v is None else v.to(dev)) for k, v in make(dcfg).items()}
    out = torch.empty(dcfg.B, dcfg.H, dcfg.dv, device=dev)
    flush = torch.empty(512 << 20, device=dev, dtype=torch.uint8)
    times = []
    for i in range(args.warmup + args.steps):
        state.copy_(state0)
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        if gdn:
            LL.loglinear_gdn_decode_step(state, inp["q"], inp["k"], inp["v"], inp["log_a"],
                                         inp["beta"], inp["lam"], dcfg.t, out=out)
        else:
            LL.loglinear_decode_step(state, inp["q"], inp["k"], inp["v"], inp["log_a"], inp["lam"],
                                     dcfg.t, out=out)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1) * 1e3)
    print(json.dumps({"mode": f"{args.decode_only}-decode-only", "B": dcfg.B, "t": dcfg.t,
                      "steps": args.steps, "warmup": args.warmup,
                      "us_mean": sum(times) / len(times), "us_min": min(times)}), flush=True)


def main():
    args = parse()
    if args.sweep_t:
        run_sweep()
        return
    if args.fwd_only or args.bwd_only:
        run_one_pass(args, backward=args.bwd_only)
        return
    if args.decode_only:
        run_decode_only(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = W.FWD_CONFIGS[W.HEADLINE_FWD]
    if args.impl == "reference":
        if rank != 0:
            return
        steps = []
        per = max(2.0, 150.0 / max(1, args.steps + args.warmup))
        for i in range(args.warmup + args.steps):
            tok_s, desc, thr = oracle_sample(cfg, per, seed=i)
            if i >= args.warmup:
                steps.append(tok_s)
        v = statistics.median(steps)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": cfg.B * cfg.T / v * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": f"{cfg.name}: direct O(T^2) oracle, B{cfg.B} H{cfg.H} "
                                       f"T{cfg.T} dk=dv={cfg.dk} L{cfg.L}"},
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok_s, desc, thr = oracle_sample(cfg, args.cpu_seconds)
        res["cpu_baseline"] = {"value": tok_s, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                               "sample": desc}
        dtok_s, ddesc, dthr = oracle_decode_sample(W.DECODE_CONFIG, max(2.0, args.cpu_seconds / 3))
        res["decode"]["cpu_baseline"] = {"value": dtok_s, "unit": "tokens/s", "cores": dthr,
                                         "kind": "oracle", "sample": ddesc}
        gtok_s, gdesc, gthr = oracle_gdn_decode_sample(W.DECODE_CONFIG, max(2.0, args.cpu_seconds / 3))
        res["gdn_decode"]["cpu_baseline"] = {"value": gtok_s, "unit": "tokens/s", "cores": gthr,
                                             "kind": "oracle", "sample": gdesc}
        ftok_s, fdesc, fthr = oracle_gdn_fwd_sample(cfg, max(2.0, args.cpu_seconds / 5))
        res["gdn_fwd"]["cpu_baseline"] = {"value": ftok_s, "unit": "tokens/s", "cores": fthr,
                                          "kind": "oracle", "sample": fdesc}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
