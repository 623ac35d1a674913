#!/usr/bin/env python
"""Benchmark of the GB300 tensor-core GEMM path.

One step = the three square GEMMs the study measures at N = 8192 ("Hand-Written
PTX Tensor-Core GEMM Kernels: A Multi-Precision Study on NVIDIA L4", Tables II
and III): FP16 -> FP32 (operands normal(0,1)/sqrt(K)), INT8 -> INT32 and packed
INT4 -> INT32 (operands uniform over their ranges), on seeded synthetic inputs
already resident in HBM.  The working set of a step (~1.2 GB) is far larger
than L2, so no flush is needed between steps.

Reported (one JSON line from rank 0):
  value        2*N^3 multiply-adds counted as operations, summed over the three
               GEMMs of every step of every rank, divided by the max-over-ranks
               device time of the timed steps  [TOPS]
  per_precision  TFLOP/s / TOPS of each call: the median over 5 batches of
               the batch's mean per-call time, and the best batch
  peak_fractions  each precision against its nominal dense peak, against the
               measured peak of the tensor-core kind it runs on, and against
               that kind's dense per-SM rate x SMs x the SM clock its kernels
               ran at (their CTAs' own cycle and global-timer counts)
  roofline     the FP16 GEMM kernel (one launch per gemm_f16 call) against the
               measured bf16 tensor-core peak (FP16 runs at the bf16 rate):
               the burst figure when the timed region is shorter than a
               second, else the sustained one; both fractions are given
  e2e          the same metric through the public API with pinned host
               buffers (the host-buffer entry points, one stream per product):
               H2D of the operands, the GEMMs, D2H of the results, every step
  cpu_baseline the CPU oracle on a bounded row sample of the same workload
  clocks       SM clocks and throttle reasons sampled during the timed region

--impl reference times the CPU oracle as the reference arm, on row samples.
--sweep times every precision at N = 512 ... 8192 (graph replays, median and
min of 5 batches, an L2-flushed variant for N <= 2048) with the CPU oracle
timed beside each configuration; it prints one JSON line per configuration
and no bench line.
Multi-GPU: one process per GPU under torchrun; every rank runs the full step
on its own data (independent problems, weak scaling); only the timing
barrier and a max-reduction of the elapsed time cross ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s / TOPS at N=8192 (FP16, INT8, INT4); fraction of GB300 dense peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM read + write bytes of one launch of the FP16 GEMM kernel at N = 8192 come
# from the record beside its ncu summary (made with
# `ncu --set full --clock-control none -k regex:gemm_kernel -s 1 -c 1
#  python -m precision_tensor_core_gb300.run --prec f16 --n 8192`), which names
# the hash of the kernel sources it was captured from; a record of other sources
# is stale and gives no traffic figure.
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "traffic_gemm_f16_n8192.txt")
KERNEL_SOURCES = ("gemm_tc.cu", "ptx.cuh", "internal.h", "convert.cuh")
# Dense tensor-core rate per SM and clock: 8192 FLOP (M = 128, N = 256, K = 16
# binary16 MMA, 2 * 128 * 256 * 16 FLOP, every 128 cycles) for the FP16 kind,
# twice that for the E4M3 kind.
PER_SM_CLOCK_FLOP = {"kind::f16": 8192.0, "kind::f8f6f4": 16384.0}
BATCHES = 5
# A timed region shorter than this is a burst: the kernel's clock has not
# settled under the power cap, so the burst peak is the denominator.
SUSTAINED_AFTER_MS = 1000.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--n", type=int, default=8192)
    p.add_argument("--e2e-steps", type=int, default=0, help="0: min(steps, 20)")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline budget")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--sweep", action="store_true",
                   help="precision x size sweep with the oracle timed beside each size (no bench line)")
    p.add_argument("--sweep-sizes", type=lambda v: [int(x) for x in v.split(",")],
                   default=[512, 1024, 2048, 4096, 8192])
    p.add_argument("--sweep-oracle-seconds", type=float, default=2.0)
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_of(text: str) -> str:
    """C++/CUDA source without comments and with whitespace runs collapsed, so
    that a comment edit does not change the kernel's identity."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(read=None) -> str:
    """First 16 hex digits of the SHA-256 of the GEMM kernel's sources (their
    code, comments removed).  `read(name)` supplies a file's text (default: the
    working tree)."""
    import hashlib
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "precision_tensor_core_gb300", "csrc", name)) as f:
                return f.read()
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(name.encode() + b"\0" + code_of(read(name)).encode())
    return h.hexdigest()[:16]


def traffic_record():
    """(DRAM bytes per launch, note) of the FP16 kernel from the committed ncu
    record, or (None, why) when it is absent or was taken from other sources."""
    if not os.path.exists(TRAFFIC_RECORD):
        return None, "no ncu traffic record"
    rec = {}
    with open(TRAFFIC_RECORD) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                rec[k.strip()] = v.strip()
    if rec.get("source_sha256_16") != kernel_source_hash():
        return None, "ncu traffic record is from other kernel sources (stale)"
    return float(rec["dram_bytes_read"]) + float(rec["dram_bytes_write"]), "profiles/traffic_gemm_f16_n8192.txt"


# ---------------------------------------------------------------- ranks
def reduce_max(dist, x: float, device) -> float:
    """Max of x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput_tops(ops_per_step: float, steps: int, world: int, elapsed_ms: float) -> float:
    """Whole-job TOPS: the operations every rank did, over the slowest rank's time."""
    return ops_per_step * steps * world / (elapsed_ms * 1e-3) / 1e12


# ---------------------------------------------------------------- inputs
def make_inputs(n):
    import datagen
    A16, B16 = datagen.f16_operands(n, "normal")
    A8, B8 = datagen.s8_operands(n)
    A4, B4 = datagen.s4_operands(n)
    return {"f16": (A16.view(np.float16), B16.view(np.float16)),
            "s8": (A8, B8), "s4": (A4, B4)}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        busy = [s for s in sm if s > 0.5 * (max(sm) if sm else 1)]
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, dist):
    import torch
    import __graft_entry__
    import precision_tensor_core_gb300 as ptc

    __graft_entry__.build()
    local = int(os.environ.get("LOCAL_RANK", 0))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n = args.n
    host = make_inputs(n)
    d = {k: (torch.from_numpy(np.ascontiguousarray(a)).to(dev),
             torch.from_numpy(np.ascontiguousarray(b)).to(dev)) for k, (a, b) in host.items()}
    C16 = torch.empty((n, n), dtype=torch.float32, device=dev)
    C8 = torch.empty((n, n), dtype=torch.int32, device=dev)
    C4 = torch.empty((n, n), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ptc.matmul_f16(d["f16"][0], d["f16"][1], out=C16)
        if ev is not None:
            ev[1].record(stream)
        ptc.matmul_s8(d["s8"][0], d["s8"][1], out=C8)
        if ev is not None:
            ev[2].record(stream)
        ptc.matmul_s4(d["s4"][0], d["s4"][1], n, out=C4)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    # Batch boundaries: the timed steps in BATCHES consecutive batches.
    nb = max(1, min(BATCHES, args.steps))
    bounds = [round(b * args.steps / nb) for b in range(nb + 1)]
    bev = [torch.cuda.Event(enable_timing=True) for _ in range(nb + 1)]
    sampler = ClockSampler(local)
    sampler.start()
    ptc.ptc_clock_probe_read()  # clear the clock record
    ptc.ptc_set_tuning("clock_probe", 1)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = ptc.ptc_kernel_launch_count()
    bev[0].record(stream)
    for b in range(nb):
        for i in range(bounds[b], bounds[b + 1]):
            step(evs[i])
        bev[b + 1].record(stream)
    torch.cuda.synchronize()
    launches = ptc.ptc_kernel_launch_count() - launches0
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    ptc.ptc_set_tuning("clock_probe", 0)
    cyc, ns, ctas = ptc.ptc_clock_probe_read()
    elapsed_ms = bev[0].elapsed_time(bev[nb])
    batch_ms = [bev[b].elapsed_time(bev[b + 1]) / (bounds[b + 1] - bounds[b]) for b in range(nb)]
    t16 = [e[0].elapsed_time(e[1]) for e in evs]
    t8 = [e[1].elapsed_time(e[2]) for e in evs]
    t4 = [e[2].elapsed_time(e[3]) for e in evs]
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK
    elapsed_ms = reduce_max(dist, elapsed_ms, dev)

    def per_batch(ts):
        """Mean per-call time of each batch (ms)."""
        return [statistics.mean(ts[bounds[b]:bounds[b + 1]]) for b in range(nb)]

    ops = 2.0 * n ** 3
    value = throughput_tops(3 * ops, args.steps, world, elapsed_ms)
    ms = {"fp16": per_batch(t16), "int8": per_batch(t8), "int4": per_batch(t4)}
    med = {k: statistics.median(v) for k, v in ms.items()}
    best = {k: min(v) for k, v in ms.items()}
    per = {"fp16_tflops": ops / (med["fp16"] * 1e-3) / 1e12,
           "int8_tops": ops / (med["int8"] * 1e-3) / 1e12,
           "int4_tops": ops / (med["int4"] * 1e-3) / 1e12,
           "ms": med, "ms_min": best,
           "best": {"fp16_tflops": ops / (best["fp16"] * 1e-3) / 1e12,
                    "int8_tops": ops / (best["int8"] * 1e-3) / 1e12,
                    "int4_tops": ops / (best["int4"] * 1e-3) / 1e12},
           "statistic": f"median over {nb} batches of the batch's mean per-call time (CUDA events on the "
                        f"launching stream); ms_min / best: the fastest batch"}
    batches = {"batches": nb, "ms_per_step_median": statistics.median(batch_ms),
               "ms_per_step_min": min(batch_ms), "ms_per_step_each": batch_ms}
    # Mean SM clock each GEMM kernel family ran at, from its CTAs' own cycle and
    # global-timer counts.
    kernel_mhz = {fam: (1e3 * cyc[i] / ns[i] if ns[i] else None)
                  for i, fam in enumerate(("fp16", "int8", "int4"))}
    clocks["kernel_sm_mhz"] = kernel_mhz
    clocks["kernel_sm_mhz_how"] = ("sum of %clock64 cycles / sum of %globaltimer ns over every CTA of every "
                                   "timed GEMM kernel launch (thread 0, start of work to exit)")
    clocks["kernel_ctas"] = {fam: int(ctas[i]) for i, fam in enumerate(("fp16", "int8", "int4"))}

    # e2e through the public API with pinned host buffers
    e2e_steps = args.e2e_steps or min(args.steps, 20)
    hp = {k: (torch.from_numpy(np.ascontiguousarray(a)).pin_memory(),
              torch.from_numpy(np.ascontiguousarray(b)).pin_memory()) for k, (a, b) in host.items()}
    h16 = torch.empty((n, n), dtype=torch.float32, pin_memory=True)
    h8 = torch.empty((n, n), dtype=torch.int32, pin_memory=True)
    h4 = torch.empty((n, n), dtype=torch.int32, pin_memory=True)

    # The three products on three streams: each call pipelines its own copies
    # (host-buffer entry points), and the calls overlap one another.
    e2e_streams = [torch.cuda.Stream() for _ in range(3)]

    def e2e_step():
        ptc.matmul_f16(hp["f16"][0], hp["f16"][1], out=h16, stream=e2e_streams[0], sync=False)
        ptc.matmul_s8(hp["s8"][0], hp["s8"][1], out=h8, stream=e2e_streams[1], sync=False)
        ptc.matmul_s4(hp["s4"][0], hp["s4"][1], n, out=h4, stream=e2e_streams[2], sync=False)

    e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for st in e2e_streams:
        st.wait_event(e0)
    for _ in range(e2e_steps):
        e2e_step()
    for st in e2e_streams:
        stream.wait_stream(st)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(dist, e0.elapsed_time(e1), dev)
    h2d = sum(a.numel() * a.element_size() + b.numel() * b.element_size() for a, b in hp.values())
    d2h = sum(x.numel() * x.element_size() for x in (h16, h8, h4))
    e2e = {"value": throughput_tops(3 * ops, e2e_steps, world, e2e_ms), "unit": "TOPS",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
           "ms_per_step": e2e_ms / e2e_steps,
           "how": "gemm_f16_host / gemm_s8_host / gemm_s4_host on pinned host buffers, one stream each"}

    peaks, src = load_peaks()
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    is_burst = elapsed_ms < SUSTAINED_AFTER_MS
    peak = burst if is_burst else sustained
    traffic, traffic_note = traffic_record() if n == 8192 else (None, "recorded for N = 8192 only")
    if traffic is not None:
        traffic_note += " (one ncu capture, cold L2)"
    achieved = per["fp16_tflops"]
    roofline = {"bound": "tensor", "kernel": "gemm_kernel<F16, B MN-major, f32 out, CTA pair> (gemm_f16)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": (f"{'bf16_tflops (burst)' if is_burst else 'bf16_tflops_sustained'} of {src} "
                                f"MEASURED_PEAKS.json, FP16 = bf16 rate; the timed region lasted "
                                f"{elapsed_ms:.0f} ms ({'<' if is_burst else '>='} {SUSTAINED_AFTER_MS:.0f} ms)"),
                "frac_of_burst": achieved / burst, "frac_of_sustained": achieved / sustained,
                "traffic": traffic, "traffic_source": traffic_note,
                "int8_frac_of_f16_peak": per["int8_tops"] / peak,
                "int4_frac_of_fp8_peak": per["int4_tops"] / (2 * peak)}
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fractions = peak_fractions(per, peak, kernel_mhz, sms)
    return {"value": value, "elapsed_ms": elapsed_ms, "per": per, "e2e": e2e, "roofline": roofline,
            "clocks": clocks, "launches": int(launches), "fractions": fractions, "batches": batches}


# Nominal dense tensor-core rates of GB300 quoted with the metric (TFLOP/s or
# TOPS): FP16 about 2.25 P, INT8 about 4.5 P; INT4 is quoted as INT8's.
NOMINAL = {"fp16": 2250.0, "int8": 4500.0, "int4": 4500.0}


def peak_fractions(per, measured_f16_peak, kernel_mhz, sms):
    """Each precision's throughput against the denominators of the metric:
    the nominal dense peak of its precision; the measured peak of the
    tensor-core kind it actually runs on (the cuBLAS bf16 rate for kind::f16,
    FP16 and the INT8 route; twice that for the E4M3 kind of the INT4 route);
    and that kind's dense per-SM rate x SMs x the mean SM clock its own
    kernels ran at during the timed region (the clock record)."""
    rows = {"fp16": ("fp16_tflops", "kind::f16", measured_f16_peak),
            "int8": ("int8_tops", "kind::f16", measured_f16_peak),
            "int4": ("int4_tops", "kind::f8f6f4", 2 * measured_f16_peak)}
    out = {}
    for prec, (key, kind, pipe_peak) in rows.items():
        a = per[key]
        mhz = kernel_mhz.get(prec)
        clock_peak = PER_SM_CLOCK_FLOP[kind] * sms * mhz * 1e6 / 1e12 if mhz else None
        out[prec] = {"achieved": a, "nominal_peak": NOMINAL[prec], "frac_nominal": a / NOMINAL[prec],
                     "pipe": kind, "pipe_peak_measured": pipe_peak, "frac_pipe_measured": a / pipe_peak,
                     "kernel_sm_mhz": mhz,
                     "pipe_peak_clock_adjusted": clock_peak,
                     "frac_pipe_clock_adjusted": (a / clock_peak) if clock_peak else None}
    return out


# ---------------------------------------------------------------- oracle timing
def oracle_sample(host, n, rows, nthreads):
    """Run the CPU oracle on the first `rows` output rows of each precision's
    GEMM; returns (seconds, operations)."""
    import oracle
    t0 = time.perf_counter()
    A16, B16 = host["f16"]
    oracle.gemm_f16(A16[:rows].view(np.uint16), B16.view(np.uint16), nthreads=nthreads)
    A8, B8 = host["s8"]
    oracle.gemm_s8(A8[:rows], B8, nthreads=nthreads)
    A4, B4 = host["s4"]
    oracle.gemm_s4(A4[:rows], B4, n, nthreads=nthreads)
    return time.perf_counter() - t0, 3 * 2.0 * rows * n * n


def cpu_baseline(host, n, budget_s):
    cores = os.cpu_count() or 1
    rows = cores
    secs, ops = oracle_sample(host, n, rows, cores)
    if secs < budget_s / 3:
        rows = max(rows, min(n, int(rows * (budget_s / 2) / max(secs, 1e-3))) // cores * cores)
        secs, ops = oracle_sample(host, n, rows, cores)
    return {"value": ops / secs / 1e12, "unit": "TOPS", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} output rows of each of the FP16, INT8 and INT4 N={n} GEMMs "
                      f"({ops:.3g} ops, {secs:.1f} s, {cores} threads)"}


# ---------------------------------------------------------------- size sweep
def _oracle_rows(prec, A, B, n, rows, nthreads):
    """Seconds the CPU oracle takes for the first `rows` output rows."""
    import oracle
    t0 = time.perf_counter()
    if prec.startswith("f16"):
        oracle.gemm_f16(A[:rows], B, nthreads=nthreads)
    elif prec == "s8":
        oracle.gemm_s8(A[:rows], B, nthreads=nthreads)
    else:
        oracle.gemm_s4(A[:rows], B, n, nthreads=nthreads)
    return time.perf_counter() - t0


def _oracle_time(prec, A, B, n, nthreads, budget_s):
    """Oracle time of the whole N x N product on `nthreads` threads: measured
    when it fits the budget, else extrapolated from a timed row sample."""
    rows = max(1, min(n, nthreads))
    secs = _oracle_rows(prec, A, B, n, rows, nthreads)
    while rows < n and secs < budget_s / 4:
        rows = min(n, rows * 4)
        secs = _oracle_rows(prec, A, B, n, rows, nthreads)
    full = secs * n / rows
    return {"threads": nthreads, "seconds": full, "extrapolated": rows < n, "rows_timed": rows,
            "tops": 2.0 * n ** 3 / full / 1e12}


def run_sweep(args):
    """Precision x size sweep: GPU time per call (median and min over 5
    batches of CUDA-graph replays, L2 warm; for N <= 2048 also with a 512 MiB
    L2 flush before every call) and the CPU oracle on the same inputs (all
    host cores; one core too for N <= 1024).  One JSON line per configuration."""
    import torch
    import datagen
    import __graft_entry__
    import precision_tensor_core_gb300 as ptc

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cores = os.cpu_count() or 1
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    cases = [("f16u", 512)] if 512 in args.sweep_sizes else []
    cases += [(p, n) for n in args.sweep_sizes for p in ("f16", "s8", "s4")]

    def graph_of(fn, calls):
        g = torch.cuda.CUDAGraph()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(calls):
                    fn()
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        return g

    def batches(g, calls, min_ms=200.0, nb=5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        reps = max(1, int(min_ms / max(e0.elapsed_time(e1), 1e-3)) + 1)
        out = []
        for _ in range(nb):
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1) * 1e3 / (reps * calls))
        return out, reps * calls

    for prec, n in cases:
        if prec == "f16u":
            A, B = datagen.f16_operands(n, "uniform")
        elif prec == "f16":
            A, B = datagen.f16_operands(n, "normal")
        elif prec == "s8":
            A, B = datagen.s8_operands(n)
        else:
            A, B = datagen.s4_operands(n)
        if prec.startswith("f16"):
            Ad = torch.from_numpy(np.ascontiguousarray(A).view(np.float16)).to(dev)
            Bd = torch.from_numpy(np.ascontiguousarray(B).view(np.float16)).to(dev)
            C = torch.empty((n, n), dtype=torch.float32, device=dev)
            fn = lambda: ptc.matmul_f16(Ad, Bd, out=C)  # noqa: E731
        else:
            Ad, Bd = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
            C = torch.empty((n, n), dtype=torch.int32, device=dev)
            fn = ((lambda: ptc.matmul_s8(Ad, Bd, out=C)) if prec == "s8"
                  else (lambda: ptc.matmul_s4(Ad, Bd, n, out=C)))
        calls = int(max(20, min(200, 2e11 / (2.0 * n ** 3))))
        us, total = batches(graph_of(fn, calls), calls)
        ops = 2.0 * n ** 3
        gpu = {"median_us": statistics.median(us), "min_us": min(us), "batches": len(us),
               "calls_per_batch": total, "tops_median": ops / statistics.median(us) / 1e6,
               "tops_best": ops / min(us) / 1e6}
        flushed = None
        if n <= 2048:
            fc = 20
            both, _ = batches(graph_of(lambda: (flush.zero_(), fn()), fc), fc)
            alone, _ = batches(graph_of(lambda: flush.zero_(), fc), fc)
            t = statistics.median(both) - statistics.median(alone)
            flushed = {"median_us": t, "tops_median": ops / t / 1e6,
                       "how": "512 MiB buffer written before every call; flush time measured alone and subtracted"}
        assert ptc.gemm_poll_device_error() == ptc.PTC_OK
        orc_all = _oracle_time(prec, A, B, n, cores, args.sweep_oracle_seconds)
        orc_one = _oracle_time(prec, A, B, n, 1, args.sweep_oracle_seconds) if n <= 1024 else None
        line = {"sweep": True, "precision": {"f16u": "fp16", "f16": "fp16", "s8": "int8", "s4": "int4"}[prec],
                "N": n, "values": {"f16u": "uniform [-1,1]", "f16": "normal(0,1)/sqrt(K)",
                                   "s8": "uniform [-128,127]", "s4": "uniform [-8,7], packed"}[prec],
                "unit": "TFLOP/s" if prec.startswith("f16") else "TOPS",
                "gpu": gpu, "gpu_l2_flushed": flushed,
                "oracle_all_cores": orc_all, "oracle_single_thread": orc_one,
                "gpu_over_oracle_all_cores": orc_all["seconds"] * 1e6 / gpu["median_us"]}
        print(json.dumps(line), flush=True)
        del Ad, Bd, C
        torch.cuda.empty_cache()


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on bounded row samples."""
    n = args.n
    host = make_inputs(n)
    cores = os.cpu_count() or 1
    secs, _ = oracle_sample(host, n, 1, cores)
    per_step_budget = max(0.05, 150.0 / max(1, args.steps + args.warmup))
    rows = int(max(1, min(n, per_step_budget / max(secs, 1e-4))))
    for _ in range(args.warmup):
        oracle_sample(host, n, rows, cores)
    total_s, total_ops = 0.0, 0.0
    for _ in range(args.steps):
        s, o = oracle_sample(host, n, rows, cores)
        total_s += s
        total_ops += o
    value = total_ops / total_s / 1e12
    sample = f"first {rows} output rows of each of the FP16, INT8 and INT4 N={n} GEMMs per step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16->f64, s8->s64, s4->s64 (CPU oracle)", "data": "synthetic",
        "config": {"workload": f"square GEMM N={n}: FP16 normal/sqrt(K), INT8 and INT4 uniform; "
                               "reference arm = CPU oracle on a row sample", "N": n},
        "cpu_baseline": {"value": value, "unit": "TOPS", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    res = run_ours(args, rank, world, dist)
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world >= 1:
            cpu = cpu_baseline(make_inputs(args.n), args.n, args.cpu_seconds)
        line = {
            "metric": METRIC, "value": res["value"], "unit": "TOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": res["elapsed_ms"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f16->f32, s8->s32, s4->s32", "data": "synthetic",
            "config": {"workload": f"square GEMMs N={args.n}: FP16 (normal/sqrt(K)) -> FP32, "
                                   "INT8 (uniform) -> INT32, packed INT4 (uniform) -> INT32; "
                                   "one step = one GEMM of each",
                       "N": args.n, "l2": "inputs larger than L2 (~1.2 GB per step), no flush",
                       "parallelism": f"replicas x{world}"},
            "batches": res["batches"],
            "per_precision": res["per"], "peak_fractions": res["fractions"], "roofline": res["roofline"],
            "cpu_baseline": cpu,
            "e2e": res["e2e"], "gpu_launches": res["launches"], "clocks": res["clocks"],
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
