"""Tuning and size sweeps of the GEMM entry points on cuda:0.

    python -m precision_tensor_core_gb300.tune --mode knobs --n 8192
    python -m precision_tensor_core_gb300.tune --mode sizes --sizes 512,1024,2048,4096,8192
    python -m precision_tensor_core_gb300.tune --mode ab --n 8192 --settings "defaults;pair_in_ring=2"

`baselines` times the paper's kernel families on GB300 (gemm_baseline: WMMA
and mma.sync) beside the library's tcgen05 entry points at each size, and
prints the paper's speedup definitions: each kernel over the WMMA kernel of
its precision, and over the FP16 WMMA kernel.
`variants` times gemm_f16_f16acc against gemm_f16, gemm_s8_b_rowmajor (B
row-major, read MN-major) against gemm_s8 (B column-major), and
gemm_s8_scaled / gemm_s4_scaled (each output type) against gemm_s8 / gemm_s4,
at one size.
`knobs` times gemm_f16 / gemm_s8 / gemm_s4 at one size under each setting of
the library's tuning knobs (ptc_set_tuning: CTA pairs, pair ring stage depth,
tail split, K-split clusters, programmatic launches, raster group, L2 eviction
policy, INT fold length), one knob at a time from the defaults: the ablation
that shows the defaults are a local optimum.  `launch` compares launch shapes
at small sizes (K-split clusters of 2, 4, 8 CTAs, programmatic launches on
and off), reporting the median of 7 graph replays and the launch record
(grid CTAs, CTAs per tile's K range) of each; `--in-ring 0,1` repeats the
integer rows with the operand conversion as a separate pass and inside the
GEMM kernel.  `sizes` times the three
entry points at each size with the library defaults.  `cublas` times gemm_f16
against cuBLAS on the same FP16 operands (torch.mm with FP32 output, and with
FP16 output), or with `--prec s8` gemm_s8 against cuBLAS's INT8 GEMM
(torch._int_mm, int32 output, whose result it first compares with ours),
interleaved in one process so that both see the same clocks and power state:
10 rounds of one CUDA-graph replay each, then ~1 s of back-to-back replays per
kernel.

`ab` compares whole settings of the tuning knobs (`--settings`, separated by
semicolons, each a comma-separated list of key=value; "defaults" is the
library's defaults) in one process: `--rounds` rounds, each running every
setting in a shuffled order for every precision of `--precs`, with the clock
record on; it prints the median per call, the throughput, the median SM clock
the GEMM kernels ran at and the throughput per GHz of that clock.

Calls are captured in a CUDA graph (`--graph`, default on) and the graph is
replayed, so that the host-side cost of a Python call does not hide the GPU
time at small sizes; times are CUDA-event times of the replay divided by the
calls in it.  Inputs are the benchmark's seeded operands.  These are tuning
measurements, not the benchmark's reported numbers.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULTS = {"cta_pair": 0, "group_m": 8, "l2_hint": 0, "s8_chunk_kb": 16, "s4_chunk_kb": 64, "tail_split": 1,
            "split_min_kb": 64, "pair_stage_kb": 2, "ksplit": 0, "pdl": 1, "tile_n": 0, "in_ring": 1,
            "pair_in_ring": 0, "multicast": 0, "conv_fused": 0}
KNOBS = {"cta_pair": [1, 2], "pair_stage_kb": [1], "tail_split": [0], "split_min_kb": [32, 128],
         "group_m": [4, 16, 32], "l2_hint": [1, 2, 3], "s8_chunk_kb": [4, 8], "s4_chunk_kb": [2, 8, 16, 128],
         "ksplit": [1, 2, 4, 8], "pdl": [0], "tile_n": [64, 128, 256], "in_ring": [0]}
# `launch` mode: launch-shape settings compared at small sizes, each timed as
# the median of 7 replays of a CUDA graph of back-to-back calls.
LAUNCH_SETTINGS = [("256-wide, plain launches", {"tile_n": 256, "ksplit": 1, "pdl": 0}),
                   ("256-wide", {"tile_n": 256, "ksplit": 1, "pdl": 1}),
                   ("256-wide, K-split by size", {"tile_n": 256, "ksplit": 0, "pdl": 1}),
                   ("K-split 2", {"tile_n": 256, "ksplit": 2, "pdl": 1}),
                   ("K-split 4", {"tile_n": 256, "ksplit": 4, "pdl": 1}),
                   ("K-split 8", {"tile_n": 256, "ksplit": 8, "pdl": 1}),
                   ("128-wide", {"tile_n": 128, "ksplit": 1, "pdl": 1}),
                   ("128-wide, K-split 2", {"tile_n": 128, "ksplit": 2, "pdl": 1}),
                   ("128-wide, K-split 4", {"tile_n": 128, "ksplit": 4, "pdl": 1}),
                   ("64-wide", {"tile_n": 64, "ksplit": 1, "pdl": 1}),
                   ("64-wide, K-split 2", {"tile_n": 64, "ksplit": 2, "pdl": 1}),
                   ("64-wide, K-split 4", {"tile_n": 64, "ksplit": 4, "pdl": 1}),
                   ("defaults", {"tile_n": 0, "ksplit": 0, "pdl": 1})]


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--mode", choices=["knobs", "sizes", "variants", "baselines", "cublas", "launch", "ab"],
                   default="sizes")
    p.add_argument("--settings", default="defaults", help="ab mode: knob settings separated by ';'")
    p.add_argument("--precs", default="f16,s8,s4", help="ab mode: precisions")
    p.add_argument("--rounds", type=int, default=10, help="ab mode: shuffled rounds")
    p.add_argument("--n", type=int, default=8192)
    p.add_argument("--sizes", default="512,1024,2048,4096,8192")
    p.add_argument("--calls", type=int, default=0, help="calls per timing (0: by size)")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--json", default="")
    p.add_argument("--only", default="", help="comma-separated knob names to sweep (default: all)")
    p.add_argument("--in-ring", default="1", help="launch mode: in_ring settings of the integer rows")
    p.add_argument("--prec", default="f16", choices=["f16", "s8"],
                   help="cublas mode: FP16 (torch.mm) or INT8 (torch._int_mm, int32 C)")
    a = p.parse_args()

    import torch

    import datagen
    import precision_tensor_core_gb300 as ptc
    from precision_tensor_core_gb300 import build as ptc_build

    ptc_build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    def operands(n):
        A, B = datagen.f16_operands(n, "normal")
        A8, B8 = datagen.s8_operands(n)
        A4, B4 = datagen.s4_operands(n)
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        return {"f16": (t(A.view(np.float16)), t(B.view(np.float16)),
                        torch.empty((n, n), dtype=torch.float32, device=dev)),
                "s8": (t(A8), t(B8), torch.empty((n, n), dtype=torch.int32, device=dev)),
                "s4": (t(A4), t(B4), torch.empty((n, n), dtype=torch.int32, device=dev))}

    def call(prec, ops, n):
        A, B, C = ops[prec]
        if prec == "f16":
            return lambda: ptc.matmul_f16(A, B, out=C)
        if prec == "s8":
            return lambda: ptc.matmul_s8(A, B, out=C)
        return lambda: ptc.matmul_s4(A, B, n, out=C)

    def time_ms(fn, calls):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g = None
        if not a.no_graph:
            try:
                g = torch.cuda.CUDAGraph()
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    with torch.cuda.graph(g, stream=s):
                        for _ in range(calls):
                            fn()
                torch.cuda.current_stream().wait_stream(s)
                g.replay()
                torch.cuda.synchronize()
            except Exception as exc:  # capture unsupported for this call: time eagerly
                print(f"  (graph capture failed: {exc}; timing eager calls)", flush=True)
                torch.cuda.synchronize()
                g = None
        e0.record()
        if g is not None:
            g.replay()
        else:
            for _ in range(calls):
                fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / calls

    def measure(n, ops):
        calls = a.calls or max(4, min(200, int(2e13 / (2.0 * n ** 3))))
        out = {}
        for prec in ("f16", "s8", "s4"):
            ms = time_ms(call(prec, ops, n), calls)
            out[prec] = {"ms": ms, "tops": 2.0 * n ** 3 / (ms * 1e-3) / 1e12}
        return out

    results = {}
    if a.mode == "ab":
        import random
        import statistics

        settings = []
        for text in a.settings.split(";"):
            text = text.strip()
            kv = {} if text in ("", "defaults") else dict(x.split("=") for x in text.split(","))
            settings.append((text or "defaults", {k: int(v) for k, v in kv.items()}))
        precs = a.precs.split(",")
        ops = operands(a.n)
        calls = a.calls or max(4, min(200, int(2e13 / (2.0 * a.n ** 3))))
        fam = {"f16": 0, "s8": 1, "s4": 2}
        us = {(i, p): [] for i in range(len(settings)) for p in precs}
        mhz = {(i, p): [] for i in range(len(settings)) for p in precs}
        for r in range(a.rounds):
            order = list(range(len(settings)))
            random.Random(r).shuffle(order)
            for i in order:
                for k, v in settings[i][1].items():
                    ptc.ptc_set_tuning(k, v)
                for prec in precs:
                    ptc.ptc_clock_probe_read()
                    ptc.ptc_set_tuning("clock_probe", 1)
                    ms = time_ms(call(prec, ops, a.n), calls)
                    ptc.ptc_set_tuning("clock_probe", 0)
                    cyc, ns, _ = ptc.ptc_clock_probe_read()
                    us[(i, prec)].append(ms * 1e3)
                    mhz[(i, prec)].append(1e3 * cyc[fam[prec]] / max(1, ns[fam[prec]]))
                for k, v in DEFAULTS.items():
                    ptc.ptc_set_tuning(k, v)
        print(f"{'N':>6} {'setting':>28} {'prec':>5} {'us/call':>9} {'TOPS':>8} {'MHz':>6} {'TOPS/GHz':>9}")
        for i, (name, _) in enumerate(settings):
            results[name] = {}
            for prec in precs:
                u = statistics.median(us[(i, prec)])
                m = statistics.median(mhz[(i, prec)])
                tops = 2.0 * a.n ** 3 / (u * 1e-6) / 1e12
                results[name][prec] = {"us": u, "tops": tops, "mhz": m, "rounds": us[(i, prec)]}
                print(f"{a.n:>6} {name:>28} {prec:>5} {u:>9.1f} {tops:>8.1f} {m:>6.0f} {tops / m * 1e3:>9.1f}",
                      flush=True)
    elif a.mode == "launch":
        import statistics

        def graph_median_us(fn, calls):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    for _ in range(calls):
                        fn()
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            v = []
            for _ in range(7):
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize()
                v.append(e0.elapsed_time(e1) / calls * 1000.0)
            return statistics.median(v)

        print("each entry: microseconds per call (grid CTAs / CTAs per K range / tile width)")
        print(f"{'N':>6} {'prec':>4} " + " ".join(f"{name:>26}" for name, _ in LAUNCH_SETTINGS))
        for n in [int(x) for x in a.sizes.split(",")]:
            ops = operands(n)
            calls = a.calls or max(20, min(200, int(2e11 / (2.0 * n ** 3))))
            results[str(n)] = {}
            rows = [("f16", 1)] + [(p, int(r)) for p in ("s8", "s4") for r in a.in_ring.split(",")]
            for prec, ring in rows:
                row = {}
                for name, kv in LAUNCH_SETTINGS:
                    for k, v in kv.items():
                        ptc.ptc_set_tuning(k, v)
                    ptc.ptc_set_tuning("in_ring", ring)
                    us = graph_median_us(call(prec, ops, n), calls)
                    grid, _, ks, bn = ptc.ptc_last_launch()
                    row[name] = {"us": us, "grid": grid, "ksplit": ks, "tile_n": bn,
                                 "conversion": ptc.ptc_last_conversion()}
                for k, v in DEFAULTS.items():
                    ptc.ptc_set_tuning(k, v)
                label = prec if prec == "f16" else f"{prec}/r{ring}"
                results[str(n)][label] = row
                print(f"{n:>6} {label:>5} " + " ".join(
                    f"{r['us']:>10.2f} ({r['grid']:>3}/{r['ksplit']}/{r['tile_n']:>3})" for r in row.values()),
                    flush=True)
    elif a.mode == "cublas":
        import statistics
        n = a.n
        if a.prec == "f16":
            A, B, C = operands(n)["f16"]
            fns = {"gemm_f16 (FP32 C)": lambda: ptc.matmul_f16(A, B, out=C),
                   "cuBLAS torch.mm (FP32 C)": lambda: torch.mm(A, B, out_dtype=torch.float32),
                   "cuBLAS torch.mm (FP16 C)": lambda: torch.mm(A, B)}
        else:
            # INT8 -> int32 (B column-major: the K x N view of N rows of K).
            A, Bt, C = operands(n)["s8"]
            fns = {"gemm_s8 (int32 C)": lambda: ptc.matmul_s8(A, Bt, out=C)}
            try:
                ref = torch._int_mm(A, Bt.t())
                torch.cuda.synchronize()
                ptc.matmul_s8(A, Bt, out=C)
                torch.cuda.synchronize()
                print("torch._int_mm equals gemm_s8:", bool(torch.equal(ref, C)), flush=True)
                del ref
                fns["cuBLAS torch._int_mm"] = lambda: torch._int_mm(A, Bt.t())
            except RuntimeError as exc:
                print(f"torch._int_mm unavailable here: {exc}", flush=True)
        calls = a.calls or 20
        graphs = {}
        for k, fn in fns.items():
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    for _ in range(calls):
                        fn()
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            graphs[k] = g
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        rounds = {k: [] for k in graphs}
        for _ in range(10):
            for k, g in graphs.items():
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize()
                rounds[k].append(2.0 * n ** 3 / (e0.elapsed_time(e1) / calls * 1e-3) / 1e12)
        print(f"{'kernel':>26} {'interleaved median':>19} {'min':>8} {'max':>8} {'sustained ~1 s':>15}")
        for k, g in graphs.items():
            reps = max(1, int(1000.0 / (calls * 0.7)))
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            sus = 2.0 * n ** 3 * calls * reps / (e0.elapsed_time(e1) * 1e-3) / 1e12
            v = rounds[k]
            results[k] = {"median": statistics.median(v), "min": min(v), "max": max(v), "sustained": sus}
            print(f"{k:>26} {statistics.median(v):>19.1f} {min(v):>8.1f} {max(v):>8.1f} {sus:>15.1f}", flush=True)
    elif a.mode == "baselines":
        base = {"fp16_wmma": ("f16", ptc.PTC_BASELINE_F16_WMMA), "fp16_ptx_mma": ("f16", ptc.PTC_BASELINE_F16_MMA),
                "int8_wmma": ("s8", ptc.PTC_BASELINE_S8_WMMA), "int8_ptx_mma_k32": ("s8", ptc.PTC_BASELINE_S8_MMA),
                "int4_wmma": ("s4", ptc.PTC_BASELINE_S4_WMMA), "int4_ptx_mma_k64": ("s4", ptc.PTC_BASELINE_S4_MMA),
                "fp16_ptx_ldmatrix": ("f16", ptc.PTC_BASELINE_F16_LDMATRIX),
                "int8_ptx_ldm_k32": ("s8", ptc.PTC_BASELINE_S8_LDMATRIX),
                "int4_ptx_ldm_k64": ("s4", ptc.PTC_BASELINE_S4_LDMATRIX)}
        print(f"{'N':>6} {'kernel':>18} {'ms':>10} {'TOPS':>9} {'vs same-prec WMMA':>18} {'vs FP16 WMMA':>13}")
        for n in [int(x) for x in a.sizes.split(",")]:
            ops = operands(n)
            calls = a.calls or max(2, min(50, int(5e11 / (2.0 * n ** 3))))
            row = {}
            for name, (prec, v) in base.items():
                A, B, C = ops[prec]
                # the stream is read at call time, so that graph capture sees the launch
                fn = (lambda A=A, B=B, C=C, v=v: ptc.gemm_baseline(
                    v, n, n, n, A.data_ptr(), n, B.data_ptr(), n, C.data_ptr(), n,
                    torch.cuda.current_stream().cuda_stream))
                row[name] = time_ms(fn, calls)
            for prec, name in (("f16", "tcgen05 gemm_f16"), ("s8", "tcgen05 gemm_s8"), ("s4", "tcgen05 gemm_s4")):
                row[name] = time_ms(call(prec, ops, n), calls)
            wmma_of = {"fp16": "fp16_wmma", "int8": "int8_wmma", "int4": "int4_wmma",
                       "tcgen05 gemm_f16": "fp16_wmma", "tcgen05 gemm_s8": "int8_wmma", "tcgen05 gemm_s4": "int4_wmma"}
            results[str(n)] = {}
            for name, ms in row.items():
                ref = wmma_of.get(name, wmma_of.get(name.split("_")[0], "fp16_wmma"))
                sp_same = row[ref] / ms
                sp_f16 = row["fp16_wmma"] / ms
                results[str(n)][name] = {"ms": ms, "tops": 2.0 * n ** 3 / (ms * 1e-3) / 1e12,
                                         "speedup_vs_same_precision_wmma": sp_same, "speedup_vs_fp16_wmma": sp_f16}
                print(f"{n:>6} {name:>18} {ms:>10.4f} {2.0 * n ** 3 / (ms * 1e-3) / 1e12:>9.1f} {sp_same:>17.2f}x"
                      f" {sp_f16:>12.2f}x", flush=True)
    elif a.mode == "variants":
        n = a.n
        ops = operands(n)
        sa = torch.rand(n, device=dev) + 0.5
        sb = torch.rand(n, device=dev) + 0.5
        calls = a.calls or max(4, min(200, int(2e13 / (2.0 * n ** 3))))
        print(f"{'call':>24} {'TOPS':>8} {'ms':>8}")
        A, B, C = ops["f16"]
        Ch = torch.empty((n, n), dtype=torch.float16, device=dev)
        for key, fn in (("gemm_f16 -> f32", call("f16", ops, n)),
                        ("gemm_f16_f16acc -> f16", lambda: ptc.matmul_f16_f16acc(A, B, out=Ch))):
            ms = time_ms(fn, calls)
            results[key] = {"ms": ms, "tops": 2.0 * n ** 3 / (ms * 1e-3) / 1e12}
            print(f"{key:>24} {results[key]['tops']:>8.1f} {ms:>8.4f}", flush=True)
        A8, B8, C8 = ops["s8"]
        B8_kn = B8.t().contiguous()  # the same B, row-major (K x N)
        for key, fn in (("gemm_s8 (B col-major)", call("s8", ops, n)),
                        ("gemm_s8_b_rowmajor", lambda: ptc.gemm_s8_b_rowmajor(
                            n, n, n, A8.data_ptr(), n, B8_kn.data_ptr(), n, C8.data_ptr(), n,
                            torch.cuda.current_stream().cuda_stream))):
            ms = time_ms(fn, calls)
            results[key] = {"ms": ms, "tops": 2.0 * n ** 3 / (ms * 1e-3) / 1e12}
            print(f"{key:>24} {results[key]['tops']:>8.1f} {ms:>8.4f}", flush=True)
        for prec in ("s8", "s4"):
            A, B, C = ops[prec]
            rows = [("int32", call(prec, ops, n))]
            for name, dt in (("f32", torch.float32), ("bf16", torch.bfloat16), ("f16", torch.float16)):
                Co = torch.empty((n, n), dtype=dt, device=dev)
                if prec == "s8":
                    rows.append((name, lambda Co=Co: ptc.matmul_s8_scaled(A, B, sa, sb, out=Co)))
                else:
                    rows.append((name, lambda Co=Co: ptc.matmul_s4_scaled(A, B, n, sa, sb, out=Co)))
            for name, fn in rows:
                ms = time_ms(fn, calls)
                key = f"gemm_{prec}{'' if name == 'int32' else '_scaled'} -> {name}"
                results[key] = {"ms": ms, "tops": 2.0 * n ** 3 / (ms * 1e-3) / 1e12}
                print(f"{key:>24} {results[key]['tops']:>8.1f} {ms:>8.4f}", flush=True)
    elif a.mode == "sizes":
        for k, v in DEFAULTS.items():
            ptc.ptc_set_tuning(k, v)
        print(f"{'N':>6} {'FP16 TFLOP/s':>13} {'INT8 TOPS':>10} {'INT4 TOPS':>10}   (ms per call)")
        for n in [int(x) for x in a.sizes.split(",")]:
            r = measure(n, operands(n))
            results[str(n)] = r
            print(f"{n:>6} {r['f16']['tops']:>13.1f} {r['s8']['tops']:>10.1f} {r['s4']['tops']:>10.1f}"
                  f"   ({r['f16']['ms']:.4f} / {r['s8']['ms']:.4f} / {r['s4']['ms']:.4f})", flush=True)
    else:
        ops = operands(a.n)
        chosen = [k for k in KNOBS if not a.only or k in a.only.split(",")]
        settings = [("defaults", None, None)] + [(k, k, v) for k in chosen for v in KNOBS[k]]
        print(f"{'setting':>18} {'FP16 TFLOP/s':>13} {'INT8 TOPS':>10} {'INT4 TOPS':>10} {'sum ms':>8}")
        for label, key, val in settings:
            for k, v in DEFAULTS.items():
                ptc.ptc_set_tuning(k, v)
            name = "defaults" if key is None else f"{key}={val}"
            if key is not None:
                ptc.ptc_set_tuning(key, val)
            r = measure(a.n, ops)
            results[name] = r
            total = sum(r[p]["ms"] for p in r)
            print(f"{name:>18} {r['f16']['tops']:>13.1f} {r['s8']['tops']:>10.1f} {r['s4']['tops']:>10.1f}"
                  f" {total:>8.3f}", flush=True)
        for k, v in DEFAULTS.items():
            ptc.ptc_set_tuning(k, v)
    status = ptc.gemm_poll_device_error()
    if a.json:
        with open(a.json, "w") as f:
            json.dump(results, f, indent=1)
    sys.exit(0 if status == ptc.PTC_OK else 1)


if __name__ == "__main__":
    main()
