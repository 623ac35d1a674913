"""Run one GEMM workload a few times on cuda:0 (a target for profilers).

    python -m precision_tensor_core_gb300.run --prec f16 --n 8192 --reps 2

Inputs are the seeded synthetic operands of the benchmark (FP16 normal/sqrt(K),
INT8 and INT4 uniform).  Nothing is timed or checked here; use bench.py for
numbers and the test suite for parity.  `--prec cublas_f16` runs the same FP16
product through cuBLAS instead (torch.mm with FP32 output), as a library kernel
to profile beside ours; it is not part of the library.  `--tune key=value`
(repeatable) sets a library tuning knob first (ptc_set_tuning), e.g.
`--tune in_ring=0` to profile the separate operand-conversion pass.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--prec", choices=["f16", "s8", "s4", "s8_noalloc", "cublas_f16"], default="f16")
    p.add_argument("--n", type=int, default=8192)
    p.add_argument("--reps", type=int, default=2)
    p.add_argument("--tune", action="append", default=[], metavar="KEY=VALUE")
    a = p.parse_args()

    import torch

    import datagen
    import precision_tensor_core_gb300 as ptc
    from precision_tensor_core_gb300 import build as ptc_build

    ptc_build.build()
    for kv in a.tune:
        key, value = kv.split("=", 1)
        ptc.ptc_set_tuning(key, int(value))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n = a.n
    if a.prec == "cublas_f16":
        A, B = datagen.f16_operands(n, "normal")
        Ad = torch.from_numpy(A.view(np.float16)).to(dev)
        Bd = torch.from_numpy(B.view(np.float16)).to(dev)
        run = lambda: torch.mm(Ad, Bd, out_dtype=torch.float32)
    elif a.prec == "f16":
        A, B = datagen.f16_operands(n, "normal")
        Ad = torch.from_numpy(A.view(np.float16)).to(dev)
        Bd = torch.from_numpy(B.view(np.float16)).to(dev)
        C = torch.empty((n, n), dtype=torch.float32, device=dev)
        run = lambda: ptc.matmul_f16(Ad, Bd, out=C)
    elif a.prec in ("s8", "s8_noalloc"):
        A, B = datagen.s8_operands(n)
        Ad, Bd = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
        C = torch.empty((n, n), dtype=torch.int32, device=dev)
        if a.prec == "s8":
            run = lambda: ptc.matmul_s8(Ad, Bd, out=C)
        else:
            s = torch.cuda.current_stream().cuda_stream
            run = lambda: ptc.gemm_s8_noalloc(n, n, n, Ad.data_ptr(), n, Bd.data_ptr(), n,
                                              C.data_ptr(), n, s)
    else:
        A, B = datagen.s4_operands(n)
        Ad, Bd = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
        C = torch.empty((n, n), dtype=torch.int32, device=dev)
        run = lambda: ptc.matmul_s4(Ad, Bd, n, out=C)
    for _ in range(a.reps):
        run()
    torch.cuda.synchronize()
    status = ptc.gemm_poll_device_error()
    print(f"ran {a.reps} x {a.prec} N={n}: device status {status}")
    sys.exit(0 if status == ptc.PTC_OK else 1)


if __name__ == "__main__":
    main()
