"""Build libptc.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each CUDA translation unit compiles in its own nvcc process, in parallel, then
one nvcc link produces ``precision_tensor_core_gb300/libptc.so`` with the CUDA
runtime linked statically (the driver API is reached at run time through the
runtime's entry-point query, so the library loads on machines without a GPU
driver).  ptxas register/shared-memory reports go to ``_build/ptxas.log``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libptc.so")
SOURCES = ["gemm_tc.cu", "convert.cu", "api.cu", "gemm_s8_noalloc.cu", "baseline.cu"]
GENCODE = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}\n{r.stdout}")
    return obj, r.stderr


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "ptc.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        for (obj, log), src in zip(results, SOURCES):
            f.write(f"== {src}\n{log}\n")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), GENCODE, "-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}\n{r.stdout}")
    os.replace(tmp, LIB)
    if verbose:
        sys.stdout.write(open(os.path.join(BUILD, "ptxas.log")).read())
    return LIB


_GEMM_ARGS = ("kind", "B", "epi", "CTAs", "K blocks per stage", "K-split", "tile N", "in-ring")


def _gemm_label(mangled: str) -> str | None:
    """Readable template arguments of a gemm_kernel instantiation."""
    import re
    m = re.search(r"gemm_kernelILNS_4KindE(\d)ELb(\d)ELi(\d)ELi(\d)ELi(\d)ELi(\d)ELi(\d+)ELb(\d)ELi(\d)"
                  r"(?:ELb(\d))?", mangled)
    if not m:
        return None
    kind, bmn, epi, ctas, subk, ks, bn, fu, pairs, gc = m.groups()
    return (f"gemm_kernel<{'F16' if kind == '0' else 'E4M3'}, B {'MN' if bmn == '1' else 'K'}-major, "
            f"{['EPI_F32', 'EPI_INT', 'EPI_F16ACC'][int(epi)]}, CTAS={ctas}, SUBK={subk}, KS={ks}, "
            f"BN={bn}{', in-ring' if fu == '1' else ''}{', 2 pairs, A multicast' if pairs == '2' else ''}"
            f"{', converter warps' if gc == '1' else ''}>")


def ptxas_summary(log_path: str = os.path.join(BUILD, "ptxas.log")) -> str:
    """Markdown table of every kernel in the last build's ptxas report:
    registers, barriers, static shared memory, stack frame and spills."""
    import re
    text = open(log_path).read()
    rows = []
    pat = re.compile(r"Compiling entry function '(\S+)' for '(\w+)'\n"
                     r"ptxas info\s+: Function properties for \S+\n"
                     r"\s+(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads\n"
                     r"ptxas info\s+: Used (\d+) registers(.*)")
    for name, arch, stack, sst, sld, regs, rest in pat.findall(text):
        smem = re.search(r"(\d+) bytes smem", rest)
        label = _gemm_label(name)
        if label is None:
            r = subprocess.run(["c++filt", name], capture_output=True, text=True)
            label = (r.stdout.strip() or name) if r.returncode == 0 else name
            label = label.replace("(anonymous namespace)::", "").replace("ptc::", "")
            label = re.sub(r"^void ", "", re.sub(r"\([^()]*\)$", "", label))
        rows.append((label, int(regs), int(smem.group(1)) if smem else 0, int(stack), int(sst), int(sld)))
    rows.sort()
    out = ["| kernel | registers | static smem (B) | stack (B) | spill stores (B) | spill loads (B) |",
           "|---|---|---|---|---|---|"]
    out += [f"| `{a}` | {b} | {c} | {d} | {e} | {f} |" for a, b, c, d, e, f in rows]
    spilling = sum(1 for r in rows if r[4] or r[5])
    out.append("")
    out.append(f"{len(rows)} kernels, {spilling} with spills.")
    return "\n".join(out)


if __name__ == "__main__":
    if "--ptxas-summary" in sys.argv:
        build(force="--force" in sys.argv)
        print(ptxas_summary())
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
