"""Helpers shared by the GPU parity tests: device upload of seeded operands and
element-by-element comparison with the oracle."""
import numpy as np
import torch

import oracle

DEV = torch.device("cuda", 0)


def f16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(DEV)


def int_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def check_f16(C_gpu: np.ndarray, A: np.ndarray, B: np.ndarray):
    """Full element-wise FP16 check against the oracle (tolerance of the spec:
    |C - Cref| <= 1e-3 * sum|a b| + 1e-6 per element, Frobenius <= 1e-4)."""
    Cref, S = oracle.gemm_f16(A, B)
    ok, ratio, ferr = oracle.f16_tolerance_ok(C_gpu, Cref, S)
    assert ok, f"FP16 mismatch: max err/bound = {ratio:.3g}, rel. Frobenius = {ferr:.3g}"
    return ratio, ferr


def sample_coords(M, N, n, seed=0):
    rng = np.random.default_rng(seed)
    ii = rng.integers(0, M, size=n)
    jj = rng.integers(0, N, size=n)
    # always include the four corners and the last row / column
    ii = np.concatenate([ii, [0, 0, M - 1, M - 1]])
    jj = np.concatenate([jj, [0, N - 1, 0, N - 1]])
    return ii, jj


def check_f16_sampled(C_gpu: np.ndarray, A: np.ndarray, B: np.ndarray, n=2000):
    """The FP16 acceptance test of check_f16 on sampled elements (plus the four
    corners): the per-element bound at every sample, and the relative
    Frobenius bound over the samples."""
    M, N = C_gpu.shape
    ii, jj = sample_coords(M, N, n)
    c, s = oracle.gemm_f16_at(A, B, ii, jj)
    got = C_gpu[ii, jj].astype(np.float64)
    ok, ratio, ferr = oracle.f16_tolerance_ok(got, c, s)
    assert ok, f"FP16 sampled mismatch: max err/bound = {ratio:.3g}, rel. Frobenius = {ferr:.3g}"
    return ratio


def check_f16_rows(C_gpu_rows: np.ndarray, A: np.ndarray, B: np.ndarray, r0: int, r1: int,
                   c0: int = 0, c1: int | None = None):
    """The full FP16 acceptance test on the block rows r0..r1-1, columns
    c0..c1-1 of C (the oracle computes just that block)."""
    c1 = B.shape[1] if c1 is None else c1
    Cref, S = oracle.gemm_f16(A[r0:r1], np.ascontiguousarray(B[:, c0:c1]))
    ok, ratio, ferr = oracle.f16_tolerance_ok(C_gpu_rows, Cref, S)
    assert ok, (f"FP16 mismatch in rows {r0}..{r1}, columns {c0}..{c1}: max err/bound = {ratio:.3g}, "
                f"rel. Frobenius = {ferr:.3g}")
    return ratio, ferr
