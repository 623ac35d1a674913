"""GPU parity of gemm_f16_f16acc (FP16 operands, FP16 accumulators, FP16 C).

Exact where FP16 accumulation is exact (permutation operands, the pages'
m16n8k16 worked example); elsewhere within the bound that follows from one
binary16 rounding of the running sum per 16-deep tensor-core step:
|C - sum| <= (ceil(K/16) + 1) * 2^-10 * sum|a b| + ceil(K/16) * 2^-24,
where 2^-10 is twice the binary16 unit roundoff (allowing truncation as well
as rounding to nearest) and the last term covers binary16 underflow."""
import math
import os

import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, f16_dev, sample_coords

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.fixture(params=[1, 2], ids=["cta1", "cta2"])
def cta_mode(request):
    ptc.ptc_set_tuning("cta_pair", request.param)
    yield request.param
    ptc.ptc_set_tuning("cta_pair", 0)


def bound(S, K):
    steps = math.ceil(K / 16)
    return (steps + 1) * 2.0 ** -10 * S + steps * 2.0 ** -24


def run(A, B):
    C = ptc.matmul_f16_f16acc(f16_dev(A), f16_dev(B))
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.float64)


def test_permutation_exact(cta_mode):
    M, K, N = 256, 384, 264
    perm = np.random.default_rng(3).permutation(K)[:M]
    A = np.zeros((M, K), np.float16)
    A[np.arange(M), perm] = 1
    B = np.random.default_rng(4).uniform(-100, 100, size=(K, N)).astype(np.float16)
    C = run(A.view(np.uint16), B.view(np.uint16))
    assert np.array_equal(C, B.astype(np.float64)[perm])


def test_worked_example(golden_dir):
    from tests.test_oracle_pins import _read_golden
    g = _read_golden(os.path.join(golden_dir, "mma_lab_m16n8k16.txt"))
    M, N, K = g["shape"]
    B = np.array([[8 * r + c + 1 for c in range(N)] for r in range(K)], dtype=np.float16)
    C = run(np.eye(M, K, dtype=np.float16).view(np.uint16), B.view(np.uint16))
    for (r, c, v) in g["point"]:
        assert C[r, c] == v
    C2 = run(np.ascontiguousarray(np.eye(M, K, dtype=np.float16)[::-1]).view(np.uint16), B.view(np.uint16))
    assert C2[0].tolist() == g["reversed_row0"]


@pytest.mark.parametrize("M,N,K", [(1, 8, 1), (31, 40, 17), (129, 264, 200), (300, 520, 512),
                                   (512, 512, 512)])
def test_within_fp16_accumulation_bound(M, N, K, cta_mode):
    A, B = datagen.f16_operands(N, "uniform", seed=M * 3 + K, m=M, k=K)
    A = np.pad(A, ((0, 0), (0, (-K) % 8)))
    B = np.pad(B, ((0, 0), (0, (-N) % 8)))
    Cd = torch.empty((M, max(8, (N + 7) // 8 * 8)), dtype=torch.float16, device=DEV)
    Ad, Bd = f16_dev(A), f16_dev(B)
    ptc.gemm_f16_f16acc(M, N, K, Ad.data_ptr(), Ad.shape[1], Bd.data_ptr(), Bd.shape[1],
                        Cd.data_ptr(), Cd.shape[1], 0)
    torch.cuda.synchronize()
    C = Cd.cpu().numpy().astype(np.float64)[:, :N]
    Cref, S = oracle.gemm_f16(A[:, :K], B[:K, :N])
    assert np.all(np.abs(C - Cref) <= bound(S, K))
    # and far closer than the worst case on these random-sign inputs
    assert np.linalg.norm(C - Cref) <= 0.1 * np.linalg.norm(bound(S, K))


def test_full_size_sampled():
    n = 8192
    A, B = datagen.f16_operands(n, "normal")
    C = run(A, B)
    assert np.all(np.isfinite(C))
    ii, jj = sample_coords(n, n, 2000)
    c, s = oracle.gemm_f16_at(A, B, ii, jj)
    assert np.all(np.abs(C[ii, jj] - c) <= bound(s, n))


def test_guard_bands_and_zero_k():
    M, N, K = 130, 264, 96
    sentinel = 0x7E7E
    Cd = torch.full((M + 2, 272), sentinel, dtype=torch.int16, device=DEV)
    A, B = datagen.f16_operands(N, "uniform", m=M, k=K)
    Ad, Bd = f16_dev(A), f16_dev(B)
    ptc.gemm_f16_f16acc(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, Cd.data_ptr(), 272, 0)
    torch.cuda.synchronize()
    c = Cd.cpu().numpy()
    assert np.all(c[:, N:] == sentinel) and np.all(c[M:, :] == sentinel)
    Cref, S = oracle.gemm_f16(A, B)
    got = c[:M, :N].view(np.float16).astype(np.float64)
    assert np.all(np.abs(got - Cref) <= bound(S, K))
    ptc.gemm_f16_f16acc(M, N, 0, 0, 0, 0, 0, Cd.data_ptr(), 272, 0)
    torch.cuda.synchronize()
    c = Cd.cpu().numpy()
    assert np.all(c[:M, :N] == 0) and np.all(c[:, N:] == sentinel)
