"""GPU parity at extreme shapes: K far beyond the study's 8192 (the integer
routes' fold of FP32 partial sums into int32 runs hundreds of times per tile,
and the exact sum leaves the int32 range, so the result wraps mod 2^32, the
reading the library documents), and very tall and very wide outputs (tile
indices in the hundreds of thousands of rows or columns).  Outputs are checked
against the oracle at sampled coordinates (the corners and the last row and
column included), or exactly where the inputs make every output the same
closed-form value."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, check_f16_sampled, f16_dev, int_dev, sample_coords

pytestmark = pytest.mark.gpu

K_LONG = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


def _wrap(v: int) -> int:
    """Two's-complement int32 of an exact integer."""
    v &= 0xFFFFFFFF
    return v - (1 << 32) if v >= (1 << 31) else v


@pytest.mark.parametrize("a,b", [(-128, -128), (127, -128), (-127, 127)])
def test_int8_k_2_20_constant_wraps(a, b):
    """M = 128, N = 256, K = 2^20 constant operands: every output is K a b,
    outside the int32 range for a b = 16384 and -16256 (wrapped mod 2^32)."""
    M, N, K = 128, 256, K_LONG
    A = torch.full((M, K), a, dtype=torch.int8, device=DEV)
    Bt = torch.full((N, K), b, dtype=torch.int8, device=DEV)
    C = ptc.matmul_s8(A, Bt)
    torch.cuda.synchronize()
    assert torch.all(C == _wrap(K * a * b)).item()


def test_int8_k_2_20_random_sampled():
    M, N, K = 64, 128, K_LONG
    A, Bt = datagen.s8_operands(N, seed=301, m=M, k=K)
    C = ptc.matmul_s8(int_dev(A), int_dev(Bt)).cpu().numpy()
    ii, jj = sample_coords(M, N, 300, seed=302)
    assert np.array_equal(C[ii, jj], oracle.wrap_s32(oracle.gemm_s8_at(A, Bt, ii, jj)))


def test_int4_k_2_20_constant_and_random():
    M, N, K = 128, 256, K_LONG
    # -8 * -8 in every term: 64 K = 2^26, exact (the E4M3 route folds every 8192 K)
    A = torch.full((M, K // 2), 0x88, dtype=torch.uint8, device=DEV)
    Bt = torch.full((N, K // 2), 0x88, dtype=torch.uint8, device=DEV)
    C = ptc.matmul_s4(A, Bt, K)
    torch.cuda.synchronize()
    assert torch.all(C == 64 * K).item()
    M, N = 64, 128
    A, Bt = datagen.s4_operands(N, seed=303, m=M, k=K)
    C = ptc.matmul_s4(int_dev(A), int_dev(Bt), K).cpu().numpy()
    ii, jj = sample_coords(M, N, 300, seed=304)
    assert np.array_equal(C[ii, jj], oracle.wrap_s32(oracle.gemm_s4_at(A, Bt, K, ii, jj)))


def test_f16_k_2_18_sampled():
    """FP16 with K = 262144 (4096 K blocks per tile) against the oracle's
    element-wise bound at sampled outputs."""
    M, N, K = 128, 256, 1 << 18
    A, B = datagen.f16_operands(N, "normal", seed=305, m=M, k=K)
    C = ptc.matmul_f16(f16_dev(A), f16_dev(B)).cpu().numpy()
    check_f16_sampled(C, A, B, n=400)


@pytest.mark.parametrize("prec", ["f16", "s8", "s4"])
def test_tall_output(prec):
    """M = 2^20 rows, N = 40, K = 96: 8192 tile rows in the raster order."""
    M, N, K = 1 << 20, 40, 96
    ii, jj = sample_coords(M, N, 2000, seed=306)
    if prec == "f16":
        A, B = datagen.f16_operands(N, "normal", seed=307, m=M, k=K)
        C = ptc.matmul_f16(f16_dev(A), f16_dev(B)).cpu().numpy()
        check_f16_sampled(C, A, B, n=2000)
    elif prec == "s8":
        A, Bt = datagen.s8_operands(N, seed=308, m=M, k=K)
        C = ptc.matmul_s8(int_dev(A), int_dev(Bt)).cpu().numpy()
        assert np.array_equal(C[ii, jj], oracle.wrap_s32(oracle.gemm_s8_at(A, Bt, ii, jj)))
    else:
        A, Bt = datagen.s4_operands(N, seed=309, m=M, k=K)
        C = ptc.matmul_s4(int_dev(A), int_dev(Bt), K).cpu().numpy()
        assert np.array_equal(C[ii, jj], oracle.wrap_s32(oracle.gemm_s4_at(A, Bt, K, ii, jj)))


@pytest.mark.parametrize("prec", ["f16", "s8"])
def test_wide_output(prec):
    """M = 40, N = 2^20 columns, K = 96: 4096 tile columns."""
    M, N, K = 40, 1 << 20, 96
    ii, jj = sample_coords(M, N, 2000, seed=310)
    if prec == "f16":
        A, B = datagen.f16_operands(N, "normal", seed=311, m=M, k=K)
        C = ptc.matmul_f16(f16_dev(A), f16_dev(B)).cpu().numpy()
        check_f16_sampled(C, A, B, n=2000)
    else:
        A, Bt = datagen.s8_operands(N, seed=312, m=M, k=K)
        C = ptc.matmul_s8(int_dev(A), int_dev(Bt)).cpu().numpy()
        assert np.array_equal(C[ii, jj], oracle.wrap_s32(oracle.gemm_s8_at(A, Bt, ii, jj)))
