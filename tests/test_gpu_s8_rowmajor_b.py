"""GPU parity of gemm_s8_b_rowmajor (INT8 with B given row-major, K x N): the
tensor cores read the converted B as an MN-major operand.  Bit-exact against
the oracle (which takes B column-major, so the tests pass it B transposed)."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, int_dev, sample_coords

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    ptc.ptc_set_tuning("cta_pair", 0)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.fixture(params=[1, 2], ids=["cta1", "cta2"])
def cta_mode(request):
    ptc.ptc_set_tuning("cta_pair", request.param)
    yield request.param
    ptc.ptc_set_tuning("cta_pair", 0)


def _pad(a, mult):
    rows, cols = a.shape
    w = max(mult, (cols + mult - 1) // mult * mult)
    out = np.zeros((rows, w), dtype=a.dtype)
    out[:, :cols] = a
    return out


def _run(A, B_kn, M, N, K):
    """A (M x >=K), B_kn (K x >=N) int8 row-major, padded pitches."""
    Ad, Bd = int_dev(A), int_dev(B_kn)
    Cd = torch.full((M, (N + 3) // 4 * 4), 0x7eadbeef, dtype=torch.int32, device=DEV)
    ptc.gemm_s8_b_rowmajor(M, N, K, Ad.data_ptr(), A.shape[1], Bd.data_ptr(), B_kn.shape[1], Cd.data_ptr(),
                           Cd.shape[1], torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return Cd.cpu().numpy()[:, :N]


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (33, 31, 65), (200, 300, 160), (257, 513, 1000), (300, 520, 2048),
                                   (136, 264, 4160)])
def test_rowmajor_b_ragged(M, N, K, cta_mode):
    A, Bt = datagen.s8_operands(N, seed=M * 17 + K, m=M, k=K)
    B_kn = np.ascontiguousarray(Bt.T)
    C = _run(_pad(A, 16), _pad(B_kn, 16), M, N, K)
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


def test_rowmajor_b_matches_gemm_s8_at_2048():
    A, Bt = datagen.s8_operands(2048)
    C = _run(A, np.ascontiguousarray(Bt.T), 2048, 2048, 2048)
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    assert np.array_equal(C, ptc.matmul_s8(int_dev(A), int_dev(Bt)).cpu().numpy())


def test_rowmajor_b_8192_sampled():
    A, Bt = datagen.s8_operands(8192)
    C = _run(A, np.ascontiguousarray(Bt.T), 8192, 8192, 8192)
    ii, jj = sample_coords(8192, 8192, 3000)
    assert np.array_equal(C[ii, jj], oracle.wrap_s32(oracle.gemm_s8_at(A, Bt, ii, jj)))


def test_rowmajor_b_zero_k():
    Cd = torch.full((40, 44), 7, dtype=torch.int32, device=DEV)
    ptc.gemm_s8_b_rowmajor(40, 41, 0, 0, 0, 0, 0, Cd.data_ptr(), 44, 0)
    torch.cuda.synchronize()
    assert (Cd[:, :41] == 0).all() and (Cd[:, 41:] == 7).all()
