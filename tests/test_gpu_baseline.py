"""GPU parity of the paper's kernel families on GB300 (gemm_baseline):
WMMA and mma.sync kernels for FP16, INT8 and INT4, with hand-packed and
ldmatrix fragments, against the oracle (INT bit-exact, FP16 within the FP16
tolerance)."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, check_f16, f16_dev, int_dev

pytestmark = pytest.mark.gpu

VARIANTS = {
    "f16_wmma": ptc.PTC_BASELINE_F16_WMMA, "f16_mma": ptc.PTC_BASELINE_F16_MMA,
    "s8_wmma": ptc.PTC_BASELINE_S8_WMMA, "s8_mma": ptc.PTC_BASELINE_S8_MMA,
    "s4_wmma": ptc.PTC_BASELINE_S4_WMMA, "s4_mma": ptc.PTC_BASELINE_S4_MMA,
    "f16_ldmatrix": ptc.PTC_BASELINE_F16_LDMATRIX, "s8_ldmatrix": ptc.PTC_BASELINE_S8_LDMATRIX,
    "s4_ldmatrix": ptc.PTC_BASELINE_S4_LDMATRIX,
}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


def run(variant, M, N, K, seed):
    v = VARIANTS[variant]
    prec = variant.split("_")[0]
    if prec == "f16":
        A, B = datagen.f16_operands(N, "normal", seed=seed, m=M, k=K)
        Ad, Bd = f16_dev(A), f16_dev(B)
        C = torch.empty((M, N), dtype=torch.float32, device=DEV)
        ptc.gemm_baseline(v, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, C.data_ptr(), N, 0)
        torch.cuda.synchronize()
        check_f16(C.cpu().numpy(), A, B)
        return
    if prec == "s8":
        A, Bt = datagen.s8_operands(N, seed=seed, m=M, k=K)
        ref = oracle.gemm_s8(A, Bt)
        lda = ldb = K
    else:
        A, Bt = datagen.s4_operands(N, seed=seed, m=M, k=K)
        ref = oracle.gemm_s4(A, Bt, K)
        lda = ldb = K
    Ad, Bd = int_dev(A), int_dev(Bt)
    C = torch.empty((M, N), dtype=torch.int32, device=DEV)
    ptc.gemm_baseline(v, M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, C.data_ptr(), N, 0)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(ref))


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("M,N,K", [(32, 64, 128), (256, 512, 512), (1024, 1024, 1024), (96, 192, 2048)])
def test_baseline_matches_oracle(variant, M, N, K):
    run(variant, M, N, K, seed=M + N + K)


def test_baseline_rejects_untiled_shapes():
    C = torch.empty((64, 64), dtype=torch.int32, device=DEV)
    A = torch.zeros((64, 128), dtype=torch.int8, device=DEV)
    for M, N, K in [(33, 64, 128), (32, 65, 128), (32, 64, 100)]:
        with pytest.raises(ptc.PtcError) as e:
            ptc.gemm_baseline(ptc.PTC_BASELINE_S8_MMA, M, N, K, A.data_ptr(), 128, A.data_ptr(), 128,
                              C.data_ptr(), 64, 0)
        assert e.value.status == ptc.PTC_ERR_INVALID
