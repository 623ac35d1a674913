"""gemm_s8_noalloc: the INT8 GEMM for callers that cannot let a library
allocate device memory (for example an application whose own allocator has
reserved the GPU's memory).  Its workspace is a fixed device array shared by
every call, so the test runs two different problems back to back: the second
call starts with the first call's data still in the array.  Each result must
equal the CPU oracle's exact sums and what gemm_s8 (the pool-allocating entry
point) returns for the same inputs, bit for bit, as all INT8 results in this
suite must.  A further test checks the property the entry point exists for:
once a first call has set it up, calls change neither the device's free
memory nor any allocator's holdings.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import gc

import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    ptc.lib()


def _both(M, N, K, seed):
    A, Bt = datagen.s8_operands(N, seed=seed, m=M, k=K)
    exact = oracle.wrap_s32(oracle.gemm_s8(A, Bt))
    Ad = torch.from_numpy(A).to(DEV)
    Bd = torch.from_numpy(Bt).to(DEV)
    ref = torch.empty((M, N), dtype=torch.int32, device=DEV)
    got = torch.full((M, N), -1, dtype=torch.int32, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    ptc.gemm_s8(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, ref.data_ptr(), N, s)
    before = ptc.ptc_kernel_launch_count()
    ptc.gemm_s8_noalloc(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, got.data_ptr(), N, s)
    launched = ptc.ptc_kernel_launch_count() - before
    torch.cuda.synchronize()
    return got.cpu().numpy(), ref.cpu().numpy(), exact, launched


def test_noalloc_matches_gemm_s8_on_two_calls_in_a_row():
    # call 1: the INT8 workload shape of the study, 2048^3 (16 MiB of workspace)
    got, ref, exact, launched = _both(2048, 2048, 2048, seed=datagen.config_seed("s8", 2048))
    assert launched == 3  # two conversions and the tensor-core kernel
    assert np.array_equal(got, exact)
    assert np.array_equal(got, ref)
    # call 2: a smaller ragged problem over the array the first call filled
    got, ref, exact, _ = _both(300, 520, 208, seed=12345)
    assert np.array_equal(got, exact)
    assert np.array_equal(got, ref)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


def test_noalloc_rejects_problems_beyond_the_scratch():
    M = N = K = 4096  # (M + N) * K * 2 = 64 MiB > 32 MiB
    A = torch.zeros((M, K), dtype=torch.int8, device=DEV)
    Bt = torch.zeros((N, K), dtype=torch.int8, device=DEV)
    C = torch.zeros((M, N), dtype=torch.int32, device=DEV)
    before = ptc.ptc_kernel_launch_count()
    with pytest.raises(ptc.PtcError) as e:
        ptc.gemm_s8_noalloc(M, N, K, A.data_ptr(), K, Bt.data_ptr(), K, C.data_ptr(), N, 0)
    assert e.value.status == ptc.PTC_ERR_INVALID
    assert "static scratch" in str(e.value)
    assert ptc.ptc_kernel_launch_count() == before


def test_noalloc_calls_allocate_nothing():
    """After a first call on the device (the set-up), repeated calls leave the
    device's free memory, torch's caching allocator and the library's
    workspace pool (whose memory would show in the free figure) unchanged."""
    M, N, K = 1024, 1536, 2048
    A, Bt = datagen.s8_operands(N, seed=777, m=M, k=K)
    Ad = torch.from_numpy(A).to(DEV)
    Bd = torch.from_numpy(Bt).to(DEV)
    C = torch.empty((M, N), dtype=torch.int32, device=DEV)
    s = torch.cuda.current_stream().cuda_stream

    def call():
        ptc.gemm_s8_noalloc(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, C.data_ptr(), N, s)

    call()  # set-up and first use of these kernels
    torch.cuda.synchronize()
    gc.collect()  # tensors of earlier tests are freed now, not during the calls
    free0, _ = torch.cuda.mem_get_info()
    reserved0, allocated0 = torch.cuda.memory_reserved(), torch.cuda.memory_allocated()
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    # torch's caching allocator holds the same memory and hands out no more
    # (the library never calls it).
    assert torch.cuda.memory_reserved() == reserved0 and torch.cuda.memory_allocated() <= allocated0
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.mark.parametrize("M,N,K", [(3, 107, 30), (120, 556, 966), (324, 749, 3), (8, 1178, 834), (43, 419, 26),
                                   (1130, 691, 509), (1, 26, 14), (995, 248, 294), (61, 23, 724), (1407, 625, 1196)])
def test_noalloc_random_shapes_exact(M, N, K):
    """Seeded random shapes (after the first-call tests above), pitches padded
    to 16 bytes: bit-exact against the oracle."""
    A, Bt = datagen.s8_operands(N, seed=M * 7 + N * 3 + K, m=M, k=K)
    lda = max(16, (K + 15) // 16 * 16)
    Ap = np.zeros((M, lda), np.int8)
    Ap[:, :K] = A
    Bp = np.zeros((N, lda), np.int8)
    Bp[:, :K] = Bt
    ldc = (N + 3) // 4 * 4
    Ad, Bd = torch.from_numpy(Ap).to(DEV), torch.from_numpy(Bp).to(DEV)
    C = torch.full((M, ldc), -1, dtype=torch.int32, device=DEV)
    ptc.gemm_s8_noalloc(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), lda, C.data_ptr(), ldc,
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy()[:, :N], oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
