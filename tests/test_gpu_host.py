"""GPU parity of the host-buffer entry points (gemm_*_host): host operands and
result, copies pipelined over row panels inside the library.  Checked against
the oracle (INT bit-exact, FP16 within the FP16 tolerance) and, for the
integer routes, bit-for-bit against the device-buffer entry points."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, check_f16, check_f16_sampled, sample_coords

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


def pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (200, 264, 160), (300, 520, 512), (1000, 1024, 777)])
def test_host_small_shapes(M, N, K):
    K16 = K + (-K) % 8
    A, B = datagen.f16_operands(N, "uniform", seed=M + K, m=M, k=K16)
    A[:, K:] = 0
    C = ptc.matmul_f16(pinned(A.view(np.float16)), pinned(B.view(np.float16)))
    check_f16(C.numpy(), A, B)
    K8 = K + (-K) % 16
    A8, B8 = datagen.s8_operands(N, seed=M * 5 + K, m=M, k=K8)
    C8 = torch.empty((M, N), dtype=torch.int32, pin_memory=True)
    hA8, hB8 = pinned(A8), pinned(B8)  # the copies are asynchronous: keep the buffers alive
    ptc.gemm_s8_host(M, N, K, hA8.data_ptr(), K8, hB8.data_ptr(), K8, C8.data_ptr(), N, 0)
    torch.cuda.synchronize()
    assert np.array_equal(C8.numpy(), oracle.wrap_s32(oracle.gemm_s8(A8[:, :K], B8[:, :K])))
    K32 = K + (-K) % 32
    A4, B4 = datagen.s4_operands(N, seed=M * 7 + K, m=M, k=K32)
    hA4, hB4 = pinned(A4), pinned(B4)
    C4 = torch.empty((M, N), dtype=torch.int32, pin_memory=True)
    ptc.gemm_s4_host(M, N, K, hA4.data_ptr(), K32, hB4.data_ptr(), K32, C4.data_ptr(), N, 0)
    torch.cuda.synchronize()
    assert np.array_equal(C4.numpy(), oracle.wrap_s32(oracle.gemm_s4(A4, B4, K)))


@pytest.mark.parametrize("prec", ["f16", "s8", "s4"])
def test_host_pipelined_full_size(prec):
    """M = 8192: four row panels, copies overlapping the kernels."""
    n = 8192
    if prec == "f16":
        A, B = datagen.f16_operands(n, "normal")
        C = ptc.matmul_f16(pinned(A.view(np.float16)), pinned(B.view(np.float16))).numpy()
        check_f16_sampled(C, A, B, n=1500)
        return
    if prec == "s8":
        A, B = datagen.s8_operands(n)
        C = ptc.matmul_s8(pinned(A), pinned(B)).numpy()
        Cd = ptc.matmul_s8(torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV)).cpu().numpy()
        ref_at = lambda ii, jj: oracle.gemm_s8_at(A, B, ii, jj)
    else:
        A, B = datagen.s4_operands(n)
        C = ptc.matmul_s4(pinned(A), pinned(B), n).numpy()
        Cd = ptc.matmul_s4(torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV), n).cpu().numpy()
        ref_at = lambda ii, jj: oracle.gemm_s4_at(A, B, n, ii, jj)
    assert np.array_equal(C, Cd)
    ii, jj = sample_coords(n, n, 3000)
    assert np.array_equal(C[ii, jj], oracle.wrap_s32(ref_at(ii, jj)))


def test_host_three_streams_concurrently():
    n = 4096
    A, B = datagen.f16_operands(n, "normal", m=8192)
    A8, B8 = datagen.s8_operands(n, m=8192)
    A4, B4 = datagen.s4_operands(n, m=8192)
    streams = [torch.cuda.Stream() for _ in range(3)]
    C16 = torch.empty((8192, n), dtype=torch.float32, pin_memory=True)
    C8 = torch.empty((8192, n), dtype=torch.int32, pin_memory=True)
    C4 = torch.empty((8192, n), dtype=torch.int32, pin_memory=True)
    keep = [pinned(A.view(np.float16)), pinned(B.view(np.float16)), pinned(A8), pinned(B8), pinned(A4), pinned(B4)]
    ptc.matmul_f16(keep[0], keep[1], out=C16, stream=streams[0], sync=False)
    ptc.matmul_s8(keep[2], keep[3], out=C8, stream=streams[1], sync=False)
    ptc.matmul_s4(keep[4], keep[5], n, out=C4, stream=streams[2], sync=False)
    for s in streams:
        s.synchronize()
    ii, jj = sample_coords(8192, n, 1000)
    c, sabs = oracle.gemm_f16_at(A, B, ii, jj)
    assert np.all(np.abs(C16.numpy()[ii, jj] - c) <= 1e-3 * sabs + 1e-6)
    assert np.array_equal(C8.numpy()[ii, jj], oracle.wrap_s32(oracle.gemm_s8_at(A8, B8, ii, jj)))
    assert np.array_equal(C4.numpy()[ii, jj], oracle.wrap_s32(oracle.gemm_s4_at(A4, B4, n, ii, jj)))


def test_host_pageable_and_zero_k():
    M, N, K = 256, 512, 256
    A8, B8 = datagen.s8_operands(N, m=M, k=K)
    C = np.empty((M, N), dtype=np.int32)  # pageable numpy memory
    ptc.gemm_s8_host(M, N, K, A8.ctypes.data, K, B8.ctypes.data, K, C.ctypes.data, N, 0)
    torch.cuda.synchronize()
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A8, B8)))
    Cz = torch.full((M, N), 5, dtype=torch.int32, pin_memory=True)
    ptc.gemm_s8_host(M, N, 0, 0, 0, 0, 0, Cz.data_ptr(), N, 0)
    torch.cuda.synchronize()
    assert np.all(Cz.numpy() == 0)
