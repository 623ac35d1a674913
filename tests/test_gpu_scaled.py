"""GPU parity of the scaled integer GEMMs (gemm_s8_scaled, gemm_s4_scaled)
against the oracle's dequantisation of the exact sums: bit-exact in every
output type, since both sides perform the same binary32 operations in the same
order and round the same way."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, int_dev, sample_coords

pytestmark = pytest.mark.gpu

OUT = {"f32": (torch.float32, oracle.OUT_F32), "bf16": (torch.bfloat16, oracle.OUT_BF16),
       "f16": (torch.float16, oracle.OUT_F16)}


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


def _scales(n, seed, spread=8):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(n) * np.exp2(rng.integers(-spread, spread + 1, size=n))).astype(np.float32)


def _bits(t):
    if t.dtype == torch.float32:
        return t.cpu().view(torch.int32).numpy().view(np.uint32)
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _operands(prec, M, N, K, seed):
    if prec == "s8":
        A, Bt = datagen.s8_operands(N, seed=seed, m=M, k=K)
        return A, Bt, oracle.gemm_s8(A, Bt)
    A, Bt = datagen.s4_operands(N, seed=seed, m=M, k=K)
    return A, Bt, oracle.gemm_s4(A, Bt, K)


def _run(prec, A, Bt, K, sa, sb, dtype):
    Ad, Bd = int_dev(A), int_dev(Bt)
    sad = None if sa is None else torch.from_numpy(sa).to(DEV)
    sbd = None if sb is None else torch.from_numpy(sb).to(DEV)
    if prec == "s8":
        C = ptc.matmul_s8_scaled(Ad, Bd, sad, sbd, out_dtype=dtype)
    else:
        C = ptc.matmul_s4_scaled(Ad, Bd, K, sad, sbd, out_dtype=dtype)
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("prec", ["s8", "s4"])
@pytest.mark.parametrize("M,N,K", [(300, 520, 192), (1024, 1024, 1024), (129, 264, 2048)])
def test_scaled_bit_exact(prec, out, M, N, K, cta_mode):
    A, Bt, exact = _operands(prec, M, N, K, seed=M + N + K)
    sa, sb = _scales(M, 1), _scales(N, 2)
    dtype, code = OUT[out]
    C = _run(prec, A, Bt, K, sa, sb, dtype)
    assert np.array_equal(_bits(C), oracle.dequant(exact, sa, sb, code))


@pytest.mark.parametrize("prec", ["s8", "s4"])
def test_scaled_without_scales_and_overflow(prec):
    M, N, K = 256, 512, 512
    A, Bt, exact = _operands(prec, M, N, K, seed=5)
    C = _run(prec, A, Bt, K, None, None, torch.float32)
    assert np.array_equal(_bits(C), oracle.dequant(exact, None, None, oracle.OUT_F32))
    # huge scales overflow binary16 to infinity on both sides
    sa = np.full(M, 300.0, np.float32)
    sb = _scales(N, 3, spread=4)
    C = _run(prec, A, Bt, K, sa, sb, torch.float16)
    ref = oracle.dequant(exact, sa, sb, oracle.OUT_F16)
    assert np.array_equal(_bits(C), ref) and np.any((ref & 0x7FFF) == 0x7C00)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_scaled_full_size_sampled(out):
    n = 8192
    A, Bt = datagen.s8_operands(n)
    sa, sb = _scales(n, 8), _scales(n, 9)
    dtype, code = OUT[out]
    C = _run("s8", A, Bt, n, sa, sb, dtype)
    ii, jj = sample_coords(n, n, 3000)
    exact = oracle.gemm_s8_at(A, Bt, ii, jj)
    # per-sample scales: dequantise each sample with its own row / column scale
    ref = np.array([oracle.dequant(np.array([[e]]), np.array([sa[i]]), np.array([sb[j]]), code)[0, 0]
                    for e, i, j in zip(exact, ii, jj)])
    assert np.array_equal(_bits(C)[ii, jj], ref)


def test_scaled_zero_k_and_bad_arguments():
    M, N = 40, 72
    C = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    ptc.gemm_s8_scaled(M, N, 0, 0, 0, 0, 0, None, None, C.data_ptr(), N, ptc.PTC_OUT_BF16, 0)
    torch.cuda.synchronize()
    assert np.all(_bits(C) == 0)
    with pytest.raises(ptc.PtcError) as e:
        ptc.gemm_s8_scaled(M, N, 16, C.data_ptr(), 16, C.data_ptr(), 16, None, None, C.data_ptr(), N, 7, 0)
    assert e.value.status == ptc.PTC_ERR_INVALID
