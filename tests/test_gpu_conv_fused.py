"""GPU parity of integer products whose operands are converted inside the GEMM
kernel (tuning key "conv_fused" = 1): six converter warps per CTA rewrite the
raw s8 / packed s4 rows into the workspace the tensor maps read, panel slice
by panel slice in the order the tiles need them, and the producer loads a
slice once its counter holds all its pieces.  Every result is bit-exact
against the oracle, in one-CTA and CTA-pair launches: ragged M, N, K (K at and
around the 256-element slice and the fold boundaries), a single wave and
several, the extremes of both ranges, the scaled outputs, the same bits as
the separate pass, the benchmark's N = 8192 products (sampled), and a
withheld piece (the producers' bounded waits report a timeout; the context
survives).  In-ring conversion is turned off so that small one-CTA products
take this route too."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, int_dev, sample_coords

pytestmark = pytest.mark.gpu

FUSED = 3


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
    ptc.ptc_set_tuning("conv_fused", 1)
    ptc.ptc_set_tuning("cta_pair", request.param)
    ptc.ptc_set_tuning("in_ring", 0)  # small one-CTA products would convert in the ring
    yield request.param
    ptc.ptc_set_tuning("conv_fused", 0)
    ptc.ptc_set_tuning("cta_pair", 0)
    ptc.ptc_set_tuning("in_ring", 1)


def padded_dev(a: np.ndarray) -> torch.Tensor:
    rows, cols = a.shape
    w = max(32, (cols + 31) // 32 * 32)
    out = np.zeros((rows, w), dtype=a.dtype)
    out[:, :cols] = a
    return int_dev(out)[:, :cols]


def out_padded(M, N, dtype=torch.int32) -> torch.Tensor:
    per = 16 // torch.empty((), dtype=dtype).element_size()
    return torch.empty((M, (N + per - 1) // per * per), dtype=dtype, device=DEV)[:, :N]


def run_s8(A, Bt):
    C = ptc.matmul_s8(padded_dev(A), padded_dev(Bt), out=out_padded(A.shape[0], Bt.shape[0]))
    mode = ptc.ptc_last_conversion()
    torch.cuda.synchronize()
    return C.cpu().numpy(), mode


def run_s4(A, Bt, K):
    C = ptc.matmul_s4(padded_dev(A), padded_dev(Bt), K, out=out_padded(A.shape[0], Bt.shape[0]))
    mode = ptc.ptc_last_conversion()
    torch.cuda.synchronize()
    return C.cpu().numpy(), mode


SHAPES = [(300, 520, 200), (100, 40, 48), (256, 256, 64), (512, 512, 1000), (777, 1300, 1100),
          (1024, 768, 2048), (2048, 2048, 2048), (1536, 2816, 1536), (2304, 4352, 640)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_conv_fused_exact(M, N, K, cta_mode):
    A, Bt = datagen.s8_operands(N, seed=M * 13 + N + K, m=M, k=K)
    C, mode = run_s8(A, Bt)
    assert mode == FUSED
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    K4 = K + (K & 1)
    A4, Bt4 = datagen.s4_operands(N, seed=M * 17 + N + K4, m=M, k=K4)
    C4, mode = run_s4(A4, Bt4, K4)
    assert mode == FUSED
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K4)))


@pytest.mark.parametrize("K", [16, 63, 64, 65, 255, 256, 257, 511, 1023, 1025, 2049])
def test_conv_fused_k_boundaries(K, cta_mode):
    M, N = 264, 520
    A, Bt = datagen.s8_operands(N, seed=K, m=M, k=K)
    C, mode = run_s8(A, Bt)
    assert mode == FUSED
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    K4 = K + (K & 1)
    A4, Bt4 = datagen.s4_operands(N, seed=K + 5, m=M, k=K4)
    C4, mode = run_s4(A4, Bt4, K4)
    assert mode == FUSED
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K4)))


def test_conv_fused_constant_extremes(cta_mode):
    """-128 * -128 and -8 * -8 over K = 2^16: C = K a b exactly (s8: 2^30)."""
    M, N, K = 256, 512, 1 << 16
    A = torch.full((M, K), -128, dtype=torch.int8, device=DEV)
    Bt = torch.full((N, K), -128, dtype=torch.int8, device=DEV)
    C = ptc.matmul_s8(A, Bt)
    assert ptc.ptc_last_conversion() == FUSED
    torch.cuda.synchronize()
    assert torch.all(C == K * 16384).item()
    A4 = torch.full((M, K // 2), 0x88, dtype=torch.uint8, device=DEV)
    B4 = torch.full((N, K // 2), 0x88, dtype=torch.uint8, device=DEV)
    C4 = ptc.matmul_s4(A4, B4, K)
    assert ptc.ptc_last_conversion() == FUSED
    torch.cuda.synchronize()
    assert torch.all(C4 == 64 * K).item()


def test_conv_fused_same_bits_as_separate_pass(cta_mode):
    M, N, K = 1536, 1280, 1536
    A, Bt = datagen.s8_operands(N, seed=71, m=M, k=K)
    C_fused, mode = run_s8(A, Bt)
    assert mode == FUSED
    ptc.ptc_set_tuning("conv_fused", 0)
    C_pass, mode = run_s8(A, Bt)
    assert mode == 1
    assert np.array_equal(C_fused, C_pass)
    assert np.array_equal(C_fused, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_conv_fused_scaled(out, cta_mode):
    M, N, K = 600, 700, 900
    rng = np.random.default_rng(5)
    A, Bt = datagen.s8_operands(N, seed=81, m=M, k=K)
    sa = rng.uniform(0.5, 2.0, M).astype(np.float32)
    sb = rng.uniform(0.5, 2.0, N).astype(np.float32)
    C = ptc.matmul_s8_scaled(padded_dev(A), padded_dev(Bt), torch.from_numpy(sa).to(DEV),
                             torch.from_numpy(sb).to(DEV), out_dtype=out, out=out_padded(M, N, out))
    assert ptc.ptc_last_conversion() == FUSED
    torch.cuda.synchronize()
    code = oracle.OUT_F32 if out == torch.float32 else oracle.OUT_BF16
    ref = oracle.dequant(oracle.gemm_s8(A, Bt), sa, sb, code)
    if out == torch.float32:
        got = C.cpu().view(torch.int32).numpy().view(np.uint32)
    else:
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("prec", ["s8", "s4"])
def test_conv_fused_bench_size(prec):
    """The benchmark's N = 8192 products on the default shape (CTA pairs),
    sampled outputs."""
    ptc.ptc_set_tuning("conv_fused", 1)
    try:
        n = 8192
        if prec == "s8":
            A, Bt = datagen.s8_operands(n)
            C = ptc.matmul_s8(int_dev(A), int_dev(Bt))
        else:
            A, Bt = datagen.s4_operands(n)
            C = ptc.matmul_s4(int_dev(A), int_dev(Bt), n)
        assert ptc.ptc_last_conversion() == FUSED
        torch.cuda.synchronize()
    finally:
        ptc.ptc_set_tuning("conv_fused", 0)
    ii, jj = sample_coords(n, n, 4000, seed=9)
    got = C.cpu().numpy()[ii, jj]
    ref = oracle.gemm_s8_at(A, Bt, ii, jj) if prec == "s8" else oracle.gemm_s4_at(A, Bt, n, ii, jj)
    assert np.array_equal(got, oracle.wrap_s32(ref))


@pytest.mark.parametrize("stall", [-2, 0], ids=["piece", "tile"])
def test_conv_fused_wait_timeout_and_recovery(stall, cta_mode):
    """-2: the first converted piece is withheld (the producers waiting for its
    slice give up); 0: tile 0's first operand block is withheld.  Either way
    the call reports PTC_ERR_TIMEOUT after 50 ms and the next call on the same
    context is exact."""
    M, N, K = 512, 512, 512
    A, Bt = datagen.s8_operands(N, seed=97, m=M, k=K)
    Ad, Bd = padded_dev(A), padded_dev(Bt)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK
    ptc.ptc_debug_set_wait_limit(50_000_000, stall_tile=stall)
    try:
        ptc.matmul_s8(Ad, Bd)
        assert ptc.ptc_last_conversion() == FUSED
        torch.cuda.synchronize()
        assert ptc.gemm_poll_device_error() == ptc.PTC_ERR_TIMEOUT
    finally:
        ptc.ptc_debug_set_wait_limit(0, -1)
    C = ptc.matmul_s8(Ad, Bd)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK
