"""GPU parity of CTA-pair products run two pairs per thread-block cluster
(tuning key "multicast" = 1): the pairs compute tile columns 2n and 2n + 1 of
one tile row and share A by TMA multicast (each CTA loads half of its 128 A
rows for itself and for its counterpart in the other pair).  FP16 within the
FP16 tolerance, INT8 / INT4 bit-exact, on ragged shapes (an odd count of tile
columns leaves the second pair's tile past N), K at the fold boundaries, the
scaled and FP16-accumulator epilogues, the N = 8192 products (sampled), and a
withheld operand block (bounded waits report a timeout; the context
survives).  cta_pair = 2 forces CTA pairs at every size."""
import math

import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, check_f16, check_f16_sampled, f16_dev, int_dev, sample_coords

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.fixture(autouse=True)
def multicast():
    ptc.ptc_set_tuning("multicast", 1)
    ptc.ptc_set_tuning("cta_pair", 2)
    yield
    ptc.ptc_set_tuning("multicast", 0)
    ptc.ptc_set_tuning("cta_pair", 0)


def padded_dev(a: np.ndarray, f16: bool = False) -> torch.Tensor:
    """Device copy with a 64-byte-multiple row pitch, viewed at the logical width."""
    rows, cols = a.shape
    per = 32 if f16 else 64
    w = max(per, (cols + per - 1) // per * per)
    out = np.zeros((rows, w), dtype=a.dtype)
    out[:, :cols] = a
    return (f16_dev(out) if f16 else int_dev(out))[:, :cols]


def out_padded(M, N, dtype=torch.int32) -> torch.Tensor:
    per = 16 // torch.empty((), dtype=dtype).element_size()
    return torch.empty((M, (N + per - 1) // per * per), dtype=dtype, device=DEV)[:, :N]


def cluster_of_last_launch() -> int:
    return ptc.ptc_last_launch()[1]


SHAPES = [(300, 520, 200), (256, 256, 64), (100, 40, 48), (1000, 1300, 700), (512, 768, 1024),
          (2048, 2048, 2048), (1536, 2816, 1536)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_multicast_fp16(M, N, K):
    A, B = datagen.f16_operands(N, "normal", seed=M + 3 * N + K, m=M, k=K)
    C = ptc.matmul_f16(padded_dev(A, True), padded_dev(B, True), out=out_padded(M, N, torch.float32))
    assert cluster_of_last_launch() == 4
    torch.cuda.synchronize()
    check_f16(C.cpu().numpy(), A, B)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_multicast_int8_int4(M, N, K):
    A, Bt = datagen.s8_operands(N, seed=M + 5 * N + K, m=M, k=K)
    C = ptc.matmul_s8(padded_dev(A), padded_dev(Bt), out=out_padded(M, N))
    assert cluster_of_last_launch() == 4 and ptc.ptc_last_conversion() != 2
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    K4 = K + (K & 1)
    A4, Bt4 = datagen.s4_operands(N, seed=M + 7 * N + K4, m=M, k=K4)
    C4 = ptc.matmul_s4(padded_dev(A4), padded_dev(Bt4), K4, out=out_padded(M, N))
    assert cluster_of_last_launch() == 4 and ptc.ptc_last_conversion() != 2
    torch.cuda.synchronize()
    assert np.array_equal(C4.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K4)))


@pytest.mark.parametrize("K", [63, 64, 65, 1023, 1024, 1025, 2049])
def test_multicast_k_boundaries(K):
    M, N = 520, 1100
    A, Bt = datagen.s8_operands(N, seed=K + 11, m=M, k=K)
    C = ptc.matmul_s8(padded_dev(A), padded_dev(Bt), out=out_padded(M, N))
    assert cluster_of_last_launch() == 4
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    K4 = K + (K & 1)
    A4, Bt4 = datagen.s4_operands(N, seed=K + 12, m=M, k=K4)
    C4 = ptc.matmul_s4(padded_dev(A4), padded_dev(Bt4), K4, out=out_padded(M, N))
    torch.cuda.synchronize()
    assert np.array_equal(C4.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K4)))


def test_multicast_constant_extremes():
    """-128 * -128 and -8 * -8 over K = 2^16: C = K a b exactly (s8: 2^30)."""
    M, N, K = 512, 768, 1 << 16
    A = torch.full((M, K), -128, dtype=torch.int8, device=DEV)
    Bt = torch.full((N, K), -128, dtype=torch.int8, device=DEV)
    C = ptc.matmul_s8(A, Bt)
    assert cluster_of_last_launch() == 4
    torch.cuda.synchronize()
    assert torch.all(C == K * 16384).item()
    A4 = torch.full((M, K // 2), 0x88, dtype=torch.uint8, device=DEV)
    B4 = torch.full((N, K // 2), 0x88, dtype=torch.uint8, device=DEV)
    C4 = ptc.matmul_s4(A4, B4, K)
    torch.cuda.synchronize()
    assert torch.all(C4 == 64 * K).item()


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_multicast_scaled(out):
    M, N, K = 700, 900, 640
    rng = np.random.default_rng(52)
    A, Bt = datagen.s8_operands(N, seed=51, m=M, k=K)
    sa = rng.uniform(0.5, 2.0, M).astype(np.float32)
    sb = rng.uniform(0.5, 2.0, N).astype(np.float32)
    C = ptc.matmul_s8_scaled(padded_dev(A), padded_dev(Bt), torch.from_numpy(sa).to(DEV),
                             torch.from_numpy(sb).to(DEV), out_dtype=out, out=out_padded(M, N, out))
    assert cluster_of_last_launch() == 4
    torch.cuda.synchronize()
    code = oracle.OUT_F32 if out == torch.float32 else oracle.OUT_BF16
    ref = oracle.dequant(oracle.gemm_s8(A, Bt), sa, sb, code)
    if out == torch.float32:
        got = C.cpu().view(torch.int32).numpy().view(np.uint32)
    else:
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_multicast_f16acc():
    """FP16 accumulators: within one binary16 rounding per 16-deep step."""
    M, N, K = 700, 900, 640
    A, B = datagen.f16_operands(N, "uniform", seed=53, m=M, k=K)
    C = ptc.matmul_f16_f16acc(padded_dev(A, True), padded_dev(B, True), out=out_padded(M, N, torch.float16))
    assert cluster_of_last_launch() == 4
    torch.cuda.synchronize()
    Cref, S = oracle.gemm_f16(A, B)
    steps = math.ceil(K / 16)
    bound = (steps + 1) * 2.0 ** -10 * S + steps * 2.0 ** -24
    assert np.all(np.abs(C.cpu().numpy().astype(np.float64) - Cref) <= bound)


def test_multicast_same_bits_as_one_pair():
    M, N, K = 1536, 1280, 1536
    A, Bt = datagen.s8_operands(N, seed=71, m=M, k=K)
    C2 = ptc.matmul_s8(padded_dev(A), padded_dev(Bt), out=out_padded(M, N))
    assert cluster_of_last_launch() == 4
    ptc.ptc_set_tuning("multicast", 0)
    C1 = ptc.matmul_s8(padded_dev(A), padded_dev(Bt), out=out_padded(M, N))
    assert cluster_of_last_launch() == 2
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    A16, B16 = datagen.f16_operands(N, "normal", seed=72, m=M, k=K)
    F1 = ptc.matmul_f16(padded_dev(A16, True), padded_dev(B16, True))
    ptc.ptc_set_tuning("multicast", 1)
    F2 = ptc.matmul_f16(padded_dev(A16, True), padded_dev(B16, True))
    assert cluster_of_last_launch() == 4
    torch.cuda.synchronize()
    # Same MMAs in the same K order on the same tile: the same bits.
    assert torch.equal(F1.view(torch.int32), F2.view(torch.int32))


@pytest.mark.parametrize("prec", ["f16", "s8", "s4"])
def test_multicast_bench_size(prec):
    """The benchmark's N = 8192 products, on sampled outputs."""
    n = 8192
    if prec == "f16":
        A, B = datagen.f16_operands(n, "normal")
        C = ptc.matmul_f16(f16_dev(A), f16_dev(B))
        assert cluster_of_last_launch() == 4
        torch.cuda.synchronize()
        check_f16_sampled(C.cpu().numpy(), A, B, n=3000)
        return
    if prec == "s8":
        A, Bt = datagen.s8_operands(n)
        C = ptc.matmul_s8(int_dev(A), int_dev(Bt))
    else:
        A, Bt = datagen.s4_operands(n)
        C = ptc.matmul_s4(int_dev(A), int_dev(Bt), n)
    assert cluster_of_last_launch() == 4
    torch.cuda.synchronize()
    ii, jj = sample_coords(n, n, 4000, seed=21)
    ref = oracle.gemm_s8_at(A, Bt, ii, jj) if prec == "s8" else oracle.gemm_s4_at(A, Bt, n, ii, jj)
    assert np.array_equal(C.cpu().numpy()[ii, jj], oracle.wrap_s32(ref))


def test_multicast_wait_timeout_and_recovery():
    """Unit 0's first K blocks are withheld by the even CTA of each pair: the
    bounded waits give up after 50 ms, the call reports PTC_ERR_TIMEOUT, and
    the next call on the same context is exact."""
    M, N, K = 512, 1024, 512
    A, Bt = datagen.s8_operands(N, seed=61, m=M, k=K)
    Ad, Bd = padded_dev(A), padded_dev(Bt)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK
    ptc.ptc_debug_set_wait_limit(50_000_000, stall_tile=0)
    try:
        ptc.matmul_s8(Ad, Bd)
        assert cluster_of_last_launch() == 4
        torch.cuda.synchronize()
        assert ptc.gemm_poll_device_error() == ptc.PTC_ERR_TIMEOUT
    finally:
        ptc.ptc_debug_set_wait_limit(0, -1)
    C = ptc.matmul_s8(Ad, Bd)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK
