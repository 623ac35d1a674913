"""GPU parity of operand conversion inside the CTA-pair kernel: integer
products on 256 x 256 pair tiles load K blocks of the raw s8 / packed s4
operands (64 bytes per row) and four dedicated converter warps per CTA write
the binary16 / E4M3 stage the pair's MMAs read, with no workspace and no
separate pass.  Every result is bit-exact against the oracle: ragged M, N, K
(a partial last K block, K below one block), K at every fold boundary, more
tiles than pairs (several tiles per pair, the epilogue overlapping the next
tile), the extremes of both ranges, the scaled outputs, the same bits as the
separate-pass route, the benchmark's N = 8192 products, and a withheld operand
block (the converter warps' bounded waits report a timeout, the context
survives).  The knob pair_in_ring = 2 selects the route, cta_pair = 2 forces
pairs at every size."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, int_dev, sample_coords

pytestmark = pytest.mark.gpu

IN_RING, SEPARATE = 2, 1


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.fixture(autouse=True)
def pair_in_ring():
    ptc.ptc_set_tuning("pair_in_ring", 2)
    ptc.ptc_set_tuning("cta_pair", 2)
    yield
    ptc.ptc_set_tuning("pair_in_ring", 0)
    ptc.ptc_set_tuning("cta_pair", 0)
    ptc.ptc_set_tuning("s8_chunk_kb", 16)
    ptc.ptc_set_tuning("s4_chunk_kb", 64)


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
    mode, launch = ptc.ptc_last_conversion(), ptc.ptc_last_launch()
    torch.cuda.synchronize()
    return C.cpu().numpy(), mode, launch


def run_s4(A, Bt, K):
    C = ptc.matmul_s4(padded_dev(A), padded_dev(Bt), K, out=out_padded(A.shape[0], Bt.shape[0]))
    mode, launch = ptc.ptc_last_conversion(), ptc.ptc_last_launch()
    torch.cuda.synchronize()
    return C.cpu().numpy(), mode, launch


SHAPES = [(300, 520, 200), (100, 40, 48), (256, 256, 64), (512, 512, 1000), (777, 1300, 1100),
          (1024, 768, 2048), (2048, 2048, 2048)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_pair_in_ring_exact(M, N, K):
    A, Bt = datagen.s8_operands(N, seed=M * 13 + N + K, m=M, k=K)
    C, mode, launch = run_s8(A, Bt)
    assert mode == IN_RING and launch[1] == 2
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    K4 = K + (K & 1)
    A4, Bt4 = datagen.s4_operands(N, seed=M * 17 + N + K4, m=M, k=K4)
    C4, mode, launch = run_s4(A4, Bt4, K4)
    assert mode == IN_RING and launch[1] == 2
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K4)))


@pytest.mark.parametrize("K", [63, 64, 65, 127, 128, 129, 1023, 1024, 1025, 2047, 2049])
def test_pair_in_ring_k_boundaries(K):
    M, N = 264, 520
    A, Bt = datagen.s8_operands(N, seed=K, m=M, k=K)
    C, mode, _ = run_s8(A, Bt)
    assert mode == IN_RING
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    K4 = K + (K & 1)
    A4, Bt4 = datagen.s4_operands(N, seed=K + 5, m=M, k=K4)
    C4, mode, _ = run_s4(A4, Bt4, K4)
    assert mode == IN_RING
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K4)))


@pytest.mark.parametrize("chunk", [2, 6, 16])
def test_pair_in_ring_folds(chunk):
    """Folds every `chunk` K blocks over 48 K blocks (s8) while the converters
    keep the ring full."""
    ptc.ptc_set_tuning("s8_chunk_kb", chunk)
    ptc.ptc_set_tuning("s4_chunk_kb", chunk)
    M, N, K = 512, 768, 3072
    A, Bt = datagen.s8_operands(N, seed=30 + chunk, m=M, k=K)
    C, mode, _ = run_s8(A, Bt)
    assert mode == IN_RING
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    A4, Bt4 = datagen.s4_operands(N, seed=40 + chunk, m=M, k=2 * K)
    C4, mode, _ = run_s4(A4, Bt4, 2 * K)
    assert mode == IN_RING
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, 2 * K)))


def test_pair_in_ring_constant_extremes():
    """-128 * -128 and -8 * -8 over K = 2^16: C = K a b exactly (s8: 2^30)."""
    M, N, K = 256, 512, 1 << 16
    A = torch.full((M, K), -128, dtype=torch.int8, device=DEV)
    Bt = torch.full((N, K), -128, dtype=torch.int8, device=DEV)
    C = ptc.matmul_s8(A, Bt)
    assert ptc.ptc_last_conversion() == IN_RING
    torch.cuda.synchronize()
    assert torch.all(C == K * 16384).item()
    A4 = torch.full((M, K // 2), 0x88, dtype=torch.uint8, device=DEV)
    B4 = torch.full((N, K // 2), 0x88, dtype=torch.uint8, device=DEV)
    C4 = ptc.matmul_s4(A4, B4, K)
    assert ptc.ptc_last_conversion() == IN_RING
    torch.cuda.synchronize()
    assert torch.all(C4 == 64 * K).item()


def test_pair_in_ring_same_bits_as_separate_pass():
    M, N, K = 1536, 1280, 1536
    A, Bt = datagen.s8_operands(N, seed=71, m=M, k=K)
    C_ring, mode, _ = run_s8(A, Bt)
    assert mode == IN_RING
    ptc.ptc_set_tuning("pair_in_ring", 0)
    C_pass, mode, _ = run_s8(A, Bt)
    assert mode == SEPARATE
    assert np.array_equal(C_ring, C_pass)
    assert np.array_equal(C_ring, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float16, torch.float32], ids=["bf16", "f16", "f32"])
def test_pair_in_ring_scaled(out):
    M, N, K = 600, 700, 900
    rng = np.random.default_rng(5)
    A, Bt = datagen.s8_operands(N, seed=81, m=M, k=K)
    sa = rng.uniform(0.5, 2.0, M).astype(np.float32)
    sb = rng.uniform(0.5, 2.0, N).astype(np.float32)
    C = ptc.matmul_s8_scaled(padded_dev(A), padded_dev(Bt), torch.from_numpy(sa).to(DEV),
                             torch.from_numpy(sb).to(DEV), out_dtype=out, out=out_padded(M, N, out))
    assert ptc.ptc_last_conversion() == IN_RING
    torch.cuda.synchronize()
    code = {torch.float32: oracle.OUT_F32, torch.bfloat16: oracle.OUT_BF16, torch.float16: oracle.OUT_F16}[out]
    ref = oracle.dequant(oracle.gemm_s8(A, Bt), sa, sb, code)
    if out == torch.float32:
        got = C.cpu().view(torch.int32).numpy().view(np.uint32)
    else:
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("prec", ["s8", "s4"])
def test_pair_in_ring_bench_size(prec):
    """The benchmark's N = 8192 products on the pair in-ring route, on
    sampled outputs (the default route is checked in full elsewhere)."""
    n = 8192
    if prec == "s8":
        A, Bt = datagen.s8_operands(n)
        C = ptc.matmul_s8(int_dev(A), int_dev(Bt))
    else:
        A, Bt = datagen.s4_operands(n)
        C = ptc.matmul_s4(int_dev(A), int_dev(Bt), n)
    assert ptc.ptc_last_conversion() == IN_RING
    torch.cuda.synchronize()
    ii, jj = sample_coords(n, n, 4000, seed=8)
    got = C.cpu().numpy()[ii, jj]
    ref = oracle.gemm_s8_at(A, Bt, ii, jj) if prec == "s8" else oracle.gemm_s4_at(A, Bt, n, ii, jj)
    assert np.array_equal(got, oracle.wrap_s32(ref))


def test_pair_in_ring_wait_timeout_and_recovery():
    """Tile 0's first raw block is withheld from the even CTA: its converter
    warps' bounded waits give up after 50 ms, the call reports
    PTC_ERR_TIMEOUT, and the next call on the same context is exact."""
    M, N, K = 512, 512, 512
    A, Bt = datagen.s8_operands(N, seed=97, m=M, k=K)
    Ad, Bd = padded_dev(A), padded_dev(Bt)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK
    ptc.ptc_debug_set_wait_limit(50_000_000, stall_tile=0)
    try:
        ptc.matmul_s8(Ad, Bd)
        assert ptc.ptc_last_conversion() == IN_RING
        torch.cuda.synchronize()
        assert ptc.gemm_poll_device_error() == ptc.PTC_ERR_TIMEOUT
    finally:
        ptc.ptc_debug_set_wait_limit(0, -1)
    C = ptc.matmul_s8(Ad, Bd)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK
