"""GPU parity on seeded random shapes: M, N, K drawn from 1 .. 1500 (K even for
packed s4), each precision, on the shape the planner picks (narrow tiles,
K-split clusters, in-ring conversion, CTA pairs) and with CTA pairs forced.
FP16 within the FP16 tolerance, INT8 / INT4 bit-exact against the oracle; on
half of the shapes also the FP16-accumulator product (within its bound), the
dequantising epilogues (bit-exact) and the host-buffer entry points."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, check_f16, f16_dev, int_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.fixture(params=[0, 2], ids=["planner", "pairs"])
def cta_mode(request):
    ptc.ptc_set_tuning("cta_pair", request.param)
    yield request.param
    ptc.ptc_set_tuning("cta_pair", 0)


def shapes(n=30, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        # half log-uniform (small and ragged shapes), half uniform (several tiles and waves)
        if i % 2 == 0:
            m, nn, k = (int(np.exp(rng.uniform(0, np.log(1500)))) for _ in range(3))
        else:
            m, nn, k = (int(rng.integers(1, 1501)) for _ in range(3))
        out.append((max(1, m), max(1, nn), max(1, k)))
    return out


SHAPES = shapes()


def padded(a: np.ndarray, per: int) -> np.ndarray:
    rows, cols = a.shape
    w = max(per, (cols + per - 1) // per * per)
    out = np.zeros((rows, w), dtype=a.dtype)
    out[:, :cols] = a
    return out


def out_padded(M, N, dtype=torch.int32):
    per = 16 // torch.empty((), dtype=dtype).element_size()
    return torch.empty((M, (N + per - 1) // per * per), dtype=dtype, device=DEV)[:, :N]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_random_shape_f16(M, N, K, cta_mode):
    A, B = datagen.f16_operands(N, "normal", seed=M * 7919 + N * 31 + K, m=M, k=K)
    Ad = f16_dev(padded(A, 8))[:, :K]
    Bd = f16_dev(padded(B, 8))[:, :N]
    C = ptc.matmul_f16(Ad, Bd, out=out_padded(M, N, torch.float32))
    torch.cuda.synchronize()
    check_f16(C.cpu().numpy(), A, B)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_random_shape_int(M, N, K, cta_mode):
    A, Bt = datagen.s8_operands(N, seed=M * 104729 + N * 37 + K, m=M, k=K)
    C = ptc.matmul_s8(int_dev(padded(A, 16))[:, :K], int_dev(padded(Bt, 16))[:, :K], out=out_padded(M, N))
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    K4 = K + (K & 1)
    A4, Bt4 = datagen.s4_operands(N, seed=M * 1299709 + N * 41 + K4, m=M, k=K4)
    C4 = ptc.matmul_s4(int_dev(padded(A4, 16))[:, :K4 // 2], int_dev(padded(Bt4, 16))[:, :K4 // 2], K4,
                       out=out_padded(M, N))
    torch.cuda.synchronize()
    assert np.array_equal(C4.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K4)))


SUBSET = SHAPES[::2]


@pytest.mark.parametrize("M,N,K", SUBSET)
def test_random_shape_f16acc(M, N, K, cta_mode):
    """FP16 accumulators: within one binary16 rounding per 16-deep step
    (|C - sum| <= (ceil(K/16) + 1) 2^-10 S + ceil(K/16) 2^-24)."""
    A, B = datagen.f16_operands(N, "uniform", seed=M * 3 + N * 5 + K, m=M, k=K)
    C = ptc.matmul_f16_f16acc(f16_dev(padded(A, 8))[:, :K], f16_dev(padded(B, 8))[:, :N],
                              out=out_padded(M, N, torch.float16))
    torch.cuda.synchronize()
    Cref, S = oracle.gemm_f16(A, B)
    steps = -(-K // 16)
    bound = (steps + 1) * 2.0 ** -10 * S + steps * 2.0 ** -24
    assert np.all(np.abs(C.cpu().numpy().astype(np.float64) - Cref) <= bound)


@pytest.mark.parametrize("i,M,N,K", [(i,) + s for i, s in enumerate(SUBSET)])
def test_random_shape_scaled(i, M, N, K, cta_mode):
    """Dequantising epilogues, the output type rotating over FP32, BF16, FP16:
    bit-exact against the oracle's rounding order."""
    out = (torch.float32, torch.bfloat16, torch.float16)[i % 3]
    code = {torch.float32: oracle.OUT_F32, torch.bfloat16: oracle.OUT_BF16, torch.float16: oracle.OUT_F16}[out]
    rng = np.random.default_rng(i)
    sa = rng.uniform(0.25, 4.0, M).astype(np.float32)
    sb = rng.uniform(0.25, 4.0, N).astype(np.float32)
    A, Bt = datagen.s8_operands(N, seed=M + N + K + 17, m=M, k=K)
    C = ptc.matmul_s8_scaled(int_dev(padded(A, 16))[:, :K], int_dev(padded(Bt, 16))[:, :K],
                             torch.from_numpy(sa).to(DEV), torch.from_numpy(sb).to(DEV), out=out_padded(M, N, out))
    K4 = K + (K & 1)
    A4, Bt4 = datagen.s4_operands(N, seed=M + N + K4 + 23, m=M, k=K4)
    C4 = ptc.matmul_s4_scaled(int_dev(padded(A4, 16))[:, :K4 // 2], int_dev(padded(Bt4, 16))[:, :K4 // 2], K4,
                              torch.from_numpy(sa).to(DEV), torch.from_numpy(sb).to(DEV), out=out_padded(M, N, out))
    torch.cuda.synchronize()

    def bits(t):
        return (t.cpu().view(torch.int32).numpy().view(np.uint32) if out == torch.float32
                else t.cpu().view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(bits(C), oracle.dequant(oracle.gemm_s8(A, Bt), sa, sb, code))
    assert np.array_equal(bits(C4), oracle.dequant(oracle.gemm_s4(A4, Bt4, K4), sa, sb, code))


@pytest.mark.parametrize("M,N,K", SUBSET)
def test_random_shape_host_buffers(M, N, K):
    """The host-buffer entry points (pinned host operands and results,
    pipelined copies inside the library)."""
    A, B = datagen.f16_operands(N, "normal", seed=M * 11 + N + K, m=M, k=K)
    hA = torch.from_numpy(padded(A, 8).view(np.float16)).pin_memory()[:, :K]
    hB = torch.from_numpy(padded(B, 8).view(np.float16)).pin_memory()[:, :N]
    hC = torch.empty((M, (N + 3) // 4 * 4), dtype=torch.float32).pin_memory()[:, :N]
    C = ptc.matmul_f16(hA, hB, out=hC)
    check_f16(C.numpy(), A, B)
    A8, Bt8 = datagen.s8_operands(N, seed=M * 13 + N + K, m=M, k=K)
    h8 = torch.empty((M, (N + 3) // 4 * 4), dtype=torch.int32).pin_memory()[:, :N]
    C8 = ptc.matmul_s8(torch.from_numpy(padded(A8, 16)).pin_memory()[:, :K],
                       torch.from_numpy(padded(Bt8, 16)).pin_memory()[:, :K], out=h8)
    assert np.array_equal(C8.numpy(), oracle.wrap_s32(oracle.gemm_s8(A8, Bt8)))
    K4 = K + (K & 1)
    A4, Bt4 = datagen.s4_operands(N, seed=M * 17 + N + K4, m=M, k=K4)
    h4 = torch.empty((M, (N + 3) // 4 * 4), dtype=torch.int32).pin_memory()[:, :N]
    C4 = ptc.matmul_s4(torch.from_numpy(padded(A4, 16)).pin_memory()[:, :K4 // 2],
                       torch.from_numpy(padded(Bt4, 16)).pin_memory()[:, :K4 // 2], K4, out=h4)
    assert np.array_equal(C4.numpy(), oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K4)))


@pytest.mark.parametrize("M,N,K", SUBSET)
def test_random_shape_s8_rowmajor_b(M, N, K, cta_mode):
    """INT8 with B row-major (K x N), read MN-major: bit-exact."""
    A, Bt = datagen.s8_operands(N, seed=M * 19 + N + K, m=M, k=K)
    B_kn = np.ascontiguousarray(Bt.T)
    Ad, Bd = int_dev(padded(A, 16)), int_dev(padded(B_kn, 16))
    C = out_padded(M, N)
    ptc.gemm_s8_b_rowmajor(M, N, K, Ad.data_ptr(), Ad.shape[1], Bd.data_ptr(), Bd.shape[1], C.data_ptr(),
                           C.stride(0), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
