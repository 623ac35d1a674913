"""GPU parity of the persistent scheduler's tail split: when the last wave of
output tiles would leave at least half of the CTAs (or CTA pairs) idle, each
of those tiles runs as two units over the two halves of K, on two CTAs (or
pairs), and the epilogue warp that finishes second adds the other's partial
sums.

The shapes below give one full wave plus a short tail in both launch modes
(one CTA per 128 x 256 tile, CTA pairs on 256 x 256 tiles), a lone partial
wave, ragged N and K (odd numbers of K blocks, so the halves differ), and a
K of one block (never split).  Each runs with the split enabled and
disabled; both must match the oracle (INT8 / INT4 bit-exact, FP16 within the
element-wise bound, scaled outputs bit-exact), and integer results must be
identical with and without the split."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, check_f16, f16_dev, int_dev

pytestmark = pytest.mark.gpu

# (M, N, K): 2560 x 2048 is 160 one-CTA tiles / 80 pair tiles, a wave plus a
# short tail on 148..152 CTAs / 74..76 pairs; 2560 x 1848 leaves a last tile
# column of 56 values; 640 x 1000 is a lone partial wave; K = 192, 136 and 320
# give odd numbers of 64-value K blocks (3, 3, 5), K = 200 four blocks; CTA
# pairs stage two blocks at a time, so their split point is a whole stage and
# K = 128 (one pair stage) is not split; K = 40 is a single block (no split).
SHAPES = [(2560, 2048, 192), (2560, 1848, 200), (640, 1000, 136), (2560, 2048, 40), (2560, 2048, 128),
          (640, 1000, 320)]



@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    ptc.ptc_set_tuning("split_min_kb", 64)
    ptc.ptc_set_tuning("tail_split", 1)
    ptc.ptc_set_tuning("cta_pair", 0)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.fixture(params=[(1, 1, 1), (1, 0, 1), (2, 1, 1), (2, 1, 0), (2, 0, 1)],
                ids=["cta1-split", "cta1-nosplit", "cta2-split-reduce", "cta2-split-exchange", "cta2-nosplit"])
def mode(request):
    """Launch mode and split setting (CTA pairs add the halves of FP32 / int32
    tiles into C by TMA reductions, or exchange partial sums through the
    workspace); the split threshold is lowered to two K blocks so that the
    oracle-sized shapes below are split."""
    ctas, split, reduce = request.param
    ptc.ptc_set_tuning("cta_pair", ctas)
    ptc.ptc_set_tuning("tail_split", split)
    ptc.ptc_set_tuning("split_reduce", reduce)
    ptc.ptc_set_tuning("split_min_kb", 2)
    ptc.ptc_set_tuning("ksplit", 1)  # the lone partial wave would otherwise run as K-split clusters
    yield request.param
    ptc.ptc_set_tuning("split_reduce", 1)
    ptc.ptc_set_tuning("ksplit", 0)
    ptc.ptc_set_tuning("split_min_kb", 64)
    ptc.ptc_set_tuning("tail_split", 1)
    ptc.ptc_set_tuning("cta_pair", 0)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_tail_f16(M, N, K, mode):
    A, B = datagen.f16_operands(N, "normal", seed=M + N + K, m=M, k=K)
    Ad, Bd = f16_dev(A), f16_dev(B)
    C = ptc.matmul_f16(Ad, Bd)
    torch.cuda.synchronize()
    check_f16(C.cpu().numpy(), A, B)
    # the split halves may add in either order: the same bits every run
    C2 = ptc.matmul_f16(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int32), C2.view(torch.int32))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_tail_s8(M, N, K, mode):
    A, Bt = datagen.s8_operands(N, seed=M + N + K, m=M, k=K)
    A16 = np.zeros((M, (K + 15) // 16 * 16), np.int8)
    B16 = np.zeros((N, A16.shape[1]), np.int8)
    A16[:, :K], B16[:, :K] = A, Bt
    Ad, Bd = int_dev(A16), int_dev(B16)
    Cd = torch.empty((M, N), dtype=torch.int32, device=DEV)
    ptc.gemm_s8(M, N, K, Ad.data_ptr(), A16.shape[1], Bd.data_ptr(), B16.shape[1], Cd.data_ptr(), N, 0)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


@pytest.mark.parametrize("M,N,K", [(2560, 2048, 256), (2560, 1848, 384), (640, 1000, 2176)])
def test_tail_s4(M, N, K, mode):
    A, Bt = datagen.s4_operands(N, seed=M + N + K, m=M, k=K)
    C = ptc.matmul_s4(int_dev(A), int_dev(Bt), K)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s4(A, Bt, K)))


@pytest.mark.parametrize("out", [(torch.bfloat16, "bf16"), (torch.float32, "f32")], ids=["bf16", "f32"])
def test_tail_s8_scaled(out, mode):
    M, N, K = 2560, 1848, 192
    A, Bt = datagen.s8_operands(N, seed=11, m=M, k=K)
    rng = np.random.default_rng(12)
    sa = (rng.standard_normal(M) * 0.01).astype(np.float32)
    sb = (rng.standard_normal(N) * 0.01).astype(np.float32)
    dtype, name = out
    C = ptc.matmul_s8_scaled(int_dev(A), int_dev(Bt), torch.from_numpy(sa).to(DEV), torch.from_numpy(sb).to(DEV),
                             out_dtype=dtype)
    torch.cuda.synchronize()
    code = {"bf16": oracle.OUT_BF16, "f32": oracle.OUT_F32}[name]
    ref = oracle.dequant(oracle.gemm_s8(A, Bt), sa, sb, code)
    if dtype == torch.float32:
        got = C.cpu().view(torch.int32).numpy().view(np.uint32)
    else:
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_tail_f16acc_permutation(mode):
    """FP16 accumulators through the split: a row permutation is exact."""
    M, K, N = 2560, 192, 1848
    perm = np.random.default_rng(5).integers(0, K, size=M)
    A = np.zeros((M, K), np.float16)
    A[np.arange(M), perm] = 1
    B = np.random.default_rng(6).uniform(-100, 100, size=(K, N)).astype(np.float16)
    C = ptc.matmul_f16_f16acc(f16_dev(A.view(np.uint16)), f16_dev(B.view(np.uint16)))
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy().astype(np.float64), B.astype(np.float64)[perm])


def test_tail_int_identical_with_and_without_split():
    """Integer sums do not depend on the split, at the default threshold
    (K = 8256 is 129 K blocks; the INT8 route folds its FP32 partial sums every
    1024 values, so each half spans several folds)."""
    M, N, K = 2560, 1848, 8256
    A, Bt = datagen.s8_operands(N, seed=21, m=M, k=K)
    Ad, Bd = int_dev(A), int_dev(Bt)
    out = []
    for split in (1, 0):
        ptc.ptc_set_tuning("tail_split", split)
        out.append(ptc.matmul_s8(Ad, Bd).cpu().numpy())
    ptc.ptc_set_tuning("tail_split", 1)
    assert np.array_equal(out[0], out[1])
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK
    ii = np.random.default_rng(22).integers(0, M, 3000)
    jj = np.random.default_rng(23).integers(0, N, 3000)
    assert np.array_equal(out[0][ii, jj], oracle.wrap_s32(oracle.gemm_s8_at(A, Bt, ii, jj)))


def test_split_region_exact_at_default_settings():
    """N = 4096 with the default settings: the last wave of CTA-pair tiles (the
    bottom-right tiles of the grouped raster order) runs as K halves added
    into C by TMA reductions.  The whole lower-right quarter of C, which holds
    those tiles, matches the oracle: INT8 bit-exact, FP16 within the bound."""
    N = 4096
    A, Bt = datagen.s8_operands(N, seed=41)
    C = ptc.matmul_s8(int_dev(A), int_dev(Bt)).cpu().numpy()
    r, c = slice(N // 2, N), slice(N // 2, N)
    assert np.array_equal(C[r, c], oracle.wrap_s32(oracle.gemm_s8(A[r], Bt[c])))
    A16, B16 = datagen.f16_operands(N, "normal", seed=42)
    C16 = ptc.matmul_f16(f16_dev(A16), f16_dev(B16)).cpu().numpy()
    r, c = slice(N - 512, N), slice(N // 2, N)
    check_f16(C16[r, c], np.ascontiguousarray(A16[r]), np.ascontiguousarray(B16[:, c]))
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK
