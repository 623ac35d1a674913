"""GPU parity of the narrow one-CTA tiles (128 x 128 and 128 x 64 outputs per
CTA), which spread a small product's C over more SMs: every route, forced to
each width, against the oracle (FP16 within the element-wise bound, integer
and scaled outputs bit-exact), on shapes with ragged M, N and K, a single
tile, and more tiles than SMs (the persistent loop then runs several narrow
tiles per CTA through both accumulator buffers).  The automatic choice is
checked against the same oracle, and its launch record against the rule
(narrow tiles only for products whose 128 x 256 tiles fit one wave)."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, check_f16, check_f16_sampled, f16_dev, int_dev, sample_coords

pytestmark = pytest.mark.gpu

# (M, N, K): 512^3 (32 / 16 narrow tiles); 300 x 700 x 200 (ragged: a last
# column tile of 60 / 60 values, 4 ragged K blocks); 100 x 40 x 1000 (one
# tile, 16 K blocks); 1000 x 1000 x 520; 1024 x 2048 x 320 (256 tiles of 64
# columns: more than one per CTA).
SHAPES = [(512, 512, 512), (300, 700, 200), (100, 40, 1000), (1000, 1000, 520), (1024, 2048, 320)]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    ptc.ptc_set_tuning("tile_n", 0)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.fixture(params=[64, 128, 0], ids=["n64", "n128", "auto"])
def tile_n(request):
    ptc.ptc_set_tuning("tile_n", request.param)
    yield request.param
    ptc.ptc_set_tuning("tile_n", 0)


def padded_dev(a: np.ndarray) -> torch.Tensor:
    rows, cols = a.shape
    w = max(16, (cols + 15) // 16 * 16)
    out = np.zeros((rows, w), dtype=a.dtype)
    out[:, :cols] = a
    return int_dev(out)[:, :cols]


def padded_f16_dev(bits: np.ndarray) -> torch.Tensor:
    rows, cols = bits.shape
    w = max(8, (cols + 7) // 8 * 8)
    out = np.zeros((rows, w), dtype=np.uint16)
    out[:, :cols] = bits
    return f16_dev(out)[:, :cols]


def out_padded(M, N, dtype) -> torch.Tensor:
    per = 16 // torch.empty((), dtype=dtype).element_size()
    return torch.empty((M, (N + per - 1) // per * per), dtype=dtype, device=DEV)[:, :N]


def _check_launch(tile_n, M, N):
    grid, cluster, ks, bn = ptc.ptc_last_launch()
    if tile_n in (64, 128):
        assert bn == tile_n and cluster == 1 and ks == 1
        tiles = ((M + 127) // 128) * ((N + tile_n - 1) // tile_n)
        assert 1 <= grid <= tiles
    elif bn != 256:
        # by size, narrow tiles only when the 128 x 256 tiles fit one wave and
        # the narrow ones too (one CTA, or one K-split cluster, per tile)
        tiles = ((M + 127) // 128) * ((N + bn - 1) // bn)
        assert grid == tiles * ks and cluster == ks


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_narrow_f16(M, N, K, tile_n):
    A, B = datagen.f16_operands(N, "normal", seed=M + 3 * N + K, m=M, k=K)
    C = ptc.matmul_f16(padded_f16_dev(A), padded_f16_dev(B), out=out_padded(M, N, torch.float32))
    _check_launch(tile_n, M, N)
    check_f16(C.cpu().numpy(), A, B)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_narrow_s8(M, N, K, tile_n):
    A, Bt = datagen.s8_operands(N, seed=M + 3 * N + K, m=M, k=K)
    C = ptc.matmul_s8(padded_dev(A), padded_dev(Bt), out=out_padded(M, N, torch.int32))
    _check_launch(tile_n, M, N)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_narrow_s4(M, N, K, tile_n):
    A, Bt = datagen.s4_operands(N, seed=M + 3 * N + K, m=M, k=K)
    C = ptc.matmul_s4(padded_dev(A), padded_dev(Bt), K, out=out_padded(M, N, torch.int32))
    _check_launch(tile_n, M, N)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s4(A, Bt, K)))


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float16, torch.float32], ids=["bf16", "f16", "f32"])
@pytest.mark.parametrize("M,N,K", [(300, 700, 200), (1024, 2048, 320)])
def test_narrow_s8_scaled(M, N, K, out, tile_n):
    A, Bt = datagen.s8_operands(N, seed=51 + K, m=M, k=K)
    rng = np.random.default_rng(52 + K)
    sa = (rng.standard_normal(M) * 0.01).astype(np.float32)
    sb = (rng.standard_normal(N) * 0.01).astype(np.float32)
    C = ptc.matmul_s8_scaled(padded_dev(A), padded_dev(Bt), torch.from_numpy(sa).to(DEV),
                             torch.from_numpy(sb).to(DEV), out_dtype=out, out=out_padded(M, N, out))
    _check_launch(tile_n, M, N)
    torch.cuda.synchronize()
    code = {torch.bfloat16: oracle.OUT_BF16, torch.float16: oracle.OUT_F16, torch.float32: oracle.OUT_F32}[out]
    ref = oracle.dequant(oracle.gemm_s8(A, Bt), sa, sb, code)
    if out == torch.float32:
        got = C.cpu().view(torch.int32).numpy().view(np.uint32)
    else:
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M,K,N", [(300, 200, 700), (1024, 320, 2048)])
def test_narrow_f16acc_permutation(M, K, N, tile_n):
    perm = np.random.default_rng(7 + K).integers(0, K, size=M)
    A = np.zeros((M, K), np.float16)
    A[np.arange(M), perm] = 1
    B = np.random.default_rng(8 + K).uniform(-100, 100, size=(K, N)).astype(np.float16)
    C = ptc.matmul_f16_f16acc(padded_f16_dev(A.view(np.uint16)), padded_f16_dev(B.view(np.uint16)),
                              out=out_padded(M, N, torch.float16))
    _check_launch(tile_n, M, N)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy().astype(np.float64), B.astype(np.float64)[perm])


@pytest.mark.parametrize("M,N,K", [(300, 700, 200), (1024, 2048, 320)])
def test_narrow_s8_rowmajor_b(M, N, K, tile_n):
    A, Bt = datagen.s8_operands(N, seed=M * 19 + K, m=M, k=K)
    B_kn = np.ascontiguousarray(Bt.T)
    Ad, Bd = padded_dev(A), padded_dev(B_kn)
    Cd = torch.empty((M, (N + 3) // 4 * 4), dtype=torch.int32, device=DEV)
    ptc.gemm_s8_b_rowmajor(M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), Cd.data_ptr(),
                           Cd.shape[1], torch.cuda.current_stream().cuda_stream)
    _check_launch(tile_n, M, N)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.cpu().numpy()[:, :N], oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


def test_narrow_long_k_sampled(tile_n):
    """A long K (FP16 K = 8192, 128 K blocks) through narrow tiles: sampled
    against the oracle."""
    M, N, K = 256, 512, 8192
    A, B = datagen.f16_operands(N, "normal", seed=61, m=M, k=K)
    C = ptc.matmul_f16(f16_dev(A), f16_dev(B))
    torch.cuda.synchronize()
    check_f16_sampled(C.cpu().numpy(), A, B, n=1500)
    A8, Bt8 = datagen.s8_operands(N, seed=62, m=M, k=K)
    C8 = ptc.matmul_s8(int_dev(A8), int_dev(Bt8)).cpu().numpy()
    ii, jj = sample_coords(M, N, 1500, seed=63)
    assert np.array_equal(C8[ii, jj], oracle.wrap_s32(oracle.gemm_s8_at(A8, Bt8, ii, jj)))


def test_auto_shapes_of_the_study_sizes():
    """The automatic choice at the square sizes of the study: narrow tiles
    where the 128 x 256 tiles leave most SMs idle, CTA pairs from N = 2048."""
    shapes = {}
    for n in (512, 1024, 1536, 2048, 4096):
        A = torch.zeros((n, n), dtype=torch.float16, device=DEV)
        ptc.matmul_f16(A, A)
        shapes[n] = ptc.ptc_last_launch()
    torch.cuda.synchronize()
    assert shapes[512][3] == 64 and shapes[1024][3] in (64, 128) and shapes[1536][3] == 128
    assert shapes[2048][1] == 2 and shapes[4096][1] == 2
    # long K over few tiles: K-split clusters (a tile's 256 or 32 K blocks
    # shared by 2-8 CTAs), of 256-wide or narrow tiles
    for (M, N, K) in ((512, 512, 16384), (128, 2048, 2048)):
        A = torch.zeros((M, K), dtype=torch.float16, device=DEV)
        B = torch.zeros((K, N), dtype=torch.float16, device=DEV)
        ptc.matmul_f16(A, B)
        grid, cluster, ks, bn = ptc.ptc_last_launch()
        assert ks > 1 and cluster == ks, (M, N, K, grid, cluster, ks, bn)
    torch.cuda.synchronize()


@pytest.fixture(params=[(64, 2), (64, 4), (128, 2), (128, 4)], ids=["n64-ks2", "n64-ks4", "n128-ks2", "n128-ks4"])
def narrow_ks(request):
    """Narrow tiles in K-split clusters (forced)."""
    bn, ks = request.param
    ptc.ptc_set_tuning("tile_n", bn)
    ptc.ptc_set_tuning("ksplit", ks)
    yield request.param
    ptc.ptc_set_tuning("ksplit", 0)
    ptc.ptc_set_tuning("tile_n", 0)


def _check_narrow_ks(bn, ks, M, N, num_kb):
    grid, cluster, used, tile_n = ptc.ptc_last_launch()
    assert tile_n == bn and used in (1, ks)
    tiles = ((M + 127) // 128) * ((N + bn - 1) // bn)
    if tiles <= 16 and num_kb >= ks:
        assert used == ks and cluster == ks and grid == ks * tiles


# (M, N, K): 512^3 (32 / 16 narrow tiles, 8 K blocks); 300 x 700 x 200 (ragged
# tiles, 4 ragged K blocks, shares 2+2 or 1+1+1+1); 100 x 40 x 1000 (one tile);
# 256 x 384 x 576 (9 K blocks: shares 5+4, 3+2+2+2).
KS_SHAPES = [(512, 512, 512), (300, 700, 200), (100, 40, 1000), (256, 384, 576)]


@pytest.mark.parametrize("M,N,K", KS_SHAPES)
def test_narrow_ksplit_f16(M, N, K, narrow_ks):
    A, B = datagen.f16_operands(N, "normal", seed=M + 5 * N + K, m=M, k=K)
    C = ptc.matmul_f16(padded_f16_dev(A), padded_f16_dev(B), out=out_padded(M, N, torch.float32))
    _check_narrow_ks(*narrow_ks, M, N, (K + 63) // 64)
    check_f16(C.cpu().numpy(), A, B)


@pytest.mark.parametrize("M,N,K", KS_SHAPES)
def test_narrow_ksplit_s8(M, N, K, narrow_ks):
    A, Bt = datagen.s8_operands(N, seed=M + 5 * N + K, m=M, k=K)
    C = ptc.matmul_s8(padded_dev(A), padded_dev(Bt), out=out_padded(M, N, torch.int32))
    _check_narrow_ks(*narrow_ks, M, N, (K + 63) // 64)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


@pytest.mark.parametrize("M,N,K", KS_SHAPES)
def test_narrow_ksplit_s4(M, N, K, narrow_ks):
    A, Bt = datagen.s4_operands(N, seed=M + 5 * N + K, m=M, k=K)
    C = ptc.matmul_s4(padded_dev(A), padded_dev(Bt), K, out=out_padded(M, N, torch.int32))
    _check_narrow_ks(*narrow_ks, M, N, (K + 127) // 128)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s4(A, Bt, K)))


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_narrow_ksplit_scaled(out, narrow_ks):
    M, N, K = 300, 700, 576
    A, Bt = datagen.s8_operands(N, seed=71, m=M, k=K)
    rng = np.random.default_rng(72)
    sa = (rng.standard_normal(M) * 0.01).astype(np.float32)
    sb = (rng.standard_normal(N) * 0.01).astype(np.float32)
    C = ptc.matmul_s8_scaled(padded_dev(A), padded_dev(Bt), torch.from_numpy(sa).to(DEV),
                             torch.from_numpy(sb).to(DEV), out_dtype=out, out=out_padded(M, N, out))
    torch.cuda.synchronize()
    code = {torch.bfloat16: oracle.OUT_BF16, torch.float32: oracle.OUT_F32}[out]
    ref = oracle.dequant(oracle.gemm_s8(A, Bt), sa, sb, code)
    if out == torch.float32:
        got = C.cpu().view(torch.int32).numpy().view(np.uint32)
    else:
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_narrow_ksplit_f16acc_permutation(narrow_ks):
    M, K, N = 300, 576, 700
    perm = np.random.default_rng(73).integers(0, K, size=M)
    A = np.zeros((M, K), np.float16)
    A[np.arange(M), perm] = 1
    B = np.random.default_rng(74).uniform(-100, 100, size=(K, N)).astype(np.float16)
    C = ptc.matmul_f16_f16acc(padded_f16_dev(A.view(np.uint16)), padded_f16_dev(B.view(np.uint16)),
                              out=out_padded(M, N, torch.float16))
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy().astype(np.float64), B.astype(np.float64)[perm])
