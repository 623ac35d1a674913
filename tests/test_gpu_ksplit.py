"""GPU parity of K-split clusters: when the 128 x 256 one-CTA tiles of a
launch fill at most half of the SMs in one wave, each tile runs on a
thread-block cluster of KS CTAs (2, 4 or 8) that share its K blocks, park
their partial sums in shared memory and add them, in rank order, through
distributed shared memory.

Every shape runs with KS forced to 2, 4 and 8, with the automatic choice and
with the split off, through every route: FP16 within the element-wise bound,
INT8 / INT4 / scaled outputs / FP16-accumulator permutations bit-exact against
the oracle.  The shapes cover ragged M, N and K (a last K block that is
partly past K, K-block counts that do not divide by KS, fewer K blocks than
KS, which runs unsplit), a single tile, and 72 tiles (KS = 2 only).  The launch
record shows which shape ran."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, check_f16, f16_dev, int_dev

pytestmark = pytest.mark.gpu

# (M, N, K): 512^3 is 8 tiles of 8 K blocks (FP16 / INT8; INT4 4 blocks of 128
# values); 300 x 700 x 200 is 9 tiles of 4 ragged blocks; 1000^3 is 32 tiles
# (too many for clusters of 8); 128 x 256 x 576 one tile of 9 blocks (shares
# 2,1,1,.. for KS = 8); 1536 x 1536 x 320 is 72 tiles of 5 blocks; 100 x 40 x
# 1000 one ragged tile of 16 blocks.
SHAPES = [(512, 512, 512), (300, 700, 200), (1000, 1000, 1000), (128, 256, 576), (1536, 1536, 320),
          (100, 40, 1000)]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    ptc.ptc_set_tuning("ksplit", 0)
    ptc.ptc_set_tuning("cta_pair", 0)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.fixture(params=[2, 4, 8, 0, 1], ids=["ks2", "ks4", "ks8", "auto", "off"])
def ks(request):
    ptc.ptc_set_tuning("ksplit", request.param)
    yield request.param
    ptc.ptc_set_tuning("ksplit", 0)


def padded_dev(a: np.ndarray) -> torch.Tensor:
    """Device copy of a (rows, cols) byte matrix with each row padded to a
    16-byte multiple (the library's pitch rule), viewed as (rows, cols)."""
    rows, cols = a.shape
    w = max(16, (cols + 15) // 16 * 16)
    out = np.zeros((rows, w), dtype=a.dtype)
    out[:, :cols] = a
    return int_dev(out)[:, :cols]


def padded_f16_dev(bits: np.ndarray) -> torch.Tensor:
    """The same for binary16 bit patterns (rows padded to 8 values)."""
    rows, cols = bits.shape
    w = max(8, (cols + 7) // 8 * 8)
    out = np.zeros((rows, w), dtype=np.uint16)
    out[:, :cols] = bits
    return f16_dev(out)[:, :cols]


def out_padded(M, N, dtype) -> torch.Tensor:
    """A (M, N) result view whose rows start on 16-byte boundaries."""
    per = 16 // torch.empty((), dtype=dtype).element_size()
    return torch.empty((M, (N + per - 1) // per * per), dtype=dtype, device=DEV)[:, :N]


def _tiles(M, N):
    return ((M + 127) // 128) * ((N + 255) // 256)


def _check_launch(ks, M, N, num_kb):
    """The recorded launch is a K-split cluster launch when it must be: a
    forced KS with at most 8 tiles (clusters of 8 then always fit one wave)
    and at least KS K blocks; by size, 256-wide tiles only when each CTA sheds
    8 or more K blocks, narrow tiles with at least two K blocks per CTA (one
    when the integer operands are converted in the kernel's ring)."""
    grid, cluster, used, tile_n = ptc.ptc_last_launch()
    assert used in (1, 2, 4, 8) and grid > 0 and tile_n in (64, 128, 256)
    tiles = _tiles(M, N)
    if ks == 1:
        assert used == 1
    elif ks in (2, 4, 8):
        assert used in (1, ks)
        if tiles <= 8 and num_kb >= ks:
            assert used == ks
    elif used > 1 and tile_n == 256:
        assert num_kb - (num_kb + used - 1) // used >= 8
    elif used > 1:
        # narrow tiles: at least two K blocks per CTA, or one with in-ring conversion
        assert num_kb >= 2 * used or ptc.ptc_last_conversion() == 2
    if used > 1:
        tiles_bn = ((M + 127) // 128) * ((N + tile_n - 1) // tile_n)
        assert num_kb >= used and cluster == used and grid == used * tiles_bn


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_ksplit_f16(M, N, K, ks):
    A, B = datagen.f16_operands(N, "normal", seed=M + N + K, m=M, k=K)
    C = ptc.matmul_f16(padded_f16_dev(A), padded_f16_dev(B), out=out_padded(M, N, torch.float32))
    _check_launch(ks, M, N, (K + 63) // 64)
    check_f16(C.cpu().numpy(), A, B)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_ksplit_s8(M, N, K, ks):
    A, Bt = datagen.s8_operands(N, seed=M + N + K, m=M, k=K)
    Ad, Bd = padded_dev(A), padded_dev(Bt)
    Cd = torch.empty((M, (N + 3) // 4 * 4), dtype=torch.int32, device=DEV)
    ptc.gemm_s8(M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), Cd.data_ptr(), Cd.shape[1], 0)
    _check_launch(ks, M, N, (K + 63) // 64)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.cpu().numpy()[:, :N], oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_ksplit_s4(M, N, K, ks):
    A, Bt = datagen.s4_operands(N, seed=M + N + K, m=M, k=K)
    C = ptc.matmul_s4(padded_dev(A), padded_dev(Bt), K, out=out_padded(M, N, torch.int32))
    _check_launch(ks, M, N, (K + 127) // 128)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s4(A, Bt, K)))


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float16, torch.float32], ids=["bf16", "f16", "f32"])
@pytest.mark.parametrize("M,N,K", [(300, 700, 200), (128, 256, 576)])
def test_ksplit_s8_scaled(M, N, K, out, ks):
    A, Bt = datagen.s8_operands(N, seed=31 + K, m=M, k=K)
    rng = np.random.default_rng(32 + K)
    sa = (rng.standard_normal(M) * 0.01).astype(np.float32)
    sb = (rng.standard_normal(N) * 0.01).astype(np.float32)
    C = ptc.matmul_s8_scaled(padded_dev(A), padded_dev(Bt), torch.from_numpy(sa).to(DEV),
                             torch.from_numpy(sb).to(DEV), out_dtype=out, out=out_padded(M, N, out))
    _check_launch(ks, M, N, (K + 63) // 64)
    torch.cuda.synchronize()
    code = {torch.bfloat16: oracle.OUT_BF16, torch.float16: oracle.OUT_F16, torch.float32: oracle.OUT_F32}[out]
    ref = oracle.dequant(oracle.gemm_s8(A, Bt), sa, sb, code)
    if out == torch.float32:
        got = C.cpu().view(torch.int32).numpy().view(np.uint32)
    else:
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_ksplit_s4_scaled_f32(ks):
    M, N, K = 300, 700, 1000
    A, Bt = datagen.s4_operands(N, seed=41, m=M, k=K)
    rng = np.random.default_rng(42)
    sa = (rng.standard_normal(M) * 0.01).astype(np.float32)
    sb = (rng.standard_normal(N) * 0.01).astype(np.float32)
    C = ptc.matmul_s4_scaled(padded_dev(A), padded_dev(Bt), K, torch.from_numpy(sa).to(DEV),
                             torch.from_numpy(sb).to(DEV), out_dtype=torch.float32,
                             out=out_padded(M, N, torch.float32))
    _check_launch(ks, M, N, (K + 127) // 128)
    torch.cuda.synchronize()
    ref = oracle.dequant(oracle.gemm_s4(A, Bt, K), sa, sb, oracle.OUT_F32)
    assert np.array_equal(C.cpu().view(torch.int32).numpy().view(np.uint32), ref)


@pytest.mark.parametrize("M,K,N", [(300, 200, 700), (128, 576, 256)])
def test_ksplit_f16acc_permutation(M, K, N, ks):
    """FP16 accumulators: each CTA's partial row is exact (one nonzero term at
    most), so the widened sum and its single rounding reproduce B's rows."""
    perm = np.random.default_rng(5 + K).integers(0, K, size=M)
    A = np.zeros((M, K), np.float16)
    A[np.arange(M), perm] = 1
    B = np.random.default_rng(6 + K).uniform(-100, 100, size=(K, N)).astype(np.float16)
    C = ptc.matmul_f16_f16acc(padded_f16_dev(A.view(np.uint16)), padded_f16_dev(B.view(np.uint16)),
                              out=out_padded(M, N, torch.float16))
    _check_launch(ks, M, N, (K + 63) // 64)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy().astype(np.float64), B.astype(np.float64)[perm])


@pytest.mark.parametrize("M,N,K", [(300, 700, 200), (512, 512, 512)])
def test_ksplit_s8_rowmajor_b(M, N, K, ks):
    A, Bt = datagen.s8_operands(N, seed=M * 17 + K, m=M, k=K)
    B_kn = np.ascontiguousarray(Bt.T)
    Ad, Bd = padded_dev(A), padded_dev(B_kn)
    Cd = torch.empty((M, (N + 3) // 4 * 4), dtype=torch.int32, device=DEV)
    ptc.gemm_s8_b_rowmajor(M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), Cd.data_ptr(),
                           Cd.shape[1], torch.cuda.current_stream().cuda_stream)
    _check_launch(ks, M, N, (K + 63) // 64)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.cpu().numpy()[:, :N], oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


def test_ksplit_reproducible_and_integer_identical():
    """The rank-ordered sum gives the same FP32 bits on every run; integer
    sums do not depend on KS at all."""
    M, N, K = 512, 512, 4096
    A, B = datagen.f16_operands(N, "normal", seed=77, m=M, k=K)
    Ad, Bd = f16_dev(A), f16_dev(B)
    A8, Bt8 = datagen.s8_operands(N, seed=78, m=M, k=K)
    A8d, B8d = int_dev(A8), int_dev(Bt8)
    ints = []
    for ks in (8, 4, 2, 1):
        ptc.ptc_set_tuning("ksplit", ks)
        c1 = ptc.matmul_f16(Ad, Bd).cpu().numpy()
        c2 = ptc.matmul_f16(Ad, Bd).cpu().numpy()
        assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32))
        ints.append(ptc.matmul_s8(A8d, B8d).cpu().numpy())
    ptc.ptc_set_tuning("ksplit", 0)
    for c in ints[1:]:
        assert np.array_equal(c, ints[0])
    assert np.array_equal(ints[0], oracle.wrap_s32(oracle.gemm_s8(A8, Bt8)))
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


def test_ksplit_noalloc():
    """gemm_s8_noalloc (fixed scratch, no workspace) takes K-split clusters too."""
    M, N, K = 300, 700, 1000
    A, Bt = datagen.s8_operands(N, seed=91, m=M, k=K)
    Ad, Bd = padded_dev(A), padded_dev(Bt)
    Cd = torch.empty((M, (N + 3) // 4 * 4), dtype=torch.int32, device=DEV)
    ptc.gemm_s8_noalloc(M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), Cd.data_ptr(),
                        Cd.shape[1], torch.cuda.current_stream().cuda_stream)
    grid, cluster, used, _ = ptc.ptc_last_launch()
    assert used > 1 and grid == used * _tiles(M, N)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.cpu().numpy()[:, :N], oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


@pytest.mark.parametrize("pdl", [0, 1], ids=["plain", "pdl"])
def test_back_to_back_dependent_calls(pdl):
    """Each call reads the previous call's output (C1 = X P, C2 = C1 P, ...,
    FP16 accumulators so that C feeds the next call directly): with
    programmatic serialization the next kernel starts early but must see
    every write of the one before it."""
    ptc.ptc_set_tuning("pdl", pdl)
    try:
        n = 512
        rng = np.random.default_rng(101)
        X = rng.integers(-8, 9, size=(n, n)).astype(np.float16)
        P = np.eye(n, dtype=np.float16)[rng.permutation(n)]
        Pd = torch.from_numpy(P).to(DEV)
        cur = torch.from_numpy(X).to(DEV)
        ref = X.astype(np.float64)
        for _ in range(16):
            cur = ptc.matmul_f16_f16acc(cur, Pd)
            ref = ref @ P.astype(np.float64)
        torch.cuda.synchronize()
        assert np.array_equal(cur.cpu().numpy().astype(np.float64), ref)
    finally:
        ptc.ptc_set_tuning("pdl", 1)


@pytest.mark.parametrize("pdl", [0, 1], ids=["plain", "pdl"])
def test_back_to_back_integer_calls(pdl):
    """Integer calls in a row reuse the stream-ordered workspace: the next
    call's conversion pass may start while the previous GEMM still reads the
    workspace, and must wait for it.  Results of calls issued back to back
    equal those of the same calls run one at a time."""
    ptc.ptc_set_tuning("pdl", pdl)
    try:
        M, N, K = 1024, 1024, 2048
        ops = [datagen.s8_operands(N, seed=200 + i, m=M, k=K) for i in range(6)]
        dev = [(int_dev(a), int_dev(b)) for a, b in ops]
        alone = []
        for a, b in dev:
            alone.append(ptc.matmul_s8(a, b))
            torch.cuda.synchronize()
        together = [ptc.matmul_s8(a, b) for a, b in dev]
        torch.cuda.synchronize()
        for x, y in zip(alone, together):
            assert torch.equal(x, y)
        A, Bt = ops[3]
        ii = np.random.default_rng(5).integers(0, M, 2000)
        jj = np.random.default_rng(6).integers(0, N, 2000)
        got = together[3].cpu().numpy()[ii, jj]
        assert np.array_equal(got, oracle.wrap_s32(oracle.gemm_s8_at(A, Bt, ii, jj)))
        assert ptc.gemm_poll_device_error() == ptc.PTC_OK
    finally:
        ptc.ptc_set_tuning("pdl", 1)
