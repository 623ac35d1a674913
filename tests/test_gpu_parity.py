"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle
on the same seeded inputs.

Bars: INT8 and INT4 bit-exact (wrapped to int32); FP16 element-wise
|C - Cref| <= 1e-3 * sum_k |a_ik b_kj| + 1e-6 and relative Frobenius error
<= 1e-4.  Sizes span several 128 x 256 output tiles with ragged tails; the
full-size workloads (N = 8192) run through the same entry points and default
launch configuration as the benchmark and are checked on sampled elements.
"""
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
    ptc.lib()
    yield
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.fixture(params=[1, 2], ids=["cta1", "cta2"])
def cta_mode(request):
    """Run the test with one CTA per 128 x 256 tile, then with CTA pairs on
    256 x 256 tiles (tcgen05 cta_group::2), whatever the problem size."""
    ptc.ptc_set_tuning("cta_pair", request.param)
    yield request.param
    ptc.ptc_set_tuning("cta_pair", 0)


def run_f16(A, B):
    C = ptc.matmul_f16(f16_dev(A), f16_dev(B))
    torch.cuda.synchronize()
    return C.cpu().numpy()


def run_s8(A, Bt):
    C = ptc.matmul_s8(int_dev(A), int_dev(Bt))
    torch.cuda.synchronize()
    return C.cpu().numpy()


def run_s4(A, Bt, K):
    C = ptc.matmul_s4(int_dev(A), int_dev(Bt), K)
    torch.cuda.synchronize()
    return C.cpu().numpy()


def pad_cols(a, mult):
    """Copy rows into a wider array so the row pitch meets the alignment rule."""
    rows, cols = a.shape
    w = max(mult, (cols + mult - 1) // mult * mult)
    out = np.zeros((rows, w), dtype=a.dtype)
    out[:, :cols] = a
    return out


def s4_packed_padded(vals):
    """Pack s4 values (rows, K) and pad each row to a 16-byte multiple."""
    K = vals.shape[1]
    v = np.zeros((vals.shape[0], K + (K & 1)), dtype=np.int8)
    v[:, :K] = vals
    return pad_cols(datagen.pack_s4_rows(v), 16)


# ---------------------------------------------------------------- workloads
def test_fp16_512_uniform_full():
    A, B = datagen.f16_operands(512, "uniform")
    check_f16(run_f16(A, B), A, B)


def test_int8_2048_full():
    A, Bt = datagen.s8_operands(2048)
    assert np.array_equal(run_s8(A, Bt), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


def test_int4_2048_full():
    A, Bt = datagen.s4_operands(2048)
    assert np.array_equal(run_s4(A, Bt, 2048), oracle.wrap_s32(oracle.gemm_s4(A, Bt, 2048)))


def test_fp16_8192_normal_sampled():
    A, B = datagen.f16_operands(8192, "normal")
    C = run_f16(A, B)
    assert np.all(np.isfinite(C))
    check_f16_sampled(C, A, B, n=3000)


@pytest.mark.parametrize("N", [512, 1024, 2048, 4096, 8192])
@pytest.mark.parametrize("prec", ["f16", "s8", "s4"])
def test_sweep(prec, N):
    if prec == "f16":
        A, B = datagen.f16_operands(N, "normal")
        C = run_f16(A, B)
        if N <= 1024:
            check_f16(C, A, B)
        else:
            check_f16_sampled(C, A, B, n=1500)
        return
    if prec == "s8":
        A, Bt = datagen.s8_operands(N)
        C = run_s8(A, Bt)
        if N <= 2048:
            assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
        else:
            ii, jj = sample_coords(N, N, 4000)
            assert np.array_equal(C[ii, jj], oracle.wrap_s32(oracle.gemm_s8_at(A, Bt, ii, jj)))
        return
    A, Bt = datagen.s4_operands(N)
    C = run_s4(A, Bt, N)
    if N <= 2048:
        assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s4(A, Bt, N)))
    else:
        ii, jj = sample_coords(N, N, 4000)
        assert np.array_equal(C[ii, jj], oracle.wrap_s32(oracle.gemm_s4_at(A, Bt, N, ii, jj)))


# ---------------------------------------------------------------- edges
RAGGED = [(1, 1, 1), (15, 17, 9), (31, 33, 64), (33, 31, 65), (127, 255, 63), (128, 256, 64),
          (129, 257, 129), (200, 300, 160), (300, 520, 200), (257, 513, 1000), (64, 1000, 33)]


@pytest.mark.parametrize("M,N,K", RAGGED)
def test_ragged_f16(M, N, K, cta_mode):
    A, B = datagen.f16_operands(N, "uniform", seed=M * 7919 + K, m=M, k=K)
    A, B = pad_cols(A, 8), pad_cols(B, 8)
    Cd = torch.empty((M, max(4, (N + 3) // 4 * 4)), dtype=torch.float32, device=DEV)
    Ad, Bd = f16_dev(A), f16_dev(B)
    ptc.gemm_f16(M, N, K, Ad.data_ptr(), Ad.shape[1], Bd.data_ptr(), Bd.shape[1],
                 Cd.data_ptr(), Cd.shape[1], torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    check_f16(Cd.cpu().numpy()[:, :N], A[:, :K], B[:K, :N])


@pytest.mark.parametrize("M,N,K", RAGGED)
def test_ragged_s8(M, N, K, cta_mode):
    A, Bt = datagen.s8_operands(N, seed=M * 31 + K, m=M, k=K)
    A, Bt = pad_cols(A, 16), pad_cols(Bt, 16)
    Cd = torch.empty((M, max(4, (N + 3) // 4 * 4)), dtype=torch.int32, device=DEV)
    Ad, Bd = int_dev(A), int_dev(Bt)
    ptc.gemm_s8(M, N, K, Ad.data_ptr(), Ad.shape[1], Bd.data_ptr(), Bd.shape[1],
                Cd.data_ptr(), Cd.shape[1], torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref = oracle.wrap_s32(oracle.gemm_s8(A[:, :K], Bt[:, :K]))
    assert np.array_equal(Cd.cpu().numpy()[:, :N], ref)


@pytest.mark.parametrize("M,N,K", RAGGED)
def test_ragged_s4(M, N, K, cta_mode):
    rng = np.random.default_rng(M * 131 + N + K)
    Av = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    Bv = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    Ap, Bp = s4_packed_padded(Av), s4_packed_padded(Bv)
    Cd = torch.empty((M, max(4, (N + 3) // 4 * 4)), dtype=torch.int32, device=DEV)
    Ad, Bd = int_dev(Ap), int_dev(Bp)
    ptc.gemm_s4(M, N, K, Ad.data_ptr(), 2 * Ap.shape[1], Bd.data_ptr(), 2 * Bp.shape[1],
                Cd.data_ptr(), Cd.shape[1], torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref = oracle.wrap_s32(oracle.gemm_s4(Ap, Bp, K))
    assert np.array_equal(Cd.cpu().numpy()[:, :N], ref)


@pytest.mark.parametrize("K", [63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1023, 1024, 1025])
def test_k_boundaries_int(K, cta_mode):
    M, N = 136, 264
    A, Bt = datagen.s8_operands(N, seed=K, m=M, k=K)
    A, Bt = pad_cols(A, 16), pad_cols(Bt, 16)
    Cd = torch.empty((M, N), dtype=torch.int32, device=DEV)
    Ad, Bd = int_dev(A), int_dev(Bt)
    ptc.gemm_s8(M, N, K, Ad.data_ptr(), A.shape[1], Bd.data_ptr(), Bt.shape[1], Cd.data_ptr(), N, 0)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A[:, :K], Bt[:, :K])))
    Av = datagen.uniform_s4_values(K + 1, M, K)
    Bv = datagen.uniform_s4_values(K + 2, N, K)
    Ap, Bp = s4_packed_padded(Av), s4_packed_padded(Bv)
    Ad, Bd = int_dev(Ap), int_dev(Bp)
    ptc.gemm_s4(M, N, K, Ad.data_ptr(), 2 * Ap.shape[1], Bd.data_ptr(), 2 * Bp.shape[1], Cd.data_ptr(), N, 0)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s4(Ap, Bp, K)))


@pytest.mark.parametrize("prec", ["f16", "s8", "s4"])
def test_zero_k_writes_zeros(prec, cta_mode):
    M, N = 70, 90
    dt = torch.float32 if prec == "f16" else torch.int32
    Cd = torch.full((M, 92), 7, dtype=dt, device=DEV)
    fn = {"f16": ptc.gemm_f16, "s8": ptc.gemm_s8, "s4": ptc.gemm_s4}[prec]
    fn(M, N, 0, 0, 0, 0, 0, Cd.data_ptr(), 92, 0)
    torch.cuda.synchronize()
    c = Cd.cpu().numpy()
    assert np.all(c[:, :N] == 0) and np.all(c[:, N:] == 7)


def test_identity_and_permutation_exact(cta_mode):
    K = N = 384
    M = 256
    A = np.zeros((M, K))
    perm = np.random.default_rng(1).permutation(K)[:M]
    A[np.arange(M), perm] = 1.0
    B = np.random.default_rng(2).uniform(-3, 3, size=(K, N)).astype(np.float16)
    C = run_f16(A.astype(np.float16).view(np.uint16), B.view(np.uint16))
    assert np.array_equal(C, B.astype(np.float32)[perm])
    A8 = A.astype(np.int8)
    Bt8 = np.random.default_rng(3).integers(-128, 128, size=(N, K)).astype(np.int8)
    assert np.array_equal(run_s8(A8, Bt8), Bt8.T[perm].astype(np.int32))
    Bt4 = np.random.default_rng(4).integers(-8, 8, size=(N, K)).astype(np.int8)
    C4 = run_s4(datagen.pack_s4_rows(A8), datagen.pack_s4_rows(Bt4), K)
    assert np.array_equal(C4, Bt4.T[perm].astype(np.int32))


def test_mma_lab_worked_example(golden_dir, cta_mode):
    import os
    from tests.test_oracle_pins import _read_golden
    g = _read_golden(os.path.join(golden_dir, "mma_lab_m16n8k16.txt"))
    M, N, K = g["shape"]
    B = np.array([[8 * r + c + 1 for c in range(N)] for r in range(K)], dtype=np.float16)
    A = np.eye(M, K, dtype=np.float16)
    C = run_f16(A.view(np.uint16), B.view(np.uint16))
    for (r, c, v) in g["point"]:
        assert C[r, c] == v
    C2 = run_f16(np.ascontiguousarray(A[::-1]).view(np.uint16), B.view(np.uint16))
    assert C2[0].tolist() == g["reversed_row0"]


@pytest.mark.parametrize("prec", ["f16", "s8", "s4"])
def test_guard_bands_untouched(prec, cta_mode):
    """Output slots outside the M x N block (row padding and rows past M) keep
    the sentinel 0xdeadbeef."""
    M, N, K = 130, 264, 96
    ldc = 272
    sentinel = np.int32(np.uint32(0xDEADBEEF).view(np.int32))
    Cd = torch.full((M + 3, ldc), int(sentinel), dtype=torch.int32, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    if prec == "f16":
        A, B = datagen.f16_operands(N, "uniform", m=M, k=K)
        Ad, Bd = f16_dev(A), f16_dev(B)
        ptc.gemm_f16(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, Cd.data_ptr(), ldc, s)
    elif prec == "s8":
        A, Bt = datagen.s8_operands(N, m=M, k=K)
        Ad, Bd = int_dev(A), int_dev(Bt)
        ptc.gemm_s8(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), ldc, s)
    else:
        A, Bt = datagen.s4_operands(N, m=M, k=K)
        Ad, Bd = int_dev(A), int_dev(Bt)
        ptc.gemm_s4(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), ldc, s)
    torch.cuda.synchronize()
    c = Cd.cpu().numpy()
    assert np.all(c[:, N:] == sentinel)
    assert np.all(c[M:, :] == sentinel)
    if prec == "f16":
        check_f16(c[:M, :N].view(np.float32), A, B)
    elif prec == "s8":
        assert np.array_equal(c[:M, :N], oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    else:
        assert np.array_equal(c[:M, :N], oracle.wrap_s32(oracle.gemm_s4(A, Bt, K)))


def test_strided_operands_padding_not_read(cta_mode):
    """Leading dimensions larger than the logical width; the padding holds
    values that would change the result if they were read."""
    M, N, K = 150, 270, 100
    A, B = datagen.f16_operands(N, "uniform", m=M, k=K)
    Ap = np.full((M, 136), np.float16(1000.0).view(np.uint16), dtype=np.uint16)
    Ap[:, :K] = A
    Bp = np.full((K, 280), np.float16(-1000.0).view(np.uint16), dtype=np.uint16)
    Bp[:, :N] = B
    Ad, Bd = f16_dev(Ap), f16_dev(Bp)
    Cd = torch.empty((M, 272), dtype=torch.float32, device=DEV)
    ptc.gemm_f16(M, N, K, Ad.data_ptr(), 136, Bd.data_ptr(), 280, Cd.data_ptr(), 272, 0)
    torch.cuda.synchronize()
    check_f16(Cd.cpu().numpy()[:, :N], A, B)
    A8, Bt8 = datagen.s8_operands(N, m=M, k=K)
    A8p = np.full((M, 128), 127, np.int8); A8p[:, :K] = A8
    B8p = np.full((N, 144), -128, np.int8); B8p[:, :K] = Bt8
    Ci = torch.empty((M, 272), dtype=torch.int32, device=DEV)
    A8d, B8d = int_dev(A8p), int_dev(B8p)  # keep the device copies alive across the call
    ptc.gemm_s8(M, N, K, A8d.data_ptr(), 128, B8d.data_ptr(), 144, Ci.data_ptr(), 272, 0)
    torch.cuda.synchronize()
    assert np.array_equal(Ci.cpu().numpy()[:, :N], oracle.wrap_s32(oracle.gemm_s8(A8, Bt8)))


# ---------------------------------------------------------------- integer exactness
def test_int8_extremes_and_cancellation_k8192(cta_mode):
    """(-128)(-128) summed over K = 8192 is 2^27 (FP32 alone would round it);
    the cancellation adversary has exact result 0 with partial sums ~2^26."""
    K, M, N = 8192, 130, 260
    A = np.full((M, K), -128, np.int8)
    Bt = np.full((N, K), -128, np.int8)
    Bt[1::2] = 127
    C = run_s8(A, Bt)
    ref = oracle.wrap_s32(oracle.gemm_s8(A, Bt))
    assert np.array_equal(C, ref) and ref[0, 0] == 2 ** 27
    A = np.full((M, K), 127, np.int8)
    Bt = np.full((N, K), 127, np.int8)
    for j in range(N):
        Bt[j, (np.arange(K) + 37 * j) % K >= K // 2] = -127
    Bt[5, 3] = 0  # one column with a nonzero exact result
    C = run_s8(A, Bt)
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


def test_int4_extremes_and_cancellation_k8192(cta_mode):
    K, M, N = 8192, 130, 260
    pk = lambda v, r: datagen.pack_s4_rows(np.full((r, K), v, np.int8))
    C = run_s4(pk(-8, M), pk(-8, N), K)
    assert np.all(C == 64 * K)
    Av = np.full((M, K), 7, np.int8)
    Bv = np.full((N, K), 7, np.int8)
    for j in range(N):
        Bv[j, (np.arange(K) + 53 * j) % K >= K // 2] = -7
    Bv[7, 11] = 3
    Ap, Bp = datagen.pack_s4_rows(Av), datagen.pack_s4_rows(Bv)
    assert np.array_equal(run_s4(Ap, Bp, K), oracle.wrap_s32(oracle.gemm_s4(Ap, Bp, K)))
    Av = np.full((M, K), -8, np.int8)
    Bv = np.full((N, K), 7, np.int8)
    Bv[::3] = -8
    Ap, Bp = datagen.pack_s4_rows(Av), datagen.pack_s4_rows(Bv)
    assert np.array_equal(run_s4(Ap, Bp, K), oracle.wrap_s32(oracle.gemm_s4(Ap, Bp, K)))


def test_int8_odd_partial_sums_up_to_2_24(cta_mode):
    """Every fold of the INT8 route sums 1024 K values; with A = 127 and B = 127
    except one 126 per 16 values, each 16-product group sums to an odd number
    and the partial sums climb to 64 * 257937 = 16,507,968 < 2^24 through odd
    values, so any accumulation narrower than 24 bits drops a unit."""
    K, M, N = 8192, 128, 256
    A = np.full((M, K), 127, np.int8)
    Bt = np.full((N, K), 127, np.int8)
    for j in range(N):
        Bt[j, (np.arange(K) % 16) == (j % 16)] = 126
        if j % 2:
            Bt[j] = -Bt[j]
    C = run_s8(A, Bt)
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))


def test_int4_odd_partial_sums(cta_mode):
    """INT4 route: A = 7, B = 7 except one 6 per 32 values, so each 32-product
    group sums to the odd 1561 and the running sums stay odd-valued as they
    grow; with a wrap pattern per column."""
    K, M, N = 8192, 128, 256
    Av = np.full((M, K), 7, np.int8)
    Bv = np.full((N, K), 7, np.int8)
    for j in range(N):
        Bv[j, (np.arange(K) % 32) == (j % 32)] = 6
        if j % 3 == 1:
            Bv[j] = -Bv[j]
    Av[1::2] = -8
    Ap, Bp = datagen.pack_s4_rows(Av), datagen.pack_s4_rows(Bv)
    assert np.array_equal(run_s4(Ap, Bp, K), oracle.wrap_s32(oracle.gemm_s4(Ap, Bp, K)))


# ---------------------------------------------------------------- runtime behaviour
@pytest.mark.parametrize("prec", ["f16", "s8", "s4"])
def test_deterministic(prec):
    N = 1024
    if prec == "f16":
        A, B = datagen.f16_operands(N, "normal")
        r1, r2 = run_f16(A, B), run_f16(A, B)
    elif prec == "s8":
        A, B = datagen.s8_operands(N)
        r1, r2 = run_s8(A, B), run_s8(A, B)
    else:
        A, B = datagen.s4_operands(N)
        r1, r2 = run_s4(A, B, N), run_s4(A, B, N)
    assert np.array_equal(r1.view(np.uint32), r2.view(np.uint32))


def test_side_stream_and_launch_count():
    A, B = datagen.f16_operands(640, "uniform")
    Ad, Bd = f16_dev(A), f16_dev(B)
    A8, B8 = datagen.s8_operands(640)
    A8d, B8d = int_dev(A8), int_dev(B8)
    s = torch.cuda.Stream()
    before = ptc.ptc_kernel_launch_count()
    with torch.cuda.stream(s):
        C = ptc.matmul_f16(Ad, Bd)
        C8 = ptc.matmul_s8(A8d, B8d)
        conv = ptc.ptc_last_conversion()
    # FP16: the GEMM; INT8: the GEMM, after a conversion pass unless the
    # operands were converted in the kernel's ring (this size: in ring)
    assert conv == 2
    assert ptc.ptc_kernel_launch_count() - before == 1 + (1 if conv == 2 else 2)
    s.synchronize()
    check_f16(C.cpu().numpy(), A, B)
    assert np.array_equal(C8.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A8, B8)))


def test_host_tensors_end_to_end():
    A, B = datagen.f16_operands(296, "uniform", m=200, k=120)
    C = ptc.matmul_f16(torch.from_numpy(A.view(np.float16)).pin_memory(),
                       torch.from_numpy(B.view(np.float16)).pin_memory())
    assert C.device.type == "cpu"
    check_f16(C.numpy(), A, B)


def test_wait_timeout_is_reported_and_context_survives(cta_mode):
    """A kernel whose operands for one tile are withheld gives up after the
    (shortened) wait limit, reports PTC_ERR_TIMEOUT, and the context stays
    usable for the next call."""
    M, N, K = 256, 512, 256
    A, B = datagen.f16_operands(N, "uniform", m=M, k=K)
    Ad, Bd = f16_dev(A), f16_dev(B)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK
    ptc.ptc_debug_set_wait_limit(50_000_000, stall_tile=0)  # 50 ms, stall tile 0
    try:
        ptc.matmul_f16(Ad, Bd)
        torch.cuda.synchronize()
        assert ptc.gemm_poll_device_error() == ptc.PTC_ERR_TIMEOUT
    finally:
        ptc.ptc_debug_set_wait_limit(0, -1)
    C = ptc.matmul_f16(Ad, Bd)
    torch.cuda.synchronize()
    check_f16(C.cpu().numpy(), A, B)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


@pytest.mark.parametrize("stage_kb", [1, 2])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (257, 513, 1000), (512, 1024, 4160), (136, 264, 129)])
def test_pair_ring_stage_depths(M, N, K, stage_kb):
    """CTA pairs with one- or two-block ring stages (odd K block counts leave a
    zero-filled block in the last two-block stage)."""
    ptc.ptc_set_tuning("cta_pair", 2)
    ptc.ptc_set_tuning("pair_stage_kb", stage_kb)
    try:
        A, B = datagen.f16_operands(N, "normal", seed=M + K, m=M, k=K)
        A, B = pad_cols(A, 8), pad_cols(B, 8)
        Cd = torch.empty((M, (N + 3) // 4 * 4), dtype=torch.float32, device=DEV)
        Ad, Bd = f16_dev(A), f16_dev(B)
        ptc.gemm_f16(M, N, K, Ad.data_ptr(), Ad.shape[1], Bd.data_ptr(), Bd.shape[1], Cd.data_ptr(), Cd.shape[1], 0)
        torch.cuda.synchronize()
        check_f16(Cd.cpu().numpy()[:, :N], A[:, :K], B[:K, :N])
        A8, Bt8 = datagen.s8_operands(N, seed=M + K + 1, m=M, k=K)
        A8, Bt8 = pad_cols(A8, 16), pad_cols(Bt8, 16)
        Ci = torch.empty((M, (N + 3) // 4 * 4), dtype=torch.int32, device=DEV)
        Ad, Bd = int_dev(A8), int_dev(Bt8)
        ptc.gemm_s8(M, N, K, Ad.data_ptr(), A8.shape[1], Bd.data_ptr(), Bt8.shape[1], Ci.data_ptr(), Ci.shape[1], 0)
        torch.cuda.synchronize()
        assert np.array_equal(Ci.cpu().numpy()[:, :N], oracle.wrap_s32(oracle.gemm_s8(A8[:, :K], Bt8[:, :K])))
        Ap = s4_packed_padded(datagen.uniform_s4_values(M + K + 2, M, K))
        Bp = s4_packed_padded(datagen.uniform_s4_values(M + K + 3, N, K))
        Ad, Bd = int_dev(Ap), int_dev(Bp)
        ptc.gemm_s4(M, N, K, Ad.data_ptr(), 2 * Ap.shape[1], Bd.data_ptr(), 2 * Bp.shape[1], Ci.data_ptr(),
                    Ci.shape[1], 0)
        torch.cuda.synchronize()
        assert np.array_equal(Ci.cpu().numpy()[:, :N], oracle.wrap_s32(oracle.gemm_s4(Ap, Bp, K)))
    finally:
        ptc.ptc_set_tuning("pair_stage_kb", 2)
        ptc.ptc_set_tuning("cta_pair", 0)


def test_clock_probe_records_each_kernel_family():
    """With the clock record on, each GEMM family's CTAs add their cycle and
    nanosecond counts; the ratio is a plausible SM clock and the results are
    unchanged."""
    ptc.ptc_clock_probe_read()
    ptc.ptc_set_tuning("clock_probe", 1)
    try:
        A, B = datagen.f16_operands(1024, "normal")
        C16 = run_f16(A, B)
        A8, Bt8 = datagen.s8_operands(1024)
        C8 = run_s8(A8, Bt8)
        A4, Bt4 = datagen.s4_operands(1024)
        C4 = run_s4(A4, Bt4, 1024)
    finally:
        ptc.ptc_set_tuning("clock_probe", 0)
    cyc, ns, ctas = ptc.ptc_clock_probe_read()
    for f in range(3):
        assert ctas[f] > 0 and ns[f] > 0
        mhz = 1e3 * cyc[f] / ns[f]
        assert 300.0 < mhz < 2500.0, (f, mhz)
    assert ptc.ptc_clock_probe_read()[2] == [0, 0, 0]  # read and cleared
    check_f16(C16, A, B)
    assert np.array_equal(C8, oracle.wrap_s32(oracle.gemm_s8(A8, Bt8)))
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, 1024)))
