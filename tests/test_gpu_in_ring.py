"""GPU parity of the in-ring operand conversion: integer products on one-CTA
shapes load K blocks of the raw s8 / packed s4 operands and convert them in
the GEMM kernel's shared memory (the epilogue warps write the binary16 / E4M3
stage in the 128-byte-swizzled layout the MMAs read).  Every result is checked
bit-exact against the oracle, on ragged M, N and K (a partial last K block,
K below one block), every one-CTA tile width with and without K-split
clusters, folds of many chunks (the conversion then interleaves with the
folds), more tiles than SMs (several units per CTA), the scaled outputs, and
a withheld operand block (the bounded waits of the converting warps report a
timeout and the context survives).  The conversion record says which path
ran: in ring where the shape planner estimates it faster (small products) or
the knob forces it (in_ring = 2, which the exactness tests use), a separate
pass for CTA pairs, for odd K of packed s4 and when the knob turns it off."""
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
    for key, value in (("tile_n", 0), ("ksplit", 0), ("in_ring", 1), ("s8_chunk_kb", 16), ("s4_chunk_kb", 64)):
        ptc.ptc_set_tuning(key, value)
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


def padded_dev(a: np.ndarray) -> torch.Tensor:
    """Device copy with a row pitch rounded up to 32 bytes (s8 pitch rule,
    and 16-byte packed-s4 rows)."""
    rows, cols = a.shape
    w = max(32, (cols + 31) // 32 * 32)
    out = np.zeros((rows, w), dtype=a.dtype)
    out[:, :cols] = a
    return int_dev(out)[:, :cols]


def out_padded(M, N, dtype=torch.int32) -> torch.Tensor:
    per = 16 // torch.empty((), dtype=dtype).element_size()
    return torch.empty((M, (N + per - 1) // per * per), dtype=dtype, device=DEV)[:, :N]


def run_s8(A, Bt):
    M, N = A.shape[0], Bt.shape[0]
    C = ptc.matmul_s8(padded_dev(A), padded_dev(Bt), out=out_padded(M, N))
    mode = ptc.ptc_last_conversion()
    torch.cuda.synchronize()
    return C.cpu().numpy(), mode


def run_s4(A, Bt, K):
    M, N = A.shape[0], Bt.shape[0]
    C = ptc.matmul_s4(padded_dev(A), padded_dev(Bt), K, out=out_padded(M, N))
    mode = ptc.ptc_last_conversion()
    torch.cuda.synchronize()
    return C.cpu().numpy(), mode


@pytest.fixture
def knobs():
    """Set tuning knobs for one test; restored afterwards."""
    saved = {"tile_n": 0, "ksplit": 0, "in_ring": 1, "s8_chunk_kb": 16, "s4_chunk_kb": 64}

    def setter(**kw):
        for k, v in kw.items():
            ptc.ptc_set_tuning(k, v)

    yield setter
    for k, v in saved.items():
        ptc.ptc_set_tuning(k, v)


# (M, N, K): one partial K block; K below one block; ragged everything; an
# exact tile grid; 16 K blocks of s8 (one chunk) / 8 of s4.
SHAPES = [(128, 64, 64), (100, 40, 48), (300, 700, 200), (256, 512, 1024), (77, 130, 1000)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("tile_n,ks", [(64, 1), (64, 4), (128, 1), (128, 2), (256, 1), (256, 2)],
                         ids=["n64", "n64-ks4", "n128", "n128-ks2", "n256", "n256-ks2"])
def test_in_ring_s8_s4_exact(M, N, K, tile_n, ks, knobs):
    knobs(tile_n=tile_n, ksplit=ks, in_ring=2)
    A, Bt = datagen.s8_operands(N, seed=M * 7 + N + K, m=M, k=K)
    C, mode = run_s8(A, Bt)
    assert mode == IN_RING
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    K4 = K + (K & 1)  # even K: the in-ring route of packed s4
    A4, Bt4 = datagen.s4_operands(N, seed=M * 11 + N + K4, m=M, k=K4)
    C4, mode = run_s4(A4, Bt4, K4)
    assert mode == IN_RING
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K4)))


@pytest.mark.parametrize("ks", [1, 2, 4, 8])
def test_in_ring_k_split_256(ks, knobs):
    """128 x 256 tiles in K-split clusters of up to 8 CTAs (M = 256, N = 512:
    four tiles; K = 4096 s8 = 64 K blocks, 32768 s4 = 256 K blocks)."""
    knobs(tile_n=256, ksplit=ks, in_ring=2)
    M, N = 256, 512
    A, Bt = datagen.s8_operands(N, seed=900 + ks, m=M, k=4096)
    C, mode = run_s8(A, Bt)
    assert mode == IN_RING and ptc.ptc_last_launch()[2] == ks
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    A4, Bt4 = datagen.s4_operands(N, seed=910 + ks, m=M, k=32768)
    C4, mode = run_s4(A4, Bt4, 32768)
    assert mode == IN_RING and ptc.ptc_last_launch()[2] == ks
    ii, jj = sample_coords(M, N, 600, seed=911 + ks)
    assert np.array_equal(C4[ii, jj], oracle.wrap_s32(oracle.gemm_s4_at(A4, Bt4, 32768, ii, jj)))


@pytest.mark.parametrize("tile_n", [64, 256])
@pytest.mark.parametrize("chunk", [2, 4, 16])
def test_in_ring_many_chunks(tile_n, chunk, knobs):
    """Folds every `chunk` K blocks over up to 64 K blocks: chunks 2 ... are
    converted between the folds (the accumulator buffers are reused while the
    conversion of later chunks proceeds)."""
    knobs(tile_n=tile_n, s8_chunk_kb=chunk, s4_chunk_kb=chunk, in_ring=2)
    M, N, K = 200, 300, 4000
    A, Bt = datagen.s8_operands(N, seed=920 + chunk, m=M, k=K)
    C, mode = run_s8(A, Bt)
    assert mode == IN_RING
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    A4, Bt4 = datagen.s4_operands(N, seed=930 + chunk, m=M, k=K)
    C4, mode = run_s4(A4, Bt4, K)
    assert mode == IN_RING
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K)))


def test_in_ring_constant_extremes(knobs):
    """Every product at its extreme (-128 * -128, -8 * -8) over K = 2^16 with
    narrow tiles: C = K a b exactly (s8: 2^30)."""
    knobs(tile_n=64, in_ring=2)
    M, N, K = 128, 192, 1 << 16
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


def test_in_ring_several_units_per_cta(knobs):
    """2048 x 2048 outputs in 128 x 64 tiles: 512 tiles over at most one CTA
    per SM, so each CTA converts and multiplies several tiles in turn."""
    knobs(tile_n=64, in_ring=2)
    M, N, K = 2048, 2048, 192
    A, Bt = datagen.s8_operands(N, seed=940, m=M, k=K)
    C, mode = run_s8(A, Bt)
    assert mode == IN_RING and ptc.ptc_last_launch()[0] < 512
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    A4, Bt4 = datagen.s4_operands(N, seed=941, m=M, k=K)
    C4, mode = run_s4(A4, Bt4, K)
    assert mode == IN_RING
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, K)))


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float16, torch.float32], ids=["bf16", "f16", "f32"])
def test_in_ring_scaled(out, knobs):
    knobs(in_ring=2)
    M, N, K = 300, 700, 200
    A, Bt = datagen.s8_operands(N, seed=950, m=M, k=K)
    rng = np.random.default_rng(951)
    sa = (rng.standard_normal(M) * 0.01).astype(np.float32)
    sb = (rng.standard_normal(N) * 0.01).astype(np.float32)
    C = ptc.matmul_s8_scaled(padded_dev(A), padded_dev(Bt), torch.from_numpy(sa).to(DEV),
                             torch.from_numpy(sb).to(DEV), out_dtype=out, out=out_padded(M, N, out))
    assert ptc.ptc_last_conversion() == IN_RING
    torch.cuda.synchronize()
    code = {torch.bfloat16: oracle.OUT_BF16, torch.float16: oracle.OUT_F16, torch.float32: oracle.OUT_F32}[out]
    ref = oracle.dequant(oracle.gemm_s8(A, Bt), sa, sb, code)
    if out == torch.float32:
        got = C.cpu().view(torch.int32).numpy().view(np.uint32)
    else:
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_conversion_record_by_route(knobs):
    """By default in ring for N = 512 (INT8 and INT4), a separate pass for
    CTA pairs, for a long K, for odd K of packed s4, and with the knob off;
    none for FP16."""
    A, Bt = datagen.s8_operands(512, seed=960, m=512, k=512)
    C, mode = run_s8(A, Bt)
    assert mode == IN_RING
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    big = torch.zeros((4096, 512), dtype=torch.int8, device=DEV)
    ptc.matmul_s8(big, big)  # 4096 x 4096 outputs: CTA pairs
    assert ptc.ptc_last_conversion() == SEPARATE and ptc.ptc_last_launch()[1] == 2
    A4e, Bt4e = datagen.s4_operands(512, seed=962)
    C4, mode = run_s4(A4e, Bt4e, 512)
    assert mode == IN_RING
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4e, Bt4e, 512)))
    long_k = torch.zeros((256, 16384), dtype=torch.int8, device=DEV)
    ptc.matmul_s8(long_k, long_k)  # 256 K blocks per tile: the pass
    assert ptc.ptc_last_conversion() == SEPARATE
    # K = 301: the high nibble of each row's last byte (random here) is ignored
    A4, Bt4 = datagen.s4_operands(300, seed=961, m=200, k=302)
    C4, mode = run_s4(A4, Bt4, 301)
    assert mode == SEPARATE
    assert np.array_equal(C4, oracle.wrap_s32(oracle.gemm_s4(A4, Bt4, 301)))
    knobs(in_ring=0)
    C, mode = run_s8(A, Bt)
    assert mode == SEPARATE
    assert np.array_equal(C, oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
    f = torch.zeros((64, 64), dtype=torch.float16, device=DEV)
    ptc.matmul_f16(f, f)
    assert ptc.ptc_last_conversion() == 0
    torch.cuda.synchronize()


def test_in_ring_same_bits_as_separate_pass(knobs):
    """The two conversion paths give the same int32 bits (here on a product
    whose exact sums exceed the int32 range: K = 2^17 of -128 * -128 wraps)."""
    M, N, K = 128, 128, 1 << 17
    A = torch.full((M, K), -128, dtype=torch.int8, device=DEV)
    got = {}
    for flag in (2, 0):
        knobs(in_ring=flag)
        got[flag] = ptc.matmul_s8(A, A).cpu()
        assert ptc.ptc_last_conversion() == (IN_RING if flag else SEPARATE)
    assert torch.equal(got[0], got[2])
    assert int(got[2][0, 0]) == K * 16384 - (1 << 32)  # 2^31 wraps to -2^31


def test_in_ring_wait_timeout_and_recovery(knobs):
    """The first operand block of tile 0 is withheld: the converting warps'
    bounded waits give up after 50 ms, the call reports PTC_ERR_TIMEOUT, and
    the next call on the same context is exact."""
    knobs(in_ring=2)
    M, N, K = 256, 256, 512
    A, Bt = datagen.s8_operands(N, seed=970, m=M, k=K)
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


@pytest.mark.parametrize("prec", ["s8", "s4"])
def test_in_ring_tall_output_many_units(prec, knobs):
    """M = 2^20 rows, N = 40, K = 96 in forced 128 x 64 tiles with in-ring
    conversion: 8192 tiles over at most one CTA per SM (dozens of units per
    CTA, each converted, multiplied and stored in turn), sampled against the
    oracle (the corners and the last row included)."""
    knobs(tile_n=64, in_ring=2)
    M, N, K = 1 << 20, 40, 96
    ii, jj = sample_coords(M, N, 2000, seed=980)
    if prec == "s8":
        A, Bt = datagen.s8_operands(N, seed=981, m=M, k=K)
        C = ptc.matmul_s8(padded_dev(A), padded_dev(Bt), out=out_padded(M, N))
        assert ptc.ptc_last_conversion() == IN_RING
        got = C.cpu().numpy()[ii, jj]
        assert np.array_equal(got, oracle.wrap_s32(oracle.gemm_s8_at(A, Bt, ii, jj)))
    else:
        A, Bt = datagen.s4_operands(N, seed=982, m=M, k=K)
        C = ptc.matmul_s4(padded_dev(A), padded_dev(Bt), K, out=out_padded(M, N))
        assert ptc.ptc_last_conversion() == IN_RING
        got = C.cpu().numpy()[ii, jj]
        assert np.array_equal(got, oracle.wrap_s32(oracle.gemm_s4_at(A, Bt, K, ii, jj)))
