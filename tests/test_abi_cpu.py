"""The C ABI without a GPU: the library loads, exports every entry point that
include/ptc.h declares, and rejects bad arguments with the documented status
codes before making any CUDA call.

Addresses passed here are never dereferenced: every case is rejected by the
host-side checks (and the one case that gets past them only runs where no GPU
is present, where it must stop at the device check)."""
import ctypes
import os
import re

import pytest
import torch

import precision_tensor_core_gb300 as ptc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ptc.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return ptc.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"gemm_f16", "gemm_s8", "gemm_s4", "gemm_status_string",
            "gemm_poll_device_error"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in ptc.h but not exported"
        # C linkage: the plain name resolves, no mangling
        ctypes.cast(getattr(L, n), ctypes.c_void_p)


def test_python_binding_has_same_names():
    for n in declared_functions():
        assert callable(getattr(ptc, n)), n


BASE = 1 << 40  # fake, 16-byte aligned, never dereferenced


def call(L, name, M, N, K, A, lda, B, ldb, C, ldc):
    return getattr(L, name)(M, N, K, A, lda, B, ldb, C, ldc, None)


def good_args(name, M=64, N=64, K=64):
    A = BASE
    B = BASE + (1 << 30)
    C = BASE + (1 << 31)
    if name in ("gemm_f16", "gemm_s8_b_rowmajor"):
        return dict(M=M, N=N, K=K, A=A, lda=K, B=B, ldb=N, C=C, ldc=N)
    return dict(M=M, N=N, K=K, A=A, lda=K, B=B, ldb=K, C=C, ldc=N)


NAMES = ["gemm_f16", "gemm_s8", "gemm_s4", "gemm_s8_b_rowmajor"]


@pytest.mark.parametrize("name", NAMES)
def test_invalid_sizes_and_pointers(L, name):
    g = good_args(name)
    for bad in [dict(M=-1), dict(N=-5), dict(K=-1), dict(M=(1 << 30) + 1), dict(K=(1 << 31))]:
        assert call(L, name, **{**g, **bad}) == ptc.PTC_ERR_INVALID, bad
    assert call(L, name, **{**g, "C": None}) == ptc.PTC_ERR_INVALID
    assert call(L, name, **{**g, "A": None}) == ptc.PTC_ERR_INVALID
    assert call(L, name, **{**g, "B": None}) == ptc.PTC_ERR_INVALID
    assert call(L, name, **{**g, "lda": g["K"] - 1}) == ptc.PTC_ERR_INVALID
    assert call(L, name, **{**g, "ldc": g["N"] - 4}) == ptc.PTC_ERR_INVALID
    bad_ldb = g["N"] - 1 if name in ("gemm_f16", "gemm_s8_b_rowmajor") else g["K"] - 1
    assert call(L, name, **{**g, "ldb": bad_ldb}) == ptc.PTC_ERR_INVALID


@pytest.mark.parametrize("name", NAMES)
def test_empty_problems_are_noops(L, name):
    g = good_args(name)
    # M == 0 or N == 0: nothing to do, pointers may be NULL, no CUDA call
    assert call(L, name, **{**g, "M": 0, "A": None, "B": None, "C": None}) == ptc.PTC_OK
    assert call(L, name, **{**g, "N": 0, "A": None, "B": None, "C": None}) == ptc.PTC_OK


@pytest.mark.parametrize("name", NAMES)
def test_alignment(L, name):
    g = good_args(name)
    assert call(L, name, **{**g, "A": BASE + 8}) == ptc.PTC_ERR_ALIGN
    assert call(L, name, **{**g, "B": g["B"] + 4}) == ptc.PTC_ERR_ALIGN
    assert call(L, name, **{**g, "C": g["C"] + 4}) == ptc.PTC_ERR_ALIGN
    assert call(L, name, **{**g, "ldc": 66}) == ptc.PTC_ERR_ALIGN
    pitch_bad = {"gemm_f16": 68, "gemm_s8": 72, "gemm_s4": 80, "gemm_s8_b_rowmajor": 72}[name]
    assert call(L, name, **{**g, "lda": pitch_bad}) == ptc.PTC_ERR_ALIGN


def test_s4_odd_leading_dimension_is_invalid(L):
    g = good_args("gemm_s4", K=63)
    assert call(L, "gemm_s4", **{**g, "lda": 65}) == ptc.PTC_ERR_INVALID
    assert call(L, "gemm_s4", **{**g, "ldb": 65}) == ptc.PTC_ERR_INVALID


@pytest.mark.parametrize("name", NAMES)
def test_overlap(L, name):
    g = good_args(name)
    assert call(L, name, **{**g, "C": g["A"]}) == ptc.PTC_ERR_OVERLAP
    assert call(L, name, **{**g, "C": g["B"] + 64}) == ptc.PTC_ERR_OVERLAP
    # adjacent but disjoint is fine up to the device check
    esize = {"gemm_f16": 2, "gemm_s8": 1, "gemm_s4": 0.5, "gemm_s8_b_rowmajor": 1}[name]
    a_end = g["A"] + int(((g["M"] - 1) * g["lda"] + g["K"]) * esize)
    r = call(L, name, **{**g, "C": (a_end + 15) // 16 * 16})
    assert r != ptc.PTC_ERR_OVERLAP


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path only")
@pytest.mark.parametrize("name", NAMES)
def test_no_device_is_reported(L, name):
    assert call(L, name, **good_args(name)) == ptc.PTC_ERR_DEVICE
    assert "PTC_ERR_DEVICE" in ptc.gemm_status_string(ptc.PTC_ERR_DEVICE)
    with pytest.raises(ptc.PtcError) as e:
        getattr(ptc, name)(**good_args(name))
    assert e.value.status == ptc.PTC_ERR_DEVICE


def test_status_strings_and_tuning(L):
    for s in range(8):
        assert ptc.gemm_status_string(s)
    assert "unknown" in ptc.gemm_status_string(99)
    with pytest.raises(ptc.PtcError):
        ptc.ptc_set_tuning("no_such_key", 3)
    with pytest.raises(ptc.PtcError):
        ptc.ptc_set_tuning("s8_chunk_kb", 0)
    assert ptc.ptc_set_tuning("group_m", 16) == 0
    assert ptc.ptc_set_tuning("group_m", 8) == 0
    for key, bad, good in (("split_min_kb", 1, 64), ("tail_split", 2, 1), ("cta_pair", 3, 0),
                           ("s8_chunk_kb", 3, 16), ("s4_chunk_kb", 7, 64), ("pair_stage_kb", 3, 2),
                           ("ksplit", 3, 0), ("ksplit", 16, 0), ("pdl", 2, 1), ("split_reduce", 2, 1), ("tile_n", 32, 0),
                           ("tile_n", 192, 0), ("in_ring", 3, 1), ("in_ring", -1, 1),
                           ("s8_chunk_kb", 18, 16), ("s8_chunk_kb", 1 << 20, 16),
                           ("s4_chunk_kb", 2050, 64), ("s4_chunk_kb", 1 << 20, 64),
                           ("pair_in_ring", 1, 0), ("pair_in_ring", 3, 0),
                           ("multicast", 2, 0), ("multicast", -1, 0), ("conv_fused", 2, 0), ("conv_fused", -1, 0)):
        with pytest.raises(ptc.PtcError):
            ptc.ptc_set_tuning(key, bad)
        assert ptc.ptc_set_tuning(key, good) == 0
    assert isinstance(ptc.ptc_kernel_launch_count(), int)
    # no launch on this (GPU-less) thread yet: the launch record is empty
    assert ptc.ptc_last_launch() == (0, 0, 0, 0)
    assert L.ptc_last_launch(None, None, None, None) == ptc.PTC_ERR_INVALID
    assert ptc.ptc_last_conversion() == 0
    assert L.ptc_last_conversion(None) == ptc.PTC_ERR_INVALID
    # the plan's in_ring output is optional; the others are not
    import ctypes
    c, n, k, r = (ctypes.c_int(0) for _ in range(4))
    assert L.ptc_plan_shape(512, 512, 512, 1, 152, 76, 36, 15, ctypes.byref(c), ctypes.byref(n), ctypes.byref(k),
                            None) == 0
    assert (c.value, n.value, k.value) == ptc.ptc_plan_shape(512, 512, 512, 1)
    assert L.ptc_plan_shape(512, 512, 512, 1, 152, 76, 36, 15, None, ctypes.byref(n), ctypes.byref(k),
                            ctypes.byref(r)) == ptc.PTC_ERR_INVALID
    assert L.ptc_plan_shape(512, 512, 512, 3, 152, 76, 36, 15, ctypes.byref(c), ctypes.byref(n), ctypes.byref(k),
                            ctypes.byref(r)) == ptc.PTC_ERR_INVALID


def test_fold_lengths_are_bounded_by_exactness(L):
    """The fold-length knobs accept exactly the even lengths whose FP32 partial
    sums stay exact integers (|partial| <= 2^24): s8 K blocks of 64 values with
    |ab| <= 2^14 allow at most 16, E4M3 K blocks of 128 values with |ab| <= 2^6
    at most 2048.  A longer fold is refused with PTC_ERR_INVALID and leaves the
    previous value in place."""
    assert L.ptc_set_tuning(b"s8_chunk_kb", 18) == ptc.PTC_ERR_INVALID
    assert "16" in ptc.gemm_status_string(ptc.PTC_ERR_INVALID)
    assert L.ptc_set_tuning(b"s4_chunk_kb", 2050) == ptc.PTC_ERR_INVALID
    for v in (2, 16):
        assert L.ptc_set_tuning(b"s8_chunk_kb", v) == ptc.PTC_OK
    for v in (2, 2048):
        assert L.ptc_set_tuning(b"s4_chunk_kb", v) == ptc.PTC_OK
    assert 16 * 64 * 2 ** 14 == 2 ** 24 and 2048 * 128 * 2 ** 6 == 2 ** 24
    assert L.ptc_set_tuning(b"s8_chunk_kb", 16) == ptc.PTC_OK
    assert L.ptc_set_tuning(b"s4_chunk_kb", 64) == ptc.PTC_OK


@pytest.mark.parametrize("name", NAMES)
def test_leading_dimension_above_limit_is_invalid(L, name):
    """A leading dimension above 2^36 elements is refused before any CUDA call
    (so that the byte extents used by the overlap check cannot overflow)."""
    args = good_args(name)
    for key in ("lda", "ldb", "ldc"):
        if key not in args:
            continue
        bad = dict(args)
        bad[key] = (1 << 36) + 16 * 64
        assert call(L, name, **bad) == ptc.PTC_ERR_INVALID, key


def test_noalloc_leading_dimension_above_limit_is_invalid(L):
    g = good_args("gemm_s8")
    for key in ("lda", "ldb", "ldc"):
        assert call(L, "gemm_s8_noalloc", **{**g, key: (1 << 36) + 1024}) == ptc.PTC_ERR_INVALID, key


def test_clock_probe_read_without_device(L):
    import ctypes
    v = (ctypes.c_uint64 * 3)()
    assert L.ptc_clock_probe_read(None, v, v) == ptc.PTC_ERR_INVALID
    if not torch.cuda.is_available():
        assert L.ptc_clock_probe_read(v, v, v) == ptc.PTC_ERR_DEVICE
    for bad in (2, -1):
        assert L.ptc_set_tuning(b"clock_probe", bad) == ptc.PTC_ERR_INVALID
    assert L.ptc_set_tuning(b"clock_probe", 0) == ptc.PTC_OK


def test_baseline_argument_checks(L):
    """gemm_baseline: unknown variants, a leading dimension above 2^36 and C
    overlapping A are refused before any CUDA call."""
    args = dict(M=64, N=64, K=128, A=BASE, lda=128, B=BASE + (1 << 30), ldb=128, C=BASE + (1 << 31), ldc=64)

    def base(v, **kw):
        a = {**args, **kw}
        return L.gemm_baseline(v, a["M"], a["N"], a["K"], a["A"], a["lda"], a["B"], a["ldb"], a["C"], a["ldc"], None)

    assert base(9) == ptc.PTC_ERR_INVALID and base(-1) == ptc.PTC_ERR_INVALID
    for v in (ptc.PTC_BASELINE_S8_MMA, ptc.PTC_BASELINE_S8_LDMATRIX):
        assert base(v, ldc=(1 << 36) + 64) == ptc.PTC_ERR_INVALID
        assert base(v, C=BASE + 64 * 64) == ptc.PTC_ERR_OVERLAP
        # a pitch so large that (M - 1) * pitch leaves 64 bits is refused, not wrapped
        assert base(v, lda=(1 << 36) + 16) == ptc.PTC_ERR_INVALID
