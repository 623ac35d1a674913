"""CPU oracle for C = A.B in FP16 (FP64 sums), INT8 and packed INT4 (exact sums).

TEST INFRASTRUCTURE ONLY: the independent checker of the GPU library.  Only the
test suite, the smoke check and the benchmark's CPU-baseline leg may import
this package.  It shares no code with the CUDA path; the two meet only in the
seeded input generators of ``datagen``.

The arithmetic lives in ``oracle.c`` (plain C, one loop over k per output
element, see its header for the citations).  This module compiles it with gcc
on first use (or via ``build()``), loads it with ctypes and marshals numpy
arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared",
                               "-ffp-contract=off", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = _load(_LIB)
    return _lib


def _load(path: str):
    """Load an oracle shared library and declare its signatures."""
    L = ctypes.CDLL(path)
    L.oracle_f16_to_f64.restype = ctypes.c_double
    L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_s4_get.restype = ctypes.c_int
    L.oracle_s4_get.argtypes = [_vp, _i64]
    L.oracle_unpack_s4.argtypes = [_i64, _i64, _vp, _i64, _vp, _i64]
    L.oracle_pack_s4.argtypes = [_i64, _i64, _vp, _i64, _vp, _i64]
    L.oracle_gemm_f16.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp,
                                  _i64, ctypes.c_int]
    L.oracle_gemm_s8.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                 ctypes.c_int]
    L.oracle_gemm_s4.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                 ctypes.c_int]
    L.oracle_gemm_f16_at.argtypes = [_i64, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _vp]
    L.oracle_gemm_s8_at.argtypes = [_i64, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp]
    L.oracle_gemm_s4_at.argtypes = [_i64, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp]
    L.oracle_wrap_s32.restype = ctypes.c_int32
    L.oracle_wrap_s32.argtypes = [_i64]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_f16.restype = ctypes.c_uint16
    L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    L.oracle_dequant.argtypes = [_i64, _i64, _vp, _i64, _vp, _vp, ctypes.c_int, _vp, _i64]
    return L


class swapped_library:
    """Context manager that points this module at another build of oracle.c
    (used by the tests that plant mistakes in a copy of the oracle)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self._saved = lib()
        _lib = _load(self.path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_vp)


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def f16_to_f64(bits) -> np.ndarray:
    """Decode uint16 binary16 bit patterns to float64 (the oracle's decoder)."""
    L = lib()
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    flat = out.reshape(-1)
    for i, h in enumerate(b.reshape(-1).tolist()):
        flat[i] = L.oracle_f16_to_f64(h)
    return out


def unpack_s4(packed: np.ndarray, cols: int, ld: int | None = None) -> np.ndarray:
    """Packed s4 rows (rows, ld/2 bytes) -> int8 values (rows, cols)."""
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    ld = p.shape[1] * 2 if ld is None else ld
    out = np.empty((p.shape[0], cols), dtype=np.int8)
    lib().oracle_unpack_s4(p.shape[0], cols, _ptr(p), ld, _ptr(out), cols)
    return out


def pack_s4(values: np.ndarray, ld: int | None = None) -> np.ndarray:
    """int8 values in [-8, 7] (rows, cols) -> packed s4 rows (rows, ld/2 bytes)."""
    v = np.ascontiguousarray(values, dtype=np.int8)
    ld = v.shape[1] + (v.shape[1] & 1) if ld is None else ld
    out = np.empty((v.shape[0], ld // 2), dtype=np.uint8)
    lib().oracle_pack_s4(v.shape[0], v.shape[1], _ptr(v), v.shape[1], _ptr(out), ld)
    return out


def gemm_f16(A: np.ndarray, B: np.ndarray, nthreads: int | None = None):
    """FP16 A (M,K) and B (K,N) as uint16 bit patterns -> (C, S) float64 (M,N).

    C = sum_k A_ik B_kj in FP64, S = sum_k |A_ik B_kj|.
    """
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    lib().oracle_gemm_f16(M, N, K, _ptr(A), K, _ptr(B), N, _ptr(C), _ptr(S), N,
                          _threads(nthreads))
    return C, S


def gemm_s8(A: np.ndarray, Bt: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """INT8 A (M,K) row-major and B column-major given as Bt (N,K) -> exact int64 C."""
    A = np.ascontiguousarray(A, dtype=np.int8)
    Bt = np.ascontiguousarray(Bt, dtype=np.int8)
    M, K = A.shape
    N, K2 = Bt.shape
    assert K == K2
    C = np.empty((M, N), dtype=np.int64)
    lib().oracle_gemm_s8(M, N, K, _ptr(A), K, _ptr(Bt), K, _ptr(C), N, _threads(nthreads))
    return C


def gemm_s4(A: np.ndarray, Bt: np.ndarray, K: int, nthreads: int | None = None) -> np.ndarray:
    """Packed s4 A (M, lda/2) and column-major B as Bt (N, ldb/2) -> exact int64 C."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    Bt = np.ascontiguousarray(Bt, dtype=np.uint8)
    M, N = A.shape[0], Bt.shape[0]
    lda, ldb = 2 * A.shape[1], 2 * Bt.shape[1]
    assert K <= lda and K <= ldb
    C = np.empty((M, N), dtype=np.int64)
    lib().oracle_gemm_s4(M, N, K, _ptr(A), lda, _ptr(Bt), ldb, _ptr(C), N, _threads(nthreads))
    return C


def _coords(ii, jj):
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    assert ii.shape == jj.shape
    return ii, jj


def gemm_f16_at(A: np.ndarray, B: np.ndarray, ii, jj):
    """Sampled FP16 outputs C[ii[p], jj[p]] and S[...] (float64)."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    ii, jj = _coords(ii, jj)
    C = np.empty(ii.shape, dtype=np.float64)
    S = np.empty(ii.shape, dtype=np.float64)
    lib().oracle_gemm_f16_at(A.shape[1], _ptr(A), A.shape[1], _ptr(B), B.shape[1],
                             ii.size, _ptr(ii), _ptr(jj), _ptr(C), _ptr(S))
    return C, S


def gemm_s8_at(A: np.ndarray, Bt: np.ndarray, ii, jj) -> np.ndarray:
    """Sampled exact INT8 outputs C[ii[p], jj[p]] (int64)."""
    A = np.ascontiguousarray(A, dtype=np.int8)
    Bt = np.ascontiguousarray(Bt, dtype=np.int8)
    ii, jj = _coords(ii, jj)
    C = np.empty(ii.shape, dtype=np.int64)
    lib().oracle_gemm_s8_at(A.shape[1], _ptr(A), A.shape[1], _ptr(Bt), Bt.shape[1],
                            ii.size, _ptr(ii), _ptr(jj), _ptr(C))
    return C


def gemm_s4_at(A: np.ndarray, Bt: np.ndarray, K: int, ii, jj) -> np.ndarray:
    """Sampled exact INT4 outputs C[ii[p], jj[p]] (int64)."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    Bt = np.ascontiguousarray(Bt, dtype=np.uint8)
    ii, jj = _coords(ii, jj)
    C = np.empty(ii.shape, dtype=np.int64)
    lib().oracle_gemm_s4_at(K, _ptr(A), 2 * A.shape[1], _ptr(Bt), 2 * Bt.shape[1],
                            ii.size, _ptr(ii), _ptr(jj), _ptr(C))
    return C


OUT_F32, OUT_BF16, OUT_F16 = 0, 1, 2


def dequant(acc: np.ndarray, scale_a=None, scale_b=None, out_type: int = OUT_F32) -> np.ndarray:
    """Scaled integer GEMM epilogue applied to exact sums (int64, M x N).
    Returns bit patterns: uint32 (binary32) for OUT_F32, uint16 otherwise."""
    acc = np.ascontiguousarray(acc, dtype=np.int64)
    M, N = acc.shape
    sa = None if scale_a is None else np.ascontiguousarray(scale_a, dtype=np.float32)
    sb = None if scale_b is None else np.ascontiguousarray(scale_b, dtype=np.float32)
    out = np.empty((M, N), dtype=np.uint32 if out_type == OUT_F32 else np.uint16)
    lib().oracle_dequant(M, N, _ptr(acc), N, None if sa is None else _ptr(sa),
                         None if sb is None else _ptr(sb), out_type, _ptr(out), N)
    return out


def f32_to_bf16(x) -> np.ndarray:
    L = lib()
    x = np.asarray(x, dtype=np.float32)
    return np.array([L.oracle_f32_to_bf16(float(v)) for v in x.reshape(-1)], dtype=np.uint16).reshape(x.shape)


def f32_to_f16(x) -> np.ndarray:
    L = lib()
    x = np.asarray(x, dtype=np.float32)
    return np.array([L.oracle_f32_to_f16(float(v)) for v in x.reshape(-1)], dtype=np.uint16).reshape(x.shape)


def wrap_s32(C: np.ndarray) -> np.ndarray:
    """Exact int64 sums wrapped to int32 two's complement (the INT32 overflow reading)."""
    return np.asarray(C, dtype=np.int64).astype(np.uint64).astype(np.uint32).view(np.int32)


def f16_tolerance_ok(C_gpu: np.ndarray, C_ref: np.ndarray, S: np.ndarray,
                     rel: float = 1e-3, abs_: float = 1e-6, frob: float = 1e-4):
    """FP16 acceptance: |C_gpu - C_ref| <= rel*S + abs_ everywhere and relative
    Frobenius error <= frob.  Returns (ok, max_ratio, frob_err)."""
    C_gpu = np.asarray(C_gpu, dtype=np.float64)
    err = np.abs(C_gpu - C_ref)
    bound = rel * S + abs_
    ratio = float(np.max(err / bound)) if err.size else 0.0
    nref = float(np.linalg.norm(C_ref))
    ferr = float(np.linalg.norm(C_gpu - C_ref)) / nref if nref > 0 else float(np.linalg.norm(C_gpu))
    ok = bool(np.all(err <= bound)) and ferr <= frob
    return ok, ratio, ferr
