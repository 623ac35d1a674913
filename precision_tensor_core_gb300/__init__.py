"""Python binding of libptc, the GB300 (sm_103a) tensor-core GEMM library.

Dense matrix products C = A.B in the three precisions of "Hand-Written PTX
Tensor-Core GEMM Kernels: A Multi-Precision Study on NVIDIA L4"
(Borowski & Osinski): FP16 -> FP32, INT8 -> INT32 and packed INT4 -> INT32.

Two layers, both argument marshalling only (every arithmetic step runs in the
library's CUDA kernels):

* ``gemm_f16``, ``gemm_f16_f16acc``, ``gemm_s8``, ``gemm_s4``, ``gemm_s8_scaled``, ``gemm_s4_scaled``,
  ``gemm_s8_noalloc``, ``gemm_s8_b_rowmajor``, ``gemm_status_string``,
  ``gemm_poll_device_error``, ``ptc_kernel_launch_count``, ``ptc_last_launch``, ``ptc_last_conversion``, ``ptc_plan_shape``,
  ``ptc_debug_set_wait_limit``, ``ptc_set_tuning``: the C ABI of
  ``include/ptc.h`` under the same names, taking integers (sizes, leading
  dimensions, device addresses, a cudaStream_t handle).  A nonzero status
  raises :class:`PtcError`.
* ``matmul_f16``, ``matmul_f16_f16acc``, ``matmul_s8``, ``matmul_s4``, ``matmul_s8_scaled``,
  ``matmul_s4_scaled``: the same calls on torch tensors.  Device tensors run
  on the current CUDA stream; host (CPU) tensors of ``matmul_f16`` /
  ``matmul_s8`` / ``matmul_s4`` go through the host-buffer entry points
  (``gemm_*_host``), which pipeline the copies inside the library.

There is no CPU fallback: if ``libptc.so`` has not been built the first call
raises, and on a machine without a compute-capability 10.3 GPU every GEMM call
raises ``PtcError`` with status ``PTC_ERR_DEVICE``.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libptc.so")

PTC_OK = 0
PTC_ERR_INVALID = 1
PTC_ERR_ALIGN = 2
PTC_ERR_OVERLAP = 3
PTC_ERR_DEVICE = 4
PTC_ERR_LAUNCH = 5
PTC_ERR_TIMEOUT = 6
PTC_ERR_ALLOC = 7

PTC_BASELINE_F16_WMMA = 0
PTC_BASELINE_F16_MMA = 1
PTC_BASELINE_S8_WMMA = 2
PTC_BASELINE_S8_MMA = 3
PTC_BASELINE_S4_WMMA = 4
PTC_BASELINE_S4_MMA = 5
PTC_BASELINE_F16_LDMATRIX = 6
PTC_BASELINE_S8_LDMATRIX = 7
PTC_BASELINE_S4_LDMATRIX = 8

PTC_OUT_F32 = 0
PTC_OUT_BF16 = 1
PTC_OUT_F16 = 2

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_lib = None


class PtcError(RuntimeError):
    """A libptc call returned a nonzero status."""

    def __init__(self, status: int, message: str):
        super().__init__(f"[{status}] {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libptc.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libptc.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name in ("gemm_f16", "gemm_f16_f16acc", "gemm_s8", "gemm_s4", "gemm_s8_noalloc",
                     "gemm_s8_b_rowmajor", "gemm_f16_host", "gemm_s8_host", "gemm_s4_host"):
            fn = getattr(L, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]
        for name in ("gemm_s8_scaled", "gemm_s4_scaled"):
            fn = getattr(L, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i64, ctypes.c_int, _vp]
        L.gemm_baseline.restype = ctypes.c_int
        L.gemm_baseline.argtypes = [ctypes.c_int, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]
        L.gemm_status_string.restype = ctypes.c_char_p
        L.gemm_status_string.argtypes = [ctypes.c_int]
        L.gemm_poll_device_error.restype = ctypes.c_int
        L.gemm_poll_device_error.argtypes = []
        L.ptc_kernel_launch_count.restype = ctypes.c_uint64
        L.ptc_kernel_launch_count.argtypes = []
        L.ptc_debug_set_wait_limit.restype = ctypes.c_int
        L.ptc_debug_set_wait_limit.argtypes = [ctypes.c_uint64, _i64]
        L.ptc_set_tuning.restype = ctypes.c_int
        L.ptc_set_tuning.argtypes = [ctypes.c_char_p, _i64]
        _ip = ctypes.POINTER(ctypes.c_int)
        L.ptc_last_launch.restype = ctypes.c_int
        L.ptc_last_launch.argtypes = [_ip, _ip, _ip, _ip]
        L.ptc_last_conversion.restype = ctypes.c_int
        L.ptc_last_conversion.argtypes = [_ip]
        _u64p = ctypes.POINTER(ctypes.c_uint64)
        L.ptc_clock_probe_read.restype = ctypes.c_int
        L.ptc_clock_probe_read.argtypes = [_u64p, _u64p, _u64p]
        L.ptc_plan_shape.restype = ctypes.c_int
        L.ptc_plan_shape.argtypes = [_i64, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, _ip, _ip, _ip, _ip]
        _lib = L
    return _lib


def _check(status: int) -> int:
    if status != PTC_OK:
        raise PtcError(status, gemm_status_string(status))
    return status


def gemm_status_string(status: int) -> str:
    return lib().gemm_status_string(int(status)).decode()


# ---------------------------------------------------------------- C ABI layer
def gemm_f16(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """C[MxN] f32 = A[MxK] f16 (row-major) . B[KxN] f16 (row-major); device addresses."""
    return _check(lib().gemm_f16(M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_f16_f16acc(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """C[MxN] f16 = A[MxK] f16 . B[KxN] f16 with FP16 accumulators; device addresses."""
    return _check(lib().gemm_f16_f16acc(M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_s8(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """C[MxN] s32 = A[MxK] s8 (row-major) . B[KxN] s8 (column-major); device addresses."""
    return _check(lib().gemm_s8(M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_s8_b_rowmajor(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """C[MxN] s32 = A[MxK] s8 (row-major) . B[KxN] s8 (row-major, ldb >= N); device addresses."""
    return _check(lib().gemm_s8_b_rowmajor(M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_s4(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """C[MxN] s32 = A[MxK] packed s4 . B[KxN] packed s4 (column-major); lda/ldb in nibbles."""
    return _check(lib().gemm_s4(M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_s8_scaled(M, N, K, A, lda, B, ldb, scale_a, scale_b, C, ldc, out_type, stream=0) -> int:
    """C = out(rn(rn(float(sum_k A_ik B_kj) * scale_a[i]) * scale_b[j])), INT8 operands."""
    return _check(lib().gemm_s8_scaled(M, N, K, A, lda, B, ldb, scale_a, scale_b, C, ldc, out_type, stream))


def gemm_s4_scaled(M, N, K, A, lda, B, ldb, scale_a, scale_b, C, ldc, out_type, stream=0) -> int:
    """As gemm_s8_scaled with packed INT4 operands (lda, ldb in nibbles)."""
    return _check(lib().gemm_s4_scaled(M, N, K, A, lda, B, ldb, scale_a, scale_b, C, ldc, out_type, stream))


def gemm_s8_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """gemm_s8 that allocates nothing: its workspace is a fixed 32 MiB device
    array shared by all calls, for callers that cannot allow a library to
    allocate device memory.  Overlapping calls race; see include/ptc.h."""
    return _check(lib().gemm_s8_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_f16_host(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """gemm_f16 with host-resident A, B, C (asynchronous on `stream`; see include/ptc.h)."""
    return _check(lib().gemm_f16_host(M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_s8_host(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """gemm_s8 with host-resident A, B, C (asynchronous on `stream`)."""
    return _check(lib().gemm_s8_host(M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_s4_host(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """gemm_s4 with host-resident A, B, C (asynchronous on `stream`)."""
    return _check(lib().gemm_s4_host(M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_baseline(variant, M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """The paper's WMMA / mma.sync kernel families on GB300 (PTC_BASELINE_*); see include/ptc.h."""
    return _check(lib().gemm_baseline(variant, M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_poll_device_error() -> int:
    """Status of the device error word (read and cleared); synchronises the device."""
    return int(lib().gemm_poll_device_error())


def ptc_kernel_launch_count() -> int:
    return int(lib().ptc_kernel_launch_count())


def ptc_clock_probe_read():
    """Clock record of the GEMM kernels launched with the "clock_probe" knob
    set, per family (FP16, INT8 route, INT4 route): lists of SM cycles,
    nanoseconds and CTAs summed over CTAs.  Read and cleared; synchronous."""
    cyc, ns, ctas = (ctypes.c_uint64 * 3)(), (ctypes.c_uint64 * 3)(), (ctypes.c_uint64 * 3)()
    _check(lib().ptc_clock_probe_read(cyc, ns, ctas))
    return list(cyc), list(ns), list(ctas)


def ptc_debug_set_wait_limit(timeout_ns: int, stall_tile: int = -1) -> int:
    return _check(lib().ptc_debug_set_wait_limit(int(timeout_ns), int(stall_tile)))


def ptc_set_tuning(key: str, value: int) -> int:
    return _check(lib().ptc_set_tuning(key.encode(), int(value)))


def ptc_plan_shape(M: int, N: int, K: int, prec: int, sms: int = 152,
                   caps: tuple[int, int, int] = (76, 36, 15), with_ring: bool = False):
    """(CTAs per tile, tile width, CTAs per tile's K range) the library would
    launch for an M x N x K product of precision `prec` (0 FP16, 1 INT8,
    2 INT4) on a device of `sms` SMs with cluster capacities `caps` (clusters
    of 2, 4, 8 one-CTA tiles that fit at once), under the current knobs; with
    `with_ring`, a fourth item: whether the integer operands are converted
    inside the GEMM kernel.  Host arithmetic only; the defaults are a GB300's
    figures."""
    c, n, k, r = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().ptc_plan_shape(int(M), int(N), int(K), int(prec), int(sms), int(caps[0]), int(caps[1]),
                                int(caps[2]), ctypes.byref(c), ctypes.byref(n), ctypes.byref(k), ctypes.byref(r)))
    if with_ring:
        return c.value, n.value, k.value, bool(r.value)
    return c.value, n.value, k.value


def ptc_last_launch() -> tuple[int, int, int, int]:
    """(grid CTAs, CTAs per cluster, CTAs sharing a tile's K range, tile
    width) of the calling thread's last GEMM kernel launch."""
    g, c, k, n = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().ptc_last_launch(ctypes.byref(g), ctypes.byref(c), ctypes.byref(k), ctypes.byref(n)))
    return g.value, c.value, k.value, n.value


def ptc_last_conversion() -> int:
    """Operand conversion of the calling thread's last GEMM call: 0 none, 1 a
    separate pass into a workspace, 2 inside the GEMM kernel."""
    m = ctypes.c_int(0)
    _check(lib().ptc_last_conversion(ctypes.byref(m)))
    return m.value


# ---------------------------------------------------------------- torch layer
def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _rowmajor(t, name):
    """Row pitch in elements of a 2-D tensor with unit column stride.  A single
    row has no pitch; the smallest one that meets every alignment rule is used."""
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be a 2-D tensor with unit column stride")
    if t.shape[0] > 1:
        return t.stride(0)
    return max(32, (t.shape[1] + 31) // 32 * 32)


_HOST_FN = {}


def _run(fn, A, B, out, out_shape, out_dtype, M, N, K, lda_scale, stream, sync=True):
    """Device tensors: the device entry point on `stream`.  Host tensors: the
    host entry point (pipelined copies inside the library); the result is
    ready on return unless sync=False, in which case `stream` must be
    synchronised before `out` is read and A, B must be kept alive (and
    unchanged) until then."""
    import torch
    host = A.device.type == "cpu"
    if host != (B.device.type == "cpu"):
        raise ValueError("A and B must both be on the host or both on the device")
    if host:
        hfn = _HOST_FN.get(fn)
        if hfn is None:
            raise ValueError("this product has no host-buffer entry point")
        C = out if out is not None else torch.empty(out_shape, dtype=out_dtype, pin_memory=True)
        if C.device.type != "cpu":
            raise ValueError("host operands need a host result tensor")
        st = _stream(stream)
        hfn(M, N, K, A.data_ptr(), _rowmajor(A, "A") * lda_scale, B.data_ptr(), _rowmajor(B, "B") * lda_scale,
            C.data_ptr(), _rowmajor(C, "C"), st)
        if sync:
            torch.cuda.ExternalStream(st).synchronize() if st else torch.cuda.synchronize()
        return C
    C = out if out is not None else torch.empty(out_shape, dtype=out_dtype, device=A.device)
    fn(M, N, K, A.data_ptr(), _rowmajor(A, "A") * lda_scale, B.data_ptr(), _rowmajor(B, "B") * lda_scale,
       C.data_ptr(), _rowmajor(C, "C"), _stream(stream))
    return C


def matmul_f16(A, B, out=None, stream=None, sync=True):
    """FP16 A (M,K) @ B (K,N) -> float32 (M,N) on the tensor cores (device or host tensors)."""
    import torch
    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("matmul_f16 takes float16 operands")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    return _run(gemm_f16, A, B, out, (M, N), torch.float32, M, N, K, 1, stream, sync)


def matmul_f16_f16acc(A, B, out=None, stream=None):
    """FP16 A (M,K) @ B (K,N) -> float16 (M,N), accumulated in FP16 on the tensor cores."""
    import torch
    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("matmul_f16_f16acc takes float16 operands")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    return _run(gemm_f16_f16acc, A, B, out, (M, N), torch.float16, M, N, K, 1, stream)


def matmul_s8(A, Bt, out=None, stream=None, sync=True):
    """INT8 A (M,K) @ B where B (K,N) is column-major, given as Bt (N,K) -> int32 (M,N)."""
    import torch
    if A.dtype != torch.int8 or Bt.dtype != torch.int8:
        raise TypeError("matmul_s8 takes int8 operands")
    M, K = A.shape
    N, K2 = Bt.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    return _run(gemm_s8, A, Bt, out, (M, N), torch.int32, M, N, K, 1, stream, sync)


def matmul_s4(A, Bt, K, out=None, stream=None, sync=True):
    """Packed INT4 A (M, >=K/2 bytes) @ B, B column-major given as Bt (N, >=K/2 bytes),
    two values per byte with the low nibble first -> int32 (M,N)."""
    import torch
    if A.dtype != torch.uint8 or Bt.dtype != torch.uint8:
        raise TypeError("matmul_s4 takes packed uint8 operands")
    M, N = A.shape[0], Bt.shape[0]
    return _run(gemm_s4, A, Bt, out, (M, N), torch.int32, M, N, int(K), 2, stream, sync)


def _out_type(dtype):
    import torch
    table = {torch.float32: PTC_OUT_F32, torch.bfloat16: PTC_OUT_BF16, torch.float16: PTC_OUT_F16}
    if dtype not in table:
        raise TypeError("scaled outputs are float32, bfloat16 or float16")
    return table[dtype]


def _scaled(fn, A, Bt, K, scale_a, scale_b, out_dtype, out, stream, lda_scale):
    import torch
    M, N = A.shape[0], Bt.shape[0]
    if A.device.type == "cpu" or Bt.device.type == "cpu":
        raise ValueError("scaled products take device tensors")
    C = out if out is not None else torch.empty((M, N), dtype=out_dtype, device=A.device)
    for v, n, name in ((scale_a, M, "scale_a"), (scale_b, N, "scale_b")):
        if v is not None and (v.dtype != torch.float32 or v.numel() != n or not v.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 vector of {n} elements")
    fn(M, N, K, A.data_ptr(), _rowmajor(A, "A") * lda_scale, Bt.data_ptr(), _rowmajor(Bt, "B") * lda_scale,
       None if scale_a is None else scale_a.data_ptr(), None if scale_b is None else scale_b.data_ptr(),
       C.data_ptr(), _rowmajor(C, "C"), _out_type(C.dtype), _stream(stream))
    return C


def matmul_s8_scaled(A, Bt, scale_a=None, scale_b=None, out_dtype=None, out=None, stream=None):
    """(A (M,K) int8 @ B, B column-major as Bt (N,K) int8) * scale_a[:,None] * scale_b[None,:]
    -> float32 / bfloat16 / float16 (M,N), with the rounding order of gemm_s8_scaled."""
    import torch
    if A.dtype != torch.int8 or Bt.dtype != torch.int8:
        raise TypeError("matmul_s8_scaled takes int8 operands")
    if A.shape[1] != Bt.shape[1]:
        raise ValueError("inner dimensions differ")
    dt = out.dtype if out is not None else (out_dtype or torch.float32)
    return _scaled(gemm_s8_scaled, A, Bt, A.shape[1], scale_a, scale_b, dt, out, stream, 1)


def matmul_s4_scaled(A, Bt, K, scale_a=None, scale_b=None, out_dtype=None, out=None, stream=None):
    """As matmul_s8_scaled with packed INT4 operands (two per byte, low nibble first)."""
    import torch
    if A.dtype != torch.uint8 or Bt.dtype != torch.uint8:
        raise TypeError("matmul_s4_scaled takes packed uint8 operands")
    dt = out.dtype if out is not None else (out_dtype or torch.float32)
    return _scaled(gemm_s4_scaled, A, Bt, int(K), scale_a, scale_b, dt, out, stream, 2)


_HOST_FN.update({gemm_f16: gemm_f16_host, gemm_s8: gemm_s8_host, gemm_s4: gemm_s4_host})
