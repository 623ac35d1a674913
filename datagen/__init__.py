"""Seeded synthetic operands for the square GEMM workloads.

This module is the only code shared by the CUDA path's tests/bench and the CPU
oracle.  It draws random numbers and lays them out in the boundary's storage
formats; it holds none of the product's arithmetic (no multiply, no sum).

Generator
---------
Every operand is a counter-based stream: element ``i`` (in storage order) of
the stream with seed ``s`` is ``splitmix64_mix(s + (i + 1) * GAMMA)``, i.e. the
(i+1)-th output of Steele/Lea/Flood's SplitMix64 started at state ``s``
("Fast splittable pseudorandom number generators", OOPSLA 2014; the 64-bit
finaliser constants are the published ones).

Seeds (one per precision and size, separate sub-streams for A and B)::

    seed(prec, N) = 1_000_003 * N + {"f16": 0, "s8": 1, "s4": 2}[prec]
    A stream      = seed ^ 0xA,   B stream = seed ^ 0xB

Value maps
----------
* s8  uniform over [-128, 127]:  (u >> 56) - 128   (top byte, exactly uniform)
* s4  uniform over [-8, 7]:      (u >> 60) - 8     (top nibble, exactly uniform)
* f16 uniform in [-1, 1]:        x = 2 * (u >> 11) * 2**-53 - 1 in float64,
                                 then round-to-nearest-even to binary16
* f16 normal(0, 1) * scale:      Box-Muller on two consecutive draws of the
                                 element's own sub-stream (counters 2i, 2i+1),
                                 u1 = ((v1 >> 11) + 1) * 2**-53 in (0, 1],
                                 u2 = (v2 >> 11) * 2**-53,
                                 z = sqrt(-2 ln u1) * cos(2 pi u2), times scale,
                                 then RNE to binary16

Storage formats (the C boundary's layouts)
------------------------------------------
* f16 operands: uint16 bit patterns (numpy float16 viewed as uint16).
* A is row-major M x K.  FP16 B is row-major K x N.  INT8/INT4 B is
  column-major K x N, stored as N rows of K ("K-contiguous").
* packed s4: two signed nibbles per byte, element 2t of a row in bits 0-3 and
  element 2t+1 in bits 4-7 (low nibble = even k).
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

PREC_OFFSET = {"f16": 0, "s8": 1, "s4": 2}


def config_seed(prec: str, n: int) -> int:
    """Seed of one (precision, size) workload."""
    return 1_000_003 * int(n) + PREC_OFFSET[prec]


def operand_seed(seed: int, which: str) -> int:
    """Sub-stream seed of operand 'A' or 'B'."""
    return (int(seed) ^ {"A": 0xA, "B": 0xB}[which]) & 0xFFFFFFFFFFFFFFFF


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_stream(seed: int, count: int, start: int = 0,
                      chunk: int = 1 << 24) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the SplitMix64 stream ``seed``.

    Output ``i`` is ``mix(seed + (i + 1) * GAMMA)`` modulo 2**64.
    """
    out = np.empty(count, dtype=np.uint64)
    s = np.uint64(int(seed) & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for lo in range(0, count, chunk):
            hi = min(count, lo + chunk)
            ctr = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
            out[lo:hi] = _mix(s + ctr * GAMMA)
    return out


def uniform_s8(seed: int, rows: int, cols: int) -> np.ndarray:
    """int8 array (rows, cols), uniform over [-128, 127]."""
    u = splitmix64_stream(seed, rows * cols)
    v = (u >> np.uint64(56)).astype(np.int16) - 128
    return v.astype(np.int8).reshape(rows, cols)


def uniform_s4_values(seed: int, rows: int, cols: int) -> np.ndarray:
    """int8 array (rows, cols) of unpacked s4 values, uniform over [-8, 7]."""
    u = splitmix64_stream(seed, rows * cols)
    v = (u >> np.uint64(60)).astype(np.int16) - 8
    return v.astype(np.int8).reshape(rows, cols)


def pack_s4_rows(values: np.ndarray) -> np.ndarray:
    """Store s4 values (rows, cols) two per byte, low nibble = even column.

    ``cols`` must be even.  Returns uint8 (rows, cols // 2).
    """
    v = np.asarray(values)
    assert v.ndim == 2 and v.shape[1] % 2 == 0
    lo = v[:, 0::2].astype(np.int16) & 0xF
    hi = v[:, 1::2].astype(np.int16) & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def uniform_s4_packed(seed: int, rows: int, cols: int) -> np.ndarray:
    """Packed s4 operand (rows, cols // 2) uint8; values uniform over [-8, 7]."""
    return pack_s4_rows(uniform_s4_values(seed, rows, cols))


def _unit53(u: np.ndarray) -> np.ndarray:
    return (u >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform_f16(seed: int, rows: int, cols: int) -> np.ndarray:
    """uint16 bit patterns (rows, cols) of binary16 values uniform in [-1, 1]."""
    u = splitmix64_stream(seed, rows * cols)
    x = 2.0 * _unit53(u) - 1.0
    return x.astype(np.float16).view(np.uint16).reshape(rows, cols)


def normal_f16(seed: int, rows: int, cols: int, scale: float) -> np.ndarray:
    """uint16 bit patterns (rows, cols) of binary16 normal(0,1)*scale draws."""
    n = rows * cols
    u = splitmix64_stream(seed, 2 * n)
    u1 = ((u[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = _unit53(u[1::2])
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return (z * scale).astype(np.float16).view(np.uint16).reshape(rows, cols)


def f16_operands(n: int, dist: str, seed: int | None = None,
                 m: int | None = None, k: int | None = None):
    """(A, B) for an FP16 GEMM: A (M,K) row-major, B (K,N) row-major, uint16.

    dist: "uniform" (U[-1,1]) or "normal" (normal(0,1)/sqrt(K), both operands).
    """
    m = n if m is None else m
    k = n if k is None else k
    seed = config_seed("f16", n) if seed is None else seed
    sa, sb = operand_seed(seed, "A"), operand_seed(seed, "B")
    if dist == "uniform":
        return uniform_f16(sa, m, k), uniform_f16(sb, k, n)
    if dist == "normal":
        sc = 1.0 / np.sqrt(k) if k > 0 else 1.0
        return normal_f16(sa, m, k, sc), normal_f16(sb, k, n, sc)
    raise ValueError(dist)


def s8_operands(n: int, seed: int | None = None,
                m: int | None = None, k: int | None = None):
    """(A, Bt) for an INT8 GEMM: A (M,K) row-major, B column-major as Bt (N,K)."""
    m = n if m is None else m
    k = n if k is None else k
    seed = config_seed("s8", n) if seed is None else seed
    return (uniform_s8(operand_seed(seed, "A"), m, k),
            uniform_s8(operand_seed(seed, "B"), n, k))


def s4_operands(n: int, seed: int | None = None,
                m: int | None = None, k: int | None = None):
    """(A, Bt) packed s4: A (M, K/2) bytes row-major, Bt (N, K/2) bytes."""
    m = n if m is None else m
    k = n if k is None else k
    assert k % 2 == 0
    seed = config_seed("s4", n) if seed is None else seed
    return (uniform_s4_packed(operand_seed(seed, "A"), m, k),
            uniform_s4_packed(operand_seed(seed, "B"), n, k))
