"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test ties the oracle to a worked example printed on the pages, to a closed
form, to an invariant, or to brute force in exact arithmetic (Python ints,
fractions.Fraction), on inputs chosen so that a dropped term, a wrong sign or
index, a transposed operand or a swapped nibble order fails at least one test.
"""
import itertools
import os
from fractions import Fraction

import numpy as np
import pytest

import datagen
import oracle

F16 = np.float16


def f16bits(x):
    return np.asarray(x, dtype=np.float64).astype(F16).view(np.uint16)


# --------------------------------------------------------------------------
# binary16 decoder: exhaustive against numpy's independent conversion
# --------------------------------------------------------------------------
def test_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f64(bits)
    ref = bits.view(F16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0])
    # smallest subnormal, largest subnormal, smallest normal, max finite
    assert ours[0x0001] == 2.0 ** -24
    assert ours[0x03FF] == 1023 * 2.0 ** -24
    assert ours[0x0400] == 2.0 ** -14
    assert ours[0x7BFF] == 65504.0


# --------------------------------------------------------------------------
# worked example from the pages (m16n8k16 tile lab)
# --------------------------------------------------------------------------
def _read_golden(path):
    out = {"point": [], "reversed_row0": None}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            key, vals = line[0], [int(v) for v in line[1:]]
            if key == "shape":
                out["shape"] = tuple(vals)
            elif key == "point":
                out["point"].append(tuple(vals))
            else:
                out[key] = vals
    return out


def test_mma_lab_worked_example(golden_dir):
    g = _read_golden(os.path.join(golden_dir, "mma_lab_m16n8k16.txt"))
    M, N, K = g["shape"]
    B = np.array([[8 * r + c + 1 for c in range(N)] for r in range(K)], dtype=np.float64)
    A = np.eye(M, K)
    C, S = oracle.gemm_f16(f16bits(A), f16bits(B))
    for (r, c, v) in g["point"]:
        assert C[r, c] == v
    assert np.array_equal(C, B)
    Arev = np.eye(M, K)[::-1]
    C2, _ = oracle.gemm_f16(f16bits(Arev), f16bits(B))
    assert C2[0].tolist() == g["reversed_row0"]


# --------------------------------------------------------------------------
# identity and permutation operands, all three precisions, non-square shapes
# --------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,K", [(5, 7, 5), (16, 24, 16), (9, 3, 9)])
def test_identity_and_permutation_f16(M, N, K):
    rng = np.random.default_rng(M * 100 + N)
    B = rng.uniform(-2, 2, size=(K, N)).astype(F16).view(np.uint16)
    Bv = B.view(F16).astype(np.float64)
    perm = rng.permutation(K)
    P = np.zeros((M, K))
    P[np.arange(M), perm[:M]] = 1.0
    C, _ = oracle.gemm_f16(f16bits(P), B)
    assert np.array_equal(C, Bv[perm[:M]])
    # B = identity returns A
    A = rng.uniform(-2, 2, size=(M, K)).astype(F16).view(np.uint16)
    C2, _ = oracle.gemm_f16(A, f16bits(np.eye(K, K)))
    assert np.array_equal(C2[:, :K], A.view(F16).astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(5, 7, 6), (16, 24, 16), (9, 3, 10)])
def test_identity_and_permutation_s8_s4(M, N, K):
    rng = np.random.default_rng(M * 7 + N)
    perm = rng.permutation(K)
    P = np.zeros((M, K), dtype=np.int8)
    P[np.arange(M), perm[:M]] = 1
    Bt = rng.integers(-128, 128, size=(N, K)).astype(np.int8)   # column-major B
    C = oracle.gemm_s8(P, Bt)
    assert np.array_equal(C, Bt.T[perm[:M]].astype(np.int64))
    # identity B (column-major) returns A
    A = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    C2 = oracle.gemm_s8(A, np.eye(K, K, dtype=np.int8))
    assert np.array_equal(C2, A.astype(np.int64))
    # INT4, operands given as values, packed by the generator's packing
    Bt4 = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    C4 = oracle.gemm_s4(datagen.pack_s4_rows(P), datagen.pack_s4_rows(Bt4), K)
    assert np.array_equal(C4, Bt4.T[perm[:M]].astype(np.int64))
    A4 = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    C5 = oracle.gemm_s4(datagen.pack_s4_rows(A4), datagen.pack_s4_rows(np.eye(K, K, dtype=np.int8)), K)
    assert np.array_equal(C5, A4.astype(np.int64))


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
@pytest.mark.parametrize("K", [1, 17, 256, 1000])
def test_all_ones_and_extremes(K):
    M, N = 3, 5
    ones16 = f16bits(np.ones((M, K)))
    C, S = oracle.gemm_f16(ones16, f16bits(np.ones((K, N))))
    assert np.all(C == K) and np.all(S == K)
    C = oracle.gemm_f16(f16bits(-np.ones((M, K))), f16bits(np.ones((K, N))))[0]
    assert np.all(C == -K)
    # s8 extremes: (-128)(-128) K, 127 * (-128) K
    a = np.full((M, K), -128, np.int8)
    assert np.all(oracle.gemm_s8(a, np.full((N, K), -128, np.int8)) == 16384 * K)
    assert np.all(oracle.gemm_s8(np.full((M, K), 127, np.int8),
                                 np.full((N, K), -128, np.int8)) == -16256 * K)
    assert np.all(oracle.gemm_s8(np.ones((M, K), np.int8), np.ones((N, K), np.int8)) == K)
    # s4 extremes: (-8)(-8) K, 7 (-8) K
    if K % 2 == 0:
        p = lambda v, r: datagen.pack_s4_rows(np.full((r, K), v, np.int8))
        assert np.all(oracle.gemm_s4(p(-8, M), p(-8, N), K) == 64 * K)
        assert np.all(oracle.gemm_s4(p(7, M), p(-8, N), K) == -56 * K)
        assert np.all(oracle.gemm_s4(p(1, M), p(1, N), K) == K)


def test_rank_one():
    rng = np.random.default_rng(5)
    M, N, K = 11, 13, 40
    u = rng.integers(-128, 128, size=M)
    v = rng.integers(-128, 128, size=N)
    A = np.repeat(u[:, None], K, axis=1).astype(np.int8)
    Bt = np.repeat(v[:, None], K, axis=1).astype(np.int8)
    assert np.array_equal(oracle.gemm_s8(A, Bt), K * np.outer(u, v))
    u4, v4 = u % 16 - 8, v % 16 - 8
    A4 = datagen.pack_s4_rows(np.repeat(u4[:, None], K, axis=1).astype(np.int8))
    B4 = datagen.pack_s4_rows(np.repeat(v4[:, None], K, axis=1).astype(np.int8))
    assert np.array_equal(oracle.gemm_s4(A4, B4, K), K * np.outer(u4, v4))
    uf = rng.integers(-8, 9, size=M) / 4.0
    vf = rng.integers(-8, 9, size=N) / 8.0
    C, _ = oracle.gemm_f16(f16bits(np.repeat(uf[:, None], K, axis=1)),
                           f16bits(np.repeat(vf[None, :], K, axis=0)))
    assert np.array_equal(C, K * np.outer(uf, vf))


def test_cancellation_adversary_s8():
    """First half of K: A = B = 127; second half: A = 127, B = -127.  Exact C = 0
    although partial sums peak at (K/2)*16129; the pattern shifts per column."""
    K, M, N = 8192, 4, 6
    A = np.full((M, K), 127, np.int8)
    Bt = np.empty((N, K), np.int8)
    for j in range(N):
        s = 32 * j
        Bt[j] = 127
        Bt[j, (np.arange(K) + s) % K >= K // 2] = -127
    C = oracle.gemm_s8(A, Bt)
    assert np.all(C == 0)
    Bt[:, 0] = -127 if Bt[0, 0] == 127 else 127  # one flipped term must show
    C = oracle.gemm_s8(A, Bt)
    assert np.all(np.abs(C[:, 0]) == 2 * 127 * 127)


# --------------------------------------------------------------------------
# packing
# --------------------------------------------------------------------------
def test_s4_nibble_order_and_roundtrip():
    # low nibble = even k: byte 0x8F holds (-1, -8); 0x70 holds (0, 7)
    row = np.array([[0x8F, 0x70]], np.uint8)
    assert oracle.unpack_s4(row, 4).tolist() == [[-1, -8, 0, 7]]
    # all 256 byte values round-trip
    allb = np.arange(256, dtype=np.uint8).reshape(1, 256)
    vals = oracle.unpack_s4(allb, 512)
    assert vals.min() == -8 and vals.max() == 7
    assert np.array_equal(oracle.pack_s4(vals), allb)
    # all 16 nibble values map to [-8, 7] in two's complement
    nib = np.arange(16, dtype=np.uint8).reshape(1, 16)
    assert oracle.unpack_s4(nib, 32)[0, 0::2].tolist() == list(range(8)) + list(range(-8, 0))
    # the generator's packing and the oracle's packing agree
    v = np.random.default_rng(3).integers(-8, 8, size=(7, 30)).astype(np.int8)
    assert np.array_equal(datagen.pack_s4_rows(v), oracle.pack_s4(v))
    assert np.array_equal(oracle.unpack_s4(datagen.pack_s4_rows(v), 30), v)


# --------------------------------------------------------------------------
# brute force in exact arithmetic
# --------------------------------------------------------------------------
SHAPES = [s for s in itertools.product(range(4, 17), repeat=3)][::37]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_brute_force_int(M, N, K):
    rng = np.random.default_rng(M * 10000 + N * 100 + K)
    A = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    Bt = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    ref = [[sum(int(A[i, k]) * int(Bt[j, k]) for k in range(K)) for j in range(N)] for i in range(M)]
    assert oracle.gemm_s8(A, Bt).tolist() == ref
    K4 = K + (K & 1)
    A4 = rng.integers(-8, 8, size=(M, K4)).astype(np.int8)
    B4 = rng.integers(-8, 8, size=(N, K4)).astype(np.int8)
    ref4 = [[sum(int(A4[i, k]) * int(B4[j, k]) for k in range(K)) for j in range(N)] for i in range(M)]
    got = oracle.gemm_s4(datagen.pack_s4_rows(A4), datagen.pack_s4_rows(B4), K)
    assert got.tolist() == ref4


@pytest.mark.parametrize("M,N,K", SHAPES[::3])
def test_brute_force_f16_fraction(M, N, K):
    rng = np.random.default_rng(M * 31 + N * 7 + K)
    A = rng.normal(size=(M, K)).astype(F16)
    B = rng.normal(size=(K, N)).astype(F16)
    C, S = oracle.gemm_f16(A.view(np.uint16), B.view(np.uint16))
    Af = [[Fraction(float(x)) for x in row] for row in A.astype(np.float64)]
    Bf = [[Fraction(float(x)) for x in row] for row in B.astype(np.float64)]
    u = 2.0 ** -53
    for i in range(M):
        for j in range(N):
            exact = sum(Af[i][k] * Bf[k][j] for k in range(K))
            sabs = sum(abs(Af[i][k] * Bf[k][j]) for k in range(K))
            # recursive summation of exact products: |err| <= (K-1) u S (1 + O(u))
            assert abs(Fraction(C[i, j]) - exact) <= Fraction(K * u) * sabs
            assert abs(Fraction(S[i, j]) - sabs) <= Fraction(K * u) * sabs


def test_sampled_entry_points_match_full():
    A, B = datagen.f16_operands(64, "normal", m=40, k=72)
    C, S = oracle.gemm_f16(A, B)
    ii = np.array([0, 39, 17, 5]); jj = np.array([63, 0, 31, 5])
    c, s = oracle.gemm_f16_at(A, B, ii, jj)
    assert np.array_equal(c, C[ii, jj]) and np.array_equal(s, S[ii, jj])
    A8, B8 = datagen.s8_operands(48, m=33, k=80)
    C8 = oracle.gemm_s8(A8, B8)
    assert np.array_equal(oracle.gemm_s8_at(A8, B8, ii % 33, jj % 48), C8[ii % 33, jj % 48])
    A4, B4 = datagen.s4_operands(48, m=33, k=80)
    C4 = oracle.gemm_s4(A4, B4, 80)
    assert np.array_equal(oracle.gemm_s4_at(A4, B4, 80, ii % 33, jj % 48), C4[ii % 33, jj % 48])


def test_wrap_reading():
    assert oracle.wrap_s32(np.array([2 ** 31, -2 ** 31 - 1, 5])).tolist() == [-2 ** 31, 2 ** 31 - 1, 5]
