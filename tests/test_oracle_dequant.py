"""Pins of the oracle's scaled integer epilogue (dequantisation): the 16-bit
roundings against independent conversions, and the whole per-element value
against exact rational arithmetic with round-to-nearest-even applied at every
step of the stated order."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _specials():
    v = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 2.0 ** -14, 2.0 ** -24,
         2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -26, 3.0 * 2.0 ** -25, 1e-40, 3.4e38, -3.4e38,
         1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 0.1, -0.7,
         float("inf"), float("-inf")]
    return np.array(v, dtype=np.float32)


def _randoms(n=20000, seed=1):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # plus values in the binary16 range, where rounding decisions are dense
    y = (rng.standard_normal(n) * np.exp2(rng.integers(-26, 17, size=n))).astype(np.float32)
    return np.concatenate([x, y])


def test_bf16_rounding_against_torch():
    x = np.concatenate([_specials(), _randoms()])
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_rounding_against_numpy():
    x = np.concatenate([_specials(), _randoms()])
    ours = oracle.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# ---- exact restatement: binary32 round-to-nearest-even of a rational
def _rne_binary32(q: Fraction) -> float:
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                      # below 2^-126 the spacing stays 2^-149
    quantum = Fraction(2) ** (e - 23)
    m = a / quantum
    n = m.numerator // m.denominator
    r = m - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * quantum
    if v >= Fraction(2) ** 128 - Fraction(2) ** 103:   # halfway to the next power: overflow
        return sign * float("inf")
    return sign * float(v)


def _expected_f32(acc, sa, sb):
    v = int(np.int64(acc).astype(np.uint64).astype(np.uint32).view(np.int32))
    t = _rne_binary32(Fraction(v))
    t = _rne_binary32(Fraction(t) * Fraction(float(sa)))
    return _rne_binary32(Fraction(t) * Fraction(float(sb)))


def test_dequant_matches_exact_stepwise_rounding():
    rng = np.random.default_rng(7)
    M, N = 24, 40
    acc = rng.integers(-2 ** 31, 2 ** 31, size=(M, N), dtype=np.int64)
    acc[0, :8] = [2 ** 24 + 1, 2 ** 24 + 3, -(2 ** 24 + 1), 2 ** 25 + 2, 16777217, 0, 1, -1]
    acc[1, 0] = 2 ** 33 + 5          # wraps to 5 in int32
    sa = (rng.standard_normal(M) * np.exp2(rng.integers(-20, 20, size=M))).astype(np.float32)
    sb = (rng.standard_normal(N) * np.exp2(rng.integers(-20, 20, size=N))).astype(np.float32)
    got = oracle.dequant(acc, sa, sb, oracle.OUT_F32).view(np.float32)
    for i in range(M):
        for j in range(N):
            exp = _expected_f32(acc[i, j], sa[i], sb[j])
            assert got[i, j] == np.float32(exp) or (np.isinf(exp) and got[i, j] == exp), (i, j)
    # int -> float rounding: 2^24 + 1 ties to even (2^24), 2^24 + 3 rounds up
    one = oracle.dequant(np.array([[2 ** 24 + 1, 2 ** 24 + 3]]), None, None).view(np.float32)
    assert one.tolist() == [[16777216.0, 16777220.0]]
    # 16-bit outputs are the binary32 value rounded once more
    bf = oracle.dequant(acc, sa, sb, oracle.OUT_BF16)
    hf = oracle.dequant(acc, sa, sb, oracle.OUT_F16)
    assert np.array_equal(bf, oracle.f32_to_bf16(got))
    assert np.array_equal(hf, oracle.f32_to_f16(got))


def test_dequant_order_matters_and_is_a_then_b():
    """Find scales for which (t * sa) * sb and t * (sa * sb) round differently
    and check the oracle follows the first."""
    rng = np.random.default_rng(11)
    for _ in range(20000):
        t = np.float32(rng.integers(1, 2 ** 24))
        sa, sb = rng.uniform(0.5, 2.0, size=2).astype(np.float32)
        ab = np.float32(t * sa) * sb
        alt = t * np.float32(sa * sb)
        if ab != alt:
            break
    else:
        pytest.skip("no order-sensitive triple found")
    got = oracle.dequant(np.array([[int(t)]]), np.array([sa]), np.array([sb])).view(np.float32)[0, 0]
    assert got == np.float32(_expected_f32(int(t), sa, sb))
    assert got == ab and got != alt


def test_dequant_identity_scales():
    acc = np.array([[3, -7, 2 ** 20, -(2 ** 23)]], dtype=np.int64)
    got = oracle.dequant(acc, None, None).view(np.float32)
    assert got.tolist() == [[3.0, -7.0, 2.0 ** 20, -(2.0 ** 23)]]
    got = oracle.dequant(acc, np.array([0.5], np.float32), np.array([2, 4, 0.25, 1], np.float32)).view(np.float32)
    assert got.tolist() == [[3.0, -14.0, 2.0 ** 17, -(2.0 ** 22)]]
