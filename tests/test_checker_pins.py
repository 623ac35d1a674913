"""Pins of the FP16 acceptance checkers (CPU).

Every FP16 parity decision goes through oracle.f16_tolerance_ok, directly
(tests.gpu_util.check_f16, check_f16_rows) or on sampled elements
(tests.gpu_util.check_f16_sampled).  The acceptance rule is the one stated for
the FP16 product: every element within |C - Cref| <= 1e-3 * sum_k |A_ik B_kj|
+ 1e-6, and relative Frobenius error <= 1e-4.  These tests feed the checkers
results that must pass and results planted just outside each bound that must
fail, so that a slip in the checker (an inverted comparison, a dropped
Frobenius term, |C| in place of sum |ab|, a dropped absolute term, NaN let
through) turns a test red.
"""
import numpy as np
import pytest

import datagen
import oracle
from tests.gpu_util import check_f16_sampled, sample_coords


@pytest.fixture(scope="module")
def case():
    M, N, K = 160, 256, 256
    A, B = datagen.f16_operands(N, "normal", seed=4242, m=M, k=K)
    Cref, S = oracle.gemm_f16(A, B)
    return A, B, Cref, S


def bound(S):
    return 1e-3 * S + 1e-6


def frob(C, Cref):
    return float(np.linalg.norm(C - Cref) / np.linalg.norm(Cref))


def test_exact_result_passes(case):
    _, _, Cref, S = case
    ok, ratio, ferr = oracle.f16_tolerance_ok(Cref.astype(np.float32), Cref, S)
    assert ok and ferr < 1e-6
    # an FP32 rounding of every element is far inside both bounds
    assert ratio < 1e-3


@pytest.mark.parametrize("factor,expect", [(1.01, False), (0.99, True)])
def test_one_element_at_the_element_bound(case, factor, expect):
    _, _, Cref, S = case
    i, j = 17, 33
    C = Cref.copy()
    C[i, j] += factor * bound(S)[i, j]
    assert frob(C, Cref) < 1e-4  # only the element bound decides
    ok, _, _ = oracle.f16_tolerance_ok(C, Cref, S)
    assert ok is expect
    C = Cref.copy()
    C[i, j] -= factor * bound(S)[i, j]
    assert oracle.f16_tolerance_ok(C, Cref, S)[0] is expect


@pytest.mark.parametrize("rel,expect", [(2e-4, False), (0.5e-4, True)])
def test_frobenius_bound_alone(case, rel, expect):
    """C = Cref * (1 + rel): every element is inside its own bound (|C| <= S),
    so the Frobenius term alone decides."""
    _, _, Cref, S = case
    C = Cref * (1.0 + rel)
    assert np.all(np.abs(C - Cref) <= bound(S))
    assert abs(frob(C, Cref) - rel) < 1e-9
    assert oracle.f16_tolerance_ok(C, Cref, S)[0] is expect


def test_bound_uses_sum_of_absolute_products_not_abs_c(case):
    """An element whose exact sum cancels (|C| far below sum |ab|) may err by
    up to 1e-3 * sum |ab|; a checker scaling by |C| would reject it."""
    _, _, Cref, S = case
    i, j = np.unravel_index(np.argmin(np.abs(Cref) / S), Cref.shape)
    assert abs(Cref[i, j]) < 0.05 * S[i, j]
    C = Cref.copy()
    C[i, j] += 0.5 * 1e-3 * S[i, j]
    assert abs(C[i, j] - Cref[i, j]) > 1e-3 * abs(Cref[i, j]) + 1e-6
    assert frob(C, Cref) < 1e-4
    assert oracle.f16_tolerance_ok(C, Cref, S)[0]


def test_absolute_term_where_the_products_vanish():
    """A zero row of A gives Cref = S = 0 there: only the 1e-6 term allows
    an error."""
    M, N, K = 8, 16, 64
    A, B = datagen.f16_operands(N, "uniform", seed=7, m=M, k=K)
    A = A.copy()
    A[3] = 0
    Cref, S = oracle.gemm_f16(A, B)
    assert np.all(S[3] == 0) and np.all(Cref[3] == 0)
    for err, expect in ((0.5e-6, True), (2e-6, False)):
        C = Cref.copy()
        C[3, 5] = err
        assert frob(C, Cref) < 1e-4
        assert oracle.f16_tolerance_ok(C, Cref, S)[0] is expect


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
def test_non_finite_result_fails(case, bad):
    _, _, Cref, S = case
    C = Cref.copy()
    C[5, 7] = bad
    assert not oracle.f16_tolerance_ok(C, Cref, S)[0]


# ------------------------------------------------ the sampled checker
def sampled_positions(M, N):
    ii, jj = sample_coords(M, N, 2000)
    return set(zip(ii.tolist(), jj.tolist()))


def test_sampled_checker_accepts_exact(case):
    A, B, Cref, _ = case
    check_f16_sampled(Cref.astype(np.float32), A, B)


@pytest.mark.parametrize("factor,expect", [(1.01, False), (0.99, True)])
def test_sampled_checker_element_bound(case, factor, expect):
    """One element at 1.01 / 0.99 of its bound.  The samples' Frobenius norm
    is that of ~n elements, so one outlier weighs more in it than in the full
    norm: enough samples (n = 20000) keep the passing case inside 1e-4."""
    A, B, Cref, S = case
    i, j = 0, Cref.shape[1] - 1  # a corner: always sampled
    assert (i, j) in sampled_positions(*Cref.shape)
    C = Cref.copy()
    C[i, j] += factor * bound(S)[i, j]
    ii, jj = sample_coords(*Cref.shape, 20000)
    d = C[ii, jj] - Cref[ii, jj]
    assert np.linalg.norm(d) / np.linalg.norm(Cref[ii, jj]) < 1e-4
    if expect:
        check_f16_sampled(C, A, B, n=20000)
    else:
        with pytest.raises(AssertionError):
            check_f16_sampled(C, A, B, n=20000)


@pytest.mark.parametrize("rel,expect", [(2e-4, False), (0.5e-4, True)])
def test_sampled_checker_frobenius(case, rel, expect):
    A, B, Cref, _ = case
    C = Cref * (1.0 + rel)
    if expect:
        check_f16_sampled(C, A, B)
    else:
        with pytest.raises(AssertionError):
            check_f16_sampled(C, A, B)


def test_sampled_checker_catches_nan(case):
    A, B, Cref, _ = case
    C = Cref.copy()
    C[Cref.shape[0] - 1, 0] = np.nan  # a corner: always sampled
    with pytest.raises(AssertionError):
        check_f16_sampled(C, A, B)


# ------------------------------------------------ planted checker mistakes
def scenarios(case):
    """(C, Cref, S, outcome the stated rule gives) for the cases above."""
    _, _, Cref, S = case
    out = [(Cref.astype(np.float32), Cref, S, True)]
    i, j = 17, 33
    for f, v in ((1.01, False), (0.99, True)):
        C = Cref.copy()
        C[i, j] += f * bound(S)[i, j]
        out.append((C, Cref, S, v))
    for rel, v in ((2e-4, False), (0.5e-4, True)):
        out.append((Cref * (1.0 + rel), Cref, S, v))
    a, b = np.unravel_index(np.argmin(np.abs(Cref) / S), Cref.shape)
    C = Cref.copy()
    C[a, b] += 0.5e-3 * S[a, b]
    out.append((C, Cref, S, True))
    C0, S0 = Cref.copy(), S.copy()
    C0[3] = 0.0
    S0[3] = 0.0
    for err, v in ((0.5e-6, True), (2e-6, False)):
        C = C0.copy()
        C[3, 5] = err
        out.append((C, C0, S0, v))
    C = Cref.copy()
    C[5, 7] = np.nan
    out.append((C, Cref, S, False))
    return out


def _mutant(kind):
    def check(C_gpu, C_ref, S, rel=1e-3, abs_=1e-6, frob=1e-4):
        C_gpu = np.asarray(C_gpu, dtype=np.float64)
        err = np.abs(C_gpu - C_ref)
        scale = np.abs(C_ref) if kind == "abs_c" else S
        b = rel * scale + (0.0 if kind == "no_abs" else abs_)
        nref = float(np.linalg.norm(C_ref))
        ferr = float(np.linalg.norm(C_gpu - C_ref)) / nref
        if kind == "inverted":
            elem = bool(np.all(err >= b))
        elif kind == "nan_through":
            elem = not bool(np.any(err > b))
        else:
            elem = bool(np.all(err <= b))
        ok = elem if kind == "no_frob" else (elem and ferr <= frob)
        if kind == "nan_through":
            ok = elem and not ferr > frob
        if kind == "frob_abs":
            ok = elem and float(np.linalg.norm(C_gpu - C_ref)) <= frob
        return ok, 0.0, ferr
    return check


@pytest.mark.parametrize("kind", ["abs_c", "no_abs", "inverted", "nan_through", "no_frob", "frob_abs"])
def test_pins_catch_planted_checker_mistakes(case, kind, monkeypatch):
    for C, Cref, S, v in scenarios(case):
        assert oracle.f16_tolerance_ok(C, Cref, S)[0] is v
    bad = _mutant(kind)
    assert any(bad(C, Cref, S)[0] is not v for C, Cref, S, v in scenarios(case)), kind
