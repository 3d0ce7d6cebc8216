"""The backward's relative-accuracy form of 1 − 2^t, checked on the CPU.

The backward's dp has a purely relative tolerance, so 1 − 2^t (t <= 0, from the MUFU exp2 with an
absolute error of about 2^-22.5 near t = 0) must stay relatively accurate for tiny |t|. The kernel
takes the larger of two lower bounds of the exact value: the series x − x²/2 (x = −t·ln 2), which
undershoots by less than x³/6, and the difference (1 − 2^-21) − e. This test evaluates those fp32
operations in numpy (a fused multiply-add as one rounding of the exact expression), with e = 2^t
perturbed by the worst-case error of exp2 in either direction, and checks the stated bound: both
candidates stay at or below the exact value, and the larger is within 5e-5 of it, relatively, at
every t. The GPU parity tests check the kernel itself (rows of inputs down to ~1e-30)."""
import numpy as np

LN2 = np.float32(0.6931471805599453)
LN2SQ2 = np.float32(0.2402265069591007)
ONE_LOW = np.float32(1.0) - np.float32(2.0 ** -21)
EX2_ERR = 2.0 ** -22          # above the ~2^-22.5 absolute error of ex2.approx near 0


def _fma32(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def _one_minus_exp2(t32, e32):
    series = (t32 * _fma32(t32, np.full_like(t32, -LN2SQ2), np.full_like(t32, -LN2))).astype(np.float32)
    diff = (ONE_LOW - e32).astype(np.float32)
    return series, diff, np.maximum(series, diff)


def test_two_lower_bounds_relative_error():
    t = -np.concatenate([np.logspace(-12, np.log10(40.0), 400000), np.linspace(1e-4, 0.2, 200000)])
    t32 = t.astype(np.float32)
    exact = -np.expm1(t32.astype(np.float64) * np.log(2.0))          # 1 - 2^t at the fp32 argument
    for sign in (-1.0, 0.0, 1.0):
        e32 = (np.exp2(t32.astype(np.float64)) + sign * EX2_ERR).astype(np.float32)
        series, diff, got = _one_minus_exp2(t32, e32)
        # fp32 rounding of the final products can lift a lower bound by a few ulp of the result
        slack = exact * 2.0 ** -21
        assert np.all(series.astype(np.float64) <= exact + slack)
        assert np.all(diff.astype(np.float64) <= exact + slack)
        rel = np.abs(got.astype(np.float64) - exact) / exact
        assert rel.max() < 5e-5, (sign, float(rel.max()), float(t[np.argmax(rel)]))


def test_difference_alone_fails_for_tiny_arguments():
    """Why the series is needed: the plain difference 1 − e loses relative accuracy near t = 0."""
    t32 = (-np.logspace(-8, -5, 1000)).astype(np.float32)
    exact = -np.expm1(t32.astype(np.float64) * np.log(2.0))
    e32 = (np.exp2(t32.astype(np.float64)) + EX2_ERR).astype(np.float32)
    rel = np.abs((np.float32(1.0) - e32).astype(np.float64) - exact) / exact
    assert rel.max() > 1e-2
