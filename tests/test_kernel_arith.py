"""Exhaustive CPU checks of two arithmetic steps the CUDA kernels take in
place of an IEEE division (no GPU needed; these restate the kernels' steps,
not the oracle).

1. Block scale s = RN(m / d) for the constants d = qmax in {1, 7, 31, 127}
   and d = 448 (E4M3): the kernels compute q0 = RN(m * c) with c = RN(1/d),
   the remainder rem = m - q0 * d with one FMA (exact, because q0 is within an
   ulp of m / d) and s = RN(q0 + rem * c) with a second FMA. This is the
   remainder-based correction of a quotient by a known divisor (P. Markstein,
   "Computation of elementary functions on the IBM RISC System/6000
   processor", IBM J. Res. Dev. 34(1), 1990; N. Brisebarre, J.-M. Muller and
   S. K. Raina, "Accelerating correctly rounded floating-point division when
   the divisor is known in advance", IEEE Trans. Computers 53(8), 2004). It
   is not correctly rounded for every divisor, so every significand is
   checked here for the divisors used: the steps commute with scaling m by a
   power of two while every intermediate stays normal, and the kernels take
   the IEEE division outside m in [2^-100, 2^126], so the binades checked
   cover every input the fast steps see.

2. Reciprocal r ~ 1/s: the kernels refine the hardware approximation y0 with
   one Newton-Raphson step (e = RN(1 - s*y0), r = RN(y0 + y0*e)). The fast
   quantize path needs |r - 1/s| well below 2^-23 / s (its margin is 2^-19 /
   |x/s| against half an ulp of the rounding grid). For every significand of
   s and every y0 within 2 ulps of 1/s (the approximation's documented bound
   is 1 ulp), the refined r is checked to be within 2^-24 (1 + 2^-18) of 1/s,
   relative.
"""
import numpy as np
import pytest

F32 = np.float32
F64 = np.float64


def _binade(e: int) -> np.ndarray:
    """Every float32 in [2^e, 2^(e+1))."""
    bits = (np.uint32(e + 127) << np.uint32(23)) | np.arange(1 << 23, dtype=np.uint32)
    return bits.view(F32)


def _rn32_of_sum(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """RN to float32 of the exact sum a + b (float64 inputs, exact values):
    float64 TwoSum gives the sum's rounding error; a float32 rounding of the
    float64 sum can only go wrong when that sum sits exactly on a float32
    midpoint and the error is nonzero, which is settled by the error's sign."""
    s = a + b
    bb = s - a
    err = (a - (s - bb)) + (b - bb)
    r = s.astype(F32)
    # midpoint test: s halfway between two float32 neighbours
    lo = np.where(r.astype(F64) <= s, r, np.nextafter(r, F32(-np.inf)))
    hi = np.nextafter(lo, F32(np.inf))
    mid = (lo.astype(F64) + hi.astype(F64)) / 2.0  # exact in float64
    on_mid = (s == mid) & (err != 0.0)
    r = np.where(on_mid & (err > 0), hi, np.where(on_mid & (err < 0), lo, r))
    return r


def kernel_scale(m: np.ndarray, d: float) -> np.ndarray:
    """The kernels' two-FMA quotient, with exact intermediate arithmetic."""
    c = F32(1.0) / F32(d)                       # RN(1/d)
    q0 = m * c                                  # RN(m * c) in float32
    rem64 = m.astype(F64) - q0.astype(F64) * F64(d)  # exact (Sterbenz; q0*d exact)
    rem = rem64.astype(F32)
    assert np.array_equal(rem.astype(F64), rem64), "remainder not representable"
    return _rn32_of_sum(q0.astype(F64), rem.astype(F64) * F64(c))  # rem*c exact in f64


@pytest.mark.parametrize("d", [1.0, 7.0, 31.0, 127.0, 448.0])
@pytest.mark.parametrize("e", [0, -100, 125])
def test_scale_division_exhaustive(d, e):
    m = _binade(e)
    want = m / F32(d)                           # IEEE division, RN
    got = kernel_scale(m, d)
    bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, f"d={d}: {bad.size} mismatches, first m={m[bad[0]]!r}"


def test_scale_division_planted_error_is_caught():
    """The check is sharp: dropping the correction FMA (s = q0) fails."""
    m = _binade(0)
    c = F32(1.0) / F32(7.0)
    assert np.any((m * c).view(np.uint32) != (m / F32(7.0)).view(np.uint32))


@pytest.mark.parametrize("e", [0, -126, 125])
def test_newton_reciprocal_error_bound(e):
    s = _binade(e)
    s64 = s.astype(F64)
    rn = F32(1.0) / s                           # RN(1/s)
    worst = 0.0
    for k in (-2, -1, 0, 1, 2):
        y0 = rn
        for _ in range(abs(k)):
            y0 = np.nextafter(y0, F32(np.inf) if k > 0 else F32(0.0))
        y64 = y0.astype(F64)
        e32 = (1.0 - s64 * y64).astype(F32)     # 1 - s*y0 exact in float64, one rounding
        # r = RN(y0 + y0*e): y0*e is exact in float64 (24 x 24 bits), the sum
        # is not (y0*e reaches 2^-70 below y0), so it is rounded once with TwoSum
        r = _rn32_of_sum(y64, y64 * e32.astype(F64))
        rel = np.abs(r.astype(F64) * s64 - 1.0)
        worst = max(worst, float(rel.max()))
    assert worst <= 2.0 ** -24 * (1 + 2.0 ** -18), worst
