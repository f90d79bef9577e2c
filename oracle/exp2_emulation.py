"""Float32 model of the software exp2 (test infrastructure).

The method, from "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design
for Asymmetric Hardware Scaling" (fdeinterviews.com summary), bullet "Software
exponentials": compute 2^x on the ordinary FMA units by splitting x into an
integer and a fraction, evaluating a cubic polynomial on the fraction, and
adding the integer to the float's exponent bits.  The page states that after
rounding to BF16 the result agrees with the hardware exponential to within one
unit in the last place on 99% of inputs.

Readings where the page is silent:

* "integer and fraction" is n = floor(x), f = x - n in [0, 1), so the
  polynomial approximates 2^f on [1, 2);
* x is clamped below at -127 before the split (softmax arguments are <= 8, and
  anything below 2^-126 is negligible next to a row sum >= 1);
* the cubic's coefficients are this module's own fit: least squares of the
  relative error on [0, 1] with p(0) = 1 and p(1) = 2 imposed, so the result
  is continuous across integer x.  Nothing is taken from any math library.

The model evaluates Horner's rule with one rounding to float32 per step (what
a fused multiply-add does) and inserts the exponent with integer arithmetic on
the float32 bit pattern.
"""

import numpy as np


def fit_cubic_exp2(n_points=1 << 16):
    """Coefficients (c0, c1, c2, c3) of the cubic approximating 2^f on [0, 1].

    p(f) = 1 + f^3 + c1 (f - f^3) + c2 (f^2 - f^3) satisfies p(0) = 1 and
    p(1) = 2 for any c1, c2; those two are chosen to minimise the summed
    squared relative error over an even grid of [0, 1].
    """
    f = np.linspace(0.0, 1.0, n_points)
    target = np.exp2(f)
    basis = np.stack([f - f ** 3, f * f - f ** 3], axis=1) / target[:, None]
    rhs = (target - 1.0 - f ** 3) / target
    (c1, c2), *_ = np.linalg.lstsq(basis, rhs, rcond=None)
    c3 = 1.0 - c1 - c2
    return 1.0, float(c1), float(c2), float(c3)


def _fma_f32(a, b, c):
    """a*b + c rounded once to float32 (a, b, c float32)."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def emulated_exp2_f32(x, coeffs=None):
    """2^x by split + cubic + exponent insertion, float32 in and out."""
    c0, c1, c2, c3 = (np.float32(c) for c in (coeffs or fit_cubic_exp2()))
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-127.0))
    n = np.floor(x)
    f = (x - n).astype(np.float32)          # exact: x and n share the exponent range
    ones = np.ones_like(f)
    p = _fma_f32(np.full_like(f, c3), f, c2 * ones)
    p = _fma_f32(p, f, c1 * ones)
    p = _fma_f32(p, f, c0 * ones)
    bits = p.view(np.int32) + (n.astype(np.int32) << 23)
    return bits.view(np.float32)


def bf16_round_bits(x):
    """Round float32 values to BF16 (round to nearest, ties to even); uint16 bits."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)
