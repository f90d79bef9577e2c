"""Pins for the float32 model of the software exponential (CPU only).

The page's claim: split + cubic + exponent insertion agrees with the hardware
exponential within one BF16 ulp on 99% of inputs.  The hardware unit is only
on the GPU; here the model is held to the stricter reference of the correctly
rounded 2^x, and its BF16 rounding is held to torch's conversion.
"""

import numpy as np
import torch

import oracle


def test_bf16_rounding_matches_torch(rng):
    x = np.concatenate([rng.standard_normal(1 << 16).astype(np.float32) * 100,
                        np.float32([1.00390625, 1.01171875, -3.0, 0.0, 65504.0])])
    # values exactly halfway between two BF16 numbers exercise ties-to-even
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_round_bits(x), ref)


def test_fit_hits_endpoints_and_error_bound():
    c0, c1, c2, c3 = oracle.fit_cubic_exp2()
    assert c0 == 1.0 and abs(c0 + c1 + c2 + c3 - 2.0) < 1e-15
    f = np.linspace(0, 1, 100001)
    rel = np.abs((c0 + f * (c1 + f * (c2 + f * c3))) / np.exp2(f) - 1)
    assert rel.max() < 2e-4           # a cubic cannot do much better on [0,1)
    assert rel.max() > 1e-6           # ...and this is a cubic, not exp2 itself


def test_integers_are_exact():
    n = np.arange(-126, 9, dtype=np.float32)
    np.testing.assert_array_equal(oracle.emulated_exp2_f32(n), np.exp2(n.astype(np.float64)).astype(np.float32))


def test_within_one_bf16_ulp_on_99_percent(rng):
    """Dense even sweep of [-126, 8] plus seeded uniform points."""
    x = np.concatenate([np.linspace(-126.0, 8.0, 1 << 22, dtype=np.float32),
                        rng.uniform(-126.0, 8.0, 1 << 20).astype(np.float32)])
    emu = oracle.bf16_round_bits(oracle.emulated_exp2_f32(x)).astype(np.int64)
    exact = oracle.bf16_round_bits(np.exp2(x.astype(np.float64)).astype(np.float32)).astype(np.int64)
    ulp = np.abs(emu - exact)        # BF16 bit patterns of positives are monotonic
    assert np.mean(ulp <= 1) >= 0.99
    assert ulp.max() <= 2


def test_masked_input_is_negligible():
    """-inf (a masked score) clamps to 2^-127 scale, far below any row sum."""
    y = oracle.emulated_exp2_f32(np.float32([-np.inf, -500.0]))
    assert np.all(y >= 0) and np.all(y < 1e-37)
