"""Pins for the tiled online-softmax routine: lazy rescaling is exact.

The tiled routine (blocks of keys, running max and sum, eager or lazy
rescale, final fix-up) must reproduce the plain definition to fp64 rounding
for any block size, mask and logit range, while the lazy variant rescales
less often than the eager one.
"""

import numpy as np
import pytest

import oracle


def _case(rng, Sq, Sk, D, logit):
    q = logit * rng.standard_normal((Sq, D)) / np.sqrt(D) ** 0.5
    return q, rng.standard_normal((Sk, D)), rng.standard_normal((Sk, D))


@pytest.mark.parametrize("lazy", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block_n", [1, 16, 128])
@pytest.mark.parametrize("Sq,Sk", [(64, 64), (37, 300), (300, 37)])
def test_tiled_equals_plain(rng, lazy, causal, block_n, Sq, Sk):
    q, k, v = _case(rng, Sq, Sk, 16, 1.0)
    o, lse, _ = oracle.tiled_forward(q, k, v, causal, 0.25, block_n=block_n, lazy=lazy)
    o_ref, lse_ref = oracle.head_forward(q, k, v, causal, 0.25)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    fin = np.isfinite(lse_ref)
    np.testing.assert_array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_lazy_equals_eager_under_large_logits(rng, causal):
    """Logit std ~16 (Q scaled by 4 at D=128): maxima keep growing across
    blocks; lazy must agree with eager to fp64 rounding yet rescale less."""
    S, D = 512, 128
    q = 4.0 * rng.standard_normal((S, D))
    k, v = rng.standard_normal((S, D)), rng.standard_normal((S, D))
    scale = D ** -0.5
    o_e, l_e, n_e = oracle.tiled_forward(q, k, v, causal, scale, block_n=128, lazy=False)
    o_l, l_l, n_l = oracle.tiled_forward(q, k, v, causal, scale, block_n=128, lazy=True)
    o_ref, l_ref = oracle.head_forward(q, k, v, causal, scale)
    np.testing.assert_allclose(o_l, o_e, atol=1e-12)
    np.testing.assert_allclose(l_l, l_e, atol=1e-11)
    np.testing.assert_allclose(o_l, o_ref, atol=1e-12)
    assert n_e > 0 and 0 < n_l < n_e


def test_zero_threshold_rescales_like_eager(rng):
    q, k, v = _case(rng, 96, 96, 8, 3.0)
    _, _, n_e = oracle.tiled_forward(q, k, v, True, 1.0, block_n=8, lazy=False)
    _, _, n_0 = oracle.tiled_forward(q, k, v, True, 1.0, block_n=8, lazy=True, threshold=0.0)
    _, _, n_8 = oracle.tiled_forward(q, k, v, True, 1.0, block_n=8, lazy=True, threshold=8.0)
    assert n_0 == n_e and n_8 < n_e


def test_huge_threshold_never_rescales_and_overflows(rng):
    """With the threshold removed, stale maxima let exp2 overflow: the
    threshold of 8 is what keeps every weight <= 256 (final normalisation
    cannot repair an overflow)."""
    S = 64
    q = np.zeros((S, 1))
    q[:, 0] = 1.0
    k = np.zeros((S, 1))
    k[:, 0] = np.linspace(0, 2000, S)          # scores grow by ~32 per key
    v = np.ones((S, 1))
    with np.errstate(over="ignore", invalid="ignore"):
        o_bad, _, n_bad = oracle.tiled_forward(q, k, v, False, 1.0, block_n=1, lazy=True,
                                               threshold=1e9)
    o_ok, _, n_ok = oracle.tiled_forward(q, k, v, False, 1.0, block_n=1, lazy=True)
    assert n_bad == 0 and not np.all(np.isfinite(o_bad))
    np.testing.assert_allclose(o_ok, 1.0, atol=1e-12)
