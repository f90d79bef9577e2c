"""Pins for the fp64 oracle's analytic gradients (CPU only).

The gradients are those of L = sum(dO * O).  They are checked against central
finite differences of the oracle's own forward (itself pinned in
test_oracle_forward.py), against closed forms, and against identities that the
softmax Jacobian implies.
"""

import numpy as np
import pytest

import oracle


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _loss(q, k, v, do, causal, scale, cu=None):
    o, _ = oracle.attention_forward(q, k, v, causal, scale, cu_seqlens=cu)
    return float(np.sum(o * do))


def _fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + h
        fp = f()
        x[idx] = old - h
        fm = f()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Sk,Hq,Hkv", [(5, 5, 2, 1), (4, 6, 2, 2), (6, 4, 3, 1)])
def test_gradients_match_finite_differences(rng, causal, Sq, Sk, Hq, Hkv):
    B, D = 2, 3
    q, k, v = _rand(rng, B, Sq, Hq, D), _rand(rng, B, Sk, Hkv, D), _rand(rng, B, Sk, Hkv, D)
    do = _rand(rng, B, Sq, Hq, D)
    scale = 0.7
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal, scale)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        fd = _fd_grad(lambda: _loss(q, k, v, do, causal, scale), x)
        err = np.linalg.norm(fd - g) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-6, err


def test_packed_gradients_match_finite_differences(rng):
    lens = [3, 5]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, Hq, Hkv, D = int(cu[-1]), 2, 1, 2
    q, k, v, do = _rand(rng, T, Hq, D), _rand(rng, T, Hkv, D), _rand(rng, T, Hkv, D), _rand(rng, T, Hq, D)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, True, 0.9, cu_seqlens=cu)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        fd = _fd_grad(lambda: _loss(q, k, v, do, True, 0.9, cu), x)
        assert np.linalg.norm(fd - g) / np.linalg.norm(fd) < 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_averaged_dv(rng, causal):
    """Q = 0: weights are uniform over the visible keys, so
    dV_j = sum over rows i that see j of dO_i / |visible(i)|."""
    S, D = 7, 3
    q = np.zeros((S, D))
    k, v, do = _rand(rng, S, D), _rand(rng, S, D), _rand(rng, S, D)
    _, _, dv = oracle.head_backward(q, k, v, do, causal, 0.5)
    ref = np.zeros((S, D))
    for i in range(S):
        n = i + 1 if causal else S
        ref[:n] += do[i] / n
    np.testing.assert_allclose(dv, ref, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_jacobian_identities(rng, causal):
    """Each row of dS sums to zero, hence dQ is unchanged by a common shift of
    all keys and the dK rows sum to zero."""
    S, D = 9, 4
    q, k, v, do = (_rand(rng, S, D) for _ in range(4))
    u = _rand(rng, D)
    dq1, dk1, _ = oracle.head_backward(q, k, v, do, causal, 0.6)
    dq2, _, _ = oracle.head_backward(q, k + u, v, do, causal, 0.6)
    np.testing.assert_allclose(dq1, dq2, atol=1e-12)
    np.testing.assert_allclose(dk1.sum(axis=0), 0.0, atol=1e-12)


def test_grouped_kv_gradients_sum_over_the_group(rng):
    """dK, dV of a shared kv head equal the sums of the per-head gradients of
    multi-head attention on repeated K/V."""
    B, S, D = 1, 6, 3
    q, do = _rand(rng, B, S, 4, D), _rand(rng, B, S, 4, D)
    k, v = _rand(rng, B, S, 2, D), _rand(rng, B, S, 2, D)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, True, 0.5)
    dq_r, dk_r, dv_r = oracle.attention_backward(q, np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2),
                                                 do, True, 0.5)
    np.testing.assert_allclose(dq, dq_r, atol=1e-13)
    np.testing.assert_allclose(dk, dk_r.reshape(B, S, 2, 2, D).sum(axis=3), atol=1e-13)
    np.testing.assert_allclose(dv, dv_r.reshape(B, S, 2, 2, D).sum(axis=3), atol=1e-13)
