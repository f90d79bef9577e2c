"""Pins for the fp64 oracle's forward pass (CPU only).

Each test checks the oracle against something other than itself: a closed
form, an invariant of the definition, a library routine (scipy), or a
brute-force pure-Python evaluation on a tiny input.  Together they are chosen
so that a dropped scale, a wrong mask direction or offset, a transposed
operand, a wrong grouped-query head mapping, a log-sum-exp in the wrong base or
a missing max subtraction each fails at least one of them.
"""

import math

import numpy as np
import pytest
import scipy.special

import oracle


def _rand(rng, *shape):
    return rng.standard_normal(shape)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Sk", [(7, 7), (5, 9), (9, 5), (130, 130)])
def test_zero_queries_average_visible_values(rng, causal, Sq, Sk):
    """Q = 0: all visible scores are equal, so O_i is the mean of the visible V
    rows and lse_i = ln(number of visible keys)."""
    D = 4
    q = np.zeros((Sq, D))
    k, v = _rand(rng, Sk, D), _rand(rng, Sk, 3)
    o, lse = oracle.head_forward(q, k, v, causal, 0.7)
    for i in range(Sq):
        n = Sk if not causal else max(0, min(Sk, i + (Sk - Sq) + 1))
        if n == 0:
            assert np.all(o[i] == 0.0) and lse[i] == -np.inf
        else:
            np.testing.assert_allclose(o[i], v[:n].mean(axis=0) if causal else v.mean(axis=0),
                                       rtol=0, atol=1e-13)
            assert abs(lse[i] - math.log(n)) < 1e-13


def test_causal_first_row_is_first_value(rng):
    """Causal, Sq == Sk: row 0 sees key 0 only, so O_0 = V_0 and
    lse_0 = scale * q_0 . k_0."""
    q, k, v = _rand(rng, 6, 5), _rand(rng, 6, 5), _rand(rng, 6, 5)
    o, lse = oracle.head_forward(q, k, v, True, 0.3)
    np.testing.assert_allclose(o[0], v[0], rtol=0, atol=1e-15)
    assert abs(lse[0] - 0.3 * float(q[0] @ k[0])) < 1e-13


def test_causal_last_row_equals_full_attention(rng):
    """Causal with Sq == Sk: the last row sees every key."""
    q, k, v = _rand(rng, 9, 4), _rand(rng, 9, 4), _rand(rng, 9, 4)
    oc, lc = oracle.head_forward(q, k, v, True, 0.5)
    of, lf = oracle.head_forward(q, k, v, False, 0.5)
    np.testing.assert_allclose(oc[-1], of[-1], atol=1e-14)
    assert abs(lc[-1] - lf[-1]) < 1e-13
    assert not np.allclose(oc[0], of[0])


def test_single_key(rng):
    """Sk = 1: O = V_0 and lse = scale * q . k_0 on every row."""
    q, k, v = _rand(rng, 5, 3), _rand(rng, 1, 3), _rand(rng, 1, 2)
    o, lse = oracle.head_forward(q, k, v, False, 1.7)
    np.testing.assert_allclose(o, np.repeat(v, 5, axis=0), atol=1e-15)
    np.testing.assert_allclose(lse, 1.7 * (q @ k[0]), atol=1e-13)


def test_two_keys_is_a_logistic_mix(rng):
    """Two keys: weight on key 0 is 1 / (1 + exp(s1 - s0))."""
    q, k, v = _rand(rng, 4, 3), _rand(rng, 2, 3), _rand(rng, 2, 6)
    scale = 0.9
    o, lse = oracle.head_forward(q, k, v, False, scale)
    for i in range(4):
        s0, s1 = scale * q[i] @ k[0], scale * q[i] @ k[1]
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        np.testing.assert_allclose(o[i], w0 * v[0] + (1 - w0) * v[1], atol=1e-14)
        assert abs(lse[i] - (max(s0, s1) + math.log1p(math.exp(-abs(s1 - s0))))) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("logit_scale", [1.0, 1000.0])
def test_matches_scipy_softmax_and_logsumexp(rng, causal, logit_scale):
    """Weights equal scipy.special.softmax of the masked scores and lse equals
    scipy.special.logsumexp (natural log), including logits large enough to
    overflow exp() without the max subtraction."""
    Sq, Sk, D = 11, 13, 8
    q, k = logit_scale * _rand(rng, Sq, D), _rand(rng, Sk, D)
    scale = D ** -0.5
    p, lse = oracle.head_probabilities(q, k, causal, scale)
    s = scale * q @ k.T
    vis = oracle.visible_mask(np.arange(Sq), Sq, Sk, causal)
    s_masked = np.where(vis, s, -np.inf)
    # relative error of exp(x) grows like |x| * eps: ~1e-12 at |x| ~ 1e3
    np.testing.assert_allclose(p, scipy.special.softmax(s_masked, axis=1), rtol=1e-9, atol=1e-300)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(s_masked, axis=1), rtol=1e-13)
    assert np.all(np.isfinite(lse))
    if logit_scale > 1:
        # exp() of these scores overflows (> 709) or underflows every term of a
        # row (< -745) unless the row maximum is subtracted first
        assert np.max(np.abs(s_masked[np.isfinite(s_masked)])) > 745.0


@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one_and_are_nonnegative(rng, causal):
    q, k = 3 * _rand(rng, 40, 16), _rand(rng, 40, 16)
    p, _ = oracle.head_probabilities(q, k, causal, 0.25)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    if causal:
        assert np.all(p[np.triu_indices(40, 1)] == 0.0)


def test_key_permutation_invariance(rng):
    """Non-causal: permuting key/value rows together changes nothing."""
    q, k, v = _rand(rng, 10, 4), _rand(rng, 12, 4), _rand(rng, 12, 5)
    perm = rng.permutation(12)
    o1, l1 = oracle.head_forward(q, k, v, False, 0.5)
    o2, l2 = oracle.head_forward(q, k[perm], v[perm], False, 0.5)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_moves_lse_only(rng, causal):
    """Adding u to every key shifts row i's scores by scale*q_i.u: O is
    unchanged and lse moves by exactly that amount."""
    q, k, v = _rand(rng, 8, 4), _rand(rng, 8, 4), _rand(rng, 8, 4)
    u = _rand(rng, 4)
    o1, l1 = oracle.head_forward(q, k, v, causal, 0.6)
    o2, l2 = oracle.head_forward(q, k + u, v, causal, 0.6)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l2 - l1, 0.6 * q @ u, atol=1e-12)


def test_fully_masked_rows_are_zero_with_minus_inf_lse(rng):
    """Causal with Sq > Sk (bottom-right alignment): the first Sq - Sk rows see
    no key."""
    q, k, v = _rand(rng, 6, 3), _rand(rng, 4, 3), _rand(rng, 4, 3)
    o, lse = oracle.head_forward(q, k, v, True, 1.0)
    assert np.all(o[:2] == 0) and np.all(lse[:2] == -np.inf)
    np.testing.assert_allclose(o[2], v[0], atol=1e-15)
    assert np.all(np.isfinite(lse[2:]))


def test_brute_force_pure_python(rng):
    """Tiny case evaluated with Python floats and math.exp, term by term."""
    Sq, Sk, D = 3, 4, 2
    q, k, v = _rand(rng, Sq, D), _rand(rng, Sk, D), _rand(rng, Sk, D)
    scale = 0.8
    for causal in (False, True):
        o, lse = oracle.head_forward(q, k, v, causal, scale)
        for i in range(Sq):
            keys = [j for j in range(Sk) if not causal or j <= i + (Sk - Sq)]
            s = {j: scale * sum(float(q[i, d]) * float(k[j, d]) for d in range(D)) for j in keys}
            z = sum(math.exp(s[j]) for j in keys)
            for d in range(D):
                ref = sum(math.exp(s[j]) / z * float(v[j, d]) for j in keys)
                assert abs(o[i, d] - ref) < 1e-13
            assert abs(lse[i] - math.log(z)) < 1e-13


def test_grouped_query_heads_map_to_floor_division(rng):
    """Hq = 4, Hkv = 2: query heads 0,1 read kv head 0 and 2,3 read kv head 1,
    i.e. the same as plain multi-head attention on K/V heads repeated in
    place (np.repeat), not tiled."""
    B, S, D = 2, 6, 3
    q = _rand(rng, B, S, 4, D)
    k, v = _rand(rng, B, S, 2, D), _rand(rng, B, S, 2, D)
    o, lse = oracle.attention_forward(q, k, v, False, 0.5)
    o_rep, lse_rep = oracle.attention_forward(q, np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2),
                                              False, 0.5)
    np.testing.assert_allclose(o, o_rep, atol=1e-14)
    np.testing.assert_allclose(lse, lse_rep, atol=1e-13)
    oh, lh = oracle.head_forward(q[1, :, 1, :], k[1, :, 0, :], v[1, :, 0, :], False, 0.5)
    np.testing.assert_allclose(o[1, :, 1, :], oh, atol=1e-14)
    np.testing.assert_allclose(lse[1, 1], lh, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_varlen_equals_per_sequence(rng, causal):
    lens = [5, 1, 9, 4]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, Hq, Hkv, D = int(cu[-1]), 4, 2, 3
    q, k, v = _rand(rng, T, Hq, D), _rand(rng, T, Hkv, D), _rand(rng, T, Hkv, D)
    o, lse = oracle.attention_forward(q, k, v, causal, 0.4, cu_seqlens=cu)
    assert lse.shape == (Hq, T)
    for b, L in enumerate(lens):
        sl = slice(int(cu[b]), int(cu[b + 1]))
        ob, lb = oracle.attention_forward(q[None, sl], k[None, sl], v[None, sl], causal, 0.4)
        np.testing.assert_allclose(o[sl], ob[0], atol=1e-14)
        np.testing.assert_allclose(lse[:, sl], lb[0], atol=1e-13)


def test_row_subset_matches_full(rng):
    """Sampling rows (used for large-size parity) gives the same rows."""
    q, k, v = _rand(rng, 50, 4), _rand(rng, 50, 4), _rand(rng, 50, 4)
    rows = np.array([0, 7, 31, 49])
    o, lse = oracle.head_forward(q, k, v, True, 0.5)
    os_, ls_ = oracle.head_forward(q, k, v, True, 0.5, rows=rows)
    np.testing.assert_allclose(os_, o[rows], atol=1e-15)
    np.testing.assert_allclose(ls_, lse[rows], atol=1e-15)
