"""Backward pass with the main kernel on CTA pairs (paired tcgen05 MMAs over
two adjacent key blocks; dQ summed over both before it is added), through
fa_bwd_ex with paired = 1, against the fp64 oracle's analytic gradients on
seeded BF16 inputs.  Relative Frobenius error <= 1e-2 per gradient, and close
agreement with the unpaired kernel on the same inputs.

The shapes cover what is particular to pairs: an odd number of 128-key blocks
(the last pair's second block is empty or partly past Sk), causal pairs whose
second block sees fewer query blocks than the first, grouped heads, Sq != Sk,
and the deterministic mode with one ticket per (query block, feature half).
"""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_78_gb300 import workloads as W

from parity import GRAD_RTOL, f64, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_78_gb300 as fa_mod
    fa_mod.load_library(build_if_missing=True)
    return fa_mod


def _inputs(B, Hq, Hkv, Sq, Sk, seed=0, q_scale=1.0):
    w = W.Workload("case", B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, D=128, causal=False, seed=seed, q_scale=q_scale)
    (q, k, v, do), _ = W.make_inputs(w, with_grad=True)
    return q, k, v, do


def _grads(fa, q, k, v, do, causal, paired, deterministic=False):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, deterministic=deterministic, paired=paired)
    assert fa.get_device_error() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


def _check(grads, q, k, v, do, causal):
    ref = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), causal, 128 ** -0.5)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        gg = f64(g)
        assert np.all(np.isfinite(gg)), name
        if np.linalg.norm(r) < 1e-9:
            assert np.max(np.abs(gg)) <= 1e-3, name
            continue
        e = rel_fro(gg, r)
        assert e <= GRAD_RTOL, (name, e)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk", [
    (1, 2, 2, 128, 128),     # one key block: the pair's second block is empty
    (1, 2, 2, 256, 256),     # exactly one pair
    (2, 4, 2, 300, 300),     # grouped heads, ragged rows and keys (3 blocks: odd)
    (1, 2, 1, 1000, 1000),   # several pairs, last block partial
    (1, 2, 2, 129, 640),     # Sq < Sk, 5 key blocks
    (1, 2, 2, 520, 300),     # Sq > Sk: causal leaves the first rows without keys
    (1, 1, 1, 1, 1),
])
def test_paired_small_shapes(fa, causal, B, Hq, Hkv, Sq, Sk):
    q, k, v, do = _inputs(B, Hq, Hkv, Sq, Sk, seed=14)
    _check(_grads(fa, q, k, v, do, causal, paired=True), q, k, v, do, causal)


def test_paired_stress_logits(fa):
    q, k, v, do = _inputs(1, 2, 2, 768, 768, seed=3, q_scale=4.0)
    _check(_grads(fa, q, k, v, do, True, paired=True), q, k, v, do, True)


@pytest.mark.parametrize("causal", [False, True])
def test_paired_matches_unpaired(fa, causal):
    q, k, v, do = _inputs(2, 4, 4, 1100, 1100, seed=9)
    a = _grads(fa, q, k, v, do, causal, paired=True)
    b = _grads(fa, q, k, v, do, causal, paired=False)
    for name, x, y in zip(("dq", "dk", "dv"), a, b):
        assert rel_fro(f64(x), f64(y)) <= 2e-3, name


@pytest.mark.parametrize("causal", [False, True])
def test_paired_deterministic_is_bitwise_repeatable(fa, causal):
    q, k, v, do = _inputs(2, 4, 2, 700, 900, seed=8)
    a = _grads(fa, q, k, v, do, causal, paired=True, deterministic=True)
    b = _grads(fa, q, k, v, do, causal, paired=True, deterministic=True)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    _check(a, q, k, v, do, causal)


@pytest.mark.parametrize("deterministic", [False, True])
def test_paired_training_shape_sampled_heads(fa, deterministic):
    """B=2, H=16, S=8192, D=128, causal: gradients of whole heads compared."""
    w = W.train(deterministic)
    (q, k, v, do), _ = W.make_inputs(w, with_grad=True)
    dq, dk, dv = _grads(fa, q, k, v, do, True, paired=True, deterministic=deterministic)
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
    heads = [(1, 7)] if deterministic else [(0, 0), (1, 12)]
    for b, h in heads:
        gq, gk, gv = oracle.head_backward(f64(q[b, :, h]), f64(k[b, :, h]), f64(v[b, :, h]), f64(do[b, :, h]),
                                          True, w.scale)
        for name, g, r in (("dq", dq[b, :, h], gq), ("dk", dk[b, :, h], gk), ("dv", dv[b, :, h], gv)):
            e = rel_fro(f64(g), r)
            assert e <= GRAD_RTOL, (b, h, name, e)
