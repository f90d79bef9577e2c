"""Backward-pass parity on the GPU: dQ, dK, dV from the CUDA library (through
its C ABI) against the fp64 oracle's analytic gradients on the same seeded
BF16 inputs.  Relative Frobenius error <= 1e-2 per gradient.

The GPU backward uses the GPU forward's BF16 O and FP32 LSE (as a training
step would); the oracle uses its own fp64 O.  The difference is at the level
of BF16 rounding and is covered by the tolerance.
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


def _inputs(B, Hq, Hkv, Sq, Sk, seed=0, q_scale=1.0, D=128):
    w = W.Workload("case", B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, D=D, causal=False, seed=seed, q_scale=q_scale)
    (q, k, v, do), _ = W.make_inputs(w, with_grad=True)
    return q, k, v, do


def _gpu_grads(fa, q, k, v, do, causal, deterministic=False, poison=False):
    """poison: the gradient buffers start as NaN, so a finiteness check of
    the result shows that every element was written."""
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=causal)
    outs = {}
    if poison:
        outs = {n: torch.full_like(t, float("nan")) for n, t in (("dq", qd), ("dk", kd), ("dv", vd))}
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, deterministic=deterministic, **outs)
    assert fa.get_device_error() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


def _check(grads, q, k, v, do, causal):
    ref = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), causal, q.shape[-1] ** -0.5)
    errs = []
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        gg = f64(g)
        assert np.all(np.isfinite(gg)), name
        if np.linalg.norm(r) < 1e-9:
            # an identically zero gradient (e.g. a single key: dS = 0, so dQ =
            # dK = 0): only rounding noise may remain
            assert np.max(np.abs(gg)) <= 1e-3, name
            continue
        e = rel_fro(gg, r)
        errs.append(e)
        assert e <= GRAD_RTOL, (name, e)
    return errs


@pytest.mark.parametrize("causal", [False, True])
def test_single_tile(fa, causal):
    q, k, v, do = _inputs(1, 2, 2, 128, 128)
    _check(_gpu_grads(fa, q, k, v, do, causal), q, k, v, do, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk", [
    (1, 2, 2, 256, 256),
    (2, 4, 2, 300, 300),     # grouped heads, ragged rows and keys
    (1, 2, 1, 1000, 1000),   # several key blocks and query blocks
    (1, 2, 2, 129, 257),     # Sq < Sk
    (1, 2, 2, 520, 300),     # Sq > Sk: causal leaves the first rows without keys
    (1, 1, 1, 1, 1),
])
def test_small_shapes_full_compare(fa, causal, B, Hq, Hkv, Sq, Sk):
    q, k, v, do = _inputs(B, Hq, Hkv, Sq, Sk, seed=4)
    _check(_gpu_grads(fa, q, k, v, do, causal), q, k, v, do, causal)


def test_zero_queries_give_averaged_dv(fa):
    """Closed form: Q = 0 -> uniform weights over the visible keys, so
    dV_j = sum over rows i that see j of dO_i / (i + 1) (causal)."""
    q, k, v, do = _inputs(1, 1, 1, 384, 384, seed=6)
    q = torch.zeros_like(q)
    _, _, dv = _gpu_grads(fa, q, k, v, do, True)
    g = f64(do)[0, :, 0]
    w = 1.0 / np.arange(1, 385)
    ref = np.cumsum((g * w[:, None])[::-1], axis=0)[::-1]
    assert rel_fro(f64(dv)[0, :, 0], ref) <= GRAD_RTOL


def test_stress_logits(fa):
    q, k, v, do = _inputs(1, 2, 2, 512, 512, seed=1, q_scale=4.0)
    _check(_gpu_grads(fa, q, k, v, do, True), q, k, v, do, True)


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic_is_bitwise_repeatable(fa, causal):
    q, k, v, do = _inputs(2, 4, 2, 700, 700, seed=8)
    a = _gpu_grads(fa, q, k, v, do, causal, deterministic=True)
    b = _gpu_grads(fa, q, k, v, do, causal, deterministic=True)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    _check(a, q, k, v, do, causal)
    c = _gpu_grads(fa, q, k, v, do, causal, deterministic=False)
    for x, y in zip(a, c):
        assert rel_fro(f64(x), f64(y)) <= 2e-3


# ------------------------------------------------------------------ D = 64 --

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk", [
    (1, 2, 2, 128, 128),
    (2, 4, 2, 300, 300),     # grouped heads, ragged rows and keys
    (1, 2, 1, 1000, 1000),   # several key blocks and query blocks
    (1, 2, 2, 520, 300),     # Sq > Sk
])
def test_d64_shapes_full_compare(fa, causal, B, Hq, Hkv, Sq, Sk):
    q, k, v, do = _inputs(B, Hq, Hkv, Sq, Sk, seed=12, D=64)
    _check(_gpu_grads(fa, q, k, v, do, causal), q, k, v, do, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_d64_deterministic_is_bitwise_repeatable(fa, causal):
    q, k, v, do = _inputs(2, 4, 2, 700, 700, seed=13, D=64)
    a = _gpu_grads(fa, q, k, v, do, causal, deterministic=True)
    b = _gpu_grads(fa, q, k, v, do, causal, deterministic=True)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    _check(a, q, k, v, do, causal)


def test_d64_stress_logits(fa):
    q, k, v, do = _inputs(1, 2, 2, 512, 512, seed=1, q_scale=4.0, D=64)
    _check(_gpu_grads(fa, q, k, v, do, True), q, k, v, do, True)


# ---------------------------------------------------------------- full size --

@pytest.mark.parametrize("deterministic", [False, True])
def test_training_shape_sampled_heads(fa, deterministic):
    """B=2, H=16, S=8192, D=128, causal: gradients of whole heads compared."""
    w = W.train(deterministic)
    (q, k, v, do), _ = W.make_inputs(w, with_grad=True)
    dq, dk, dv = _gpu_grads(fa, q, k, v, do, True, deterministic=deterministic, poison=True)
    for t in (dq, dk, dv):   # every element written (the buffers started as NaN)
        assert bool(torch.isfinite(t.float()).all())
    heads = [(0, 0)] if deterministic else [(0, 3), (1, 15)]
    for b, h in heads:
        gq, gk, gv = oracle.head_backward(f64(q[b, :, h]), f64(k[b, :, h]), f64(v[b, :, h]), f64(do[b, :, h]),
                                          True, w.scale)
        for name, g, r in (("dq", dq[b, :, h], gq), ("dk", dk[b, :, h], gk), ("dv", dv[b, :, h], gv)):
            e = rel_fro(f64(g), r)
            assert e <= GRAD_RTOL, (b, h, name, e)


def _heads_vs_oracle(q, k, v, do, grads, causal, scale, heads):
    """Whole (batch, head) slices of the gradients against the oracle's
    analytic gradients of that head (Hq == Hkv)."""
    dq, dk, dv = grads
    worst = 0.0
    for b, h in heads:
        gq, gk, gv = oracle.head_backward(f64(q[b, :, h]), f64(k[b, :, h]), f64(v[b, :, h]), f64(do[b, :, h]),
                                          causal, scale)
        for name, g, r in (("dq", dq[b, :, h], gq), ("dk", dk[b, :, h], gk), ("dv", dv[b, :, h], gv)):
            e = rel_fro(f64(g), r)
            worst = max(worst, e)
            assert e <= GRAD_RTOL, (b, h, name, e)
    return worst


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("stress", [False, True])
def test_dense_config_sampled_heads(fa, causal, stress):
    """The benchmark's dense workload (B=4, H=16, S=4096, D=128) at full size,
    through fa_bwd's default launch (static schedule: head-major without a
    mask, key-block-major within groups of 32 heads with one), so every CTA
    runs many units.  Whole heads spread over the batch and the head range
    are compared; the Q x 4 stress seed (logit std ~16) exercises large
    maxima in the recomputed weights."""
    w = W.dense(causal=causal, stress=stress)
    (q, k, v, do), _ = W.make_inputs(w, with_grad=True)
    grads = _gpu_grads(fa, q, k, v, do, causal, poison=True)
    for t in grads:   # every element written (the buffers started as NaN)
        assert bool(torch.isfinite(t.float()).all())
    _heads_vs_oracle(q, k, v, do, grads, causal, w.scale, [(0, 0), (1, 9), (3, 15)])


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1024, 2048, 4096, 8192])
@pytest.mark.parametrize("causal", [False, True])
def test_sweep_config_sampled_heads(fa, D, S, causal):
    """Sequence-length sweep (B*S = 32768 tokens, H=16) at full size: the
    first and the last (batch, head) slice of each call."""
    w = W.sweep(S, D, causal)
    (q, k, v, do), _ = W.make_inputs(w, with_grad=True)
    grads = _gpu_grads(fa, q, k, v, do, causal, poison=True)
    for t in grads:   # every element written (the buffers started as NaN)
        assert bool(torch.isfinite(t.float()).all())
    _heads_vs_oracle(q, k, v, do, grads, causal, w.scale, [(0, 0), (w.B - 1, 15)])


def _grads_tuned(fa, q, k, v, do, causal, deterministic, tuning):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, deterministic=deterministic, tuning=tuning)
    assert fa.get_device_error() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk", [
    (2, 4, 2, 300, 300),     # grouped heads, ragged rows and keys
    (1, 2, 1, 1000, 1000),   # several 64-key blocks and query tiles
    (1, 2, 2, 129, 257),     # Sq < Sk
    (1, 2, 2, 520, 300),     # Sq > Sk: causal leaves the first rows without keys
    (1, 1, 1, 1, 1),
])
def test_split_dq_kernel(fa, D, causal, B, Hq, Hkv, Sq, Sk):
    """The split backward (dK / dV from the main kernel without its dQ
    product, dQ from the query-tile kernel): oracle parity, bitwise repeats,
    and agreement with the fused kernel's atomic dQ."""
    q, k, v, do = _inputs(B, Hq, Hkv, Sq, Sk, seed=17, D=D)
    a = _grads_tuned(fa, q, k, v, do, causal, False, {"split_dq": 1})
    _check(a, q, k, v, do, causal)
    b = _grads_tuned(fa, q, k, v, do, causal, False, {"split_dq": 1})
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    c = _grads_tuned(fa, q, k, v, do, causal, False, {"split_dq": 0})
    for x, y in zip(a, c):
        if np.linalg.norm(f64(y)) > 1e-9:
            assert rel_fro(f64(x), f64(y)) <= 2e-3


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic_ticket_path_still_available(fa, causal):
    """split_dq = 0 keeps the fused kernel's ticket-ordered dQ additions in
    deterministic mode: bitwise repeatable and equal (to rounding) to the
    default split path."""
    q, k, v, do = _inputs(2, 4, 2, 700, 700, seed=18)
    a = _grads_tuned(fa, q, k, v, do, causal, True, {"split_dq": 0})
    b = _grads_tuned(fa, q, k, v, do, causal, True, {"split_dq": 0})
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    _check(a, q, k, v, do, causal)
    c = _gpu_grads(fa, q, k, v, do, causal, deterministic=True)
    for x, y in zip(a, c):
        assert rel_fro(f64(x), f64(y)) <= 2e-3
