"""Backward parity under every work order the library can run: static and
claimed schedules, head groups, query blocks visited first to last or last
to first, and the S^T-before-read-out issue order, in atomic and
deterministic mode.  Each configuration is compared with
the fp64 oracle's analytic gradients (relative Frobenius <= 1e-2); a
deterministic configuration must also repeat bit for bit.

The knobs change only the order of the work and of the FP32 additions, so
every configuration has the same tolerance as the default one.
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


def _inputs(B, Hq, Hkv, Sq, Sk, seed, D=128):
    w = W.Workload("case", B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, D=D, causal=False, seed=seed)
    (q, k, v, do), _ = W.make_inputs(w, with_grad=True)
    return q, k, v, do


def _grads(fa, q, k, v, do, causal, deterministic, tuning, cu=None):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    cud = None if cu is None else cu.cuda()
    o, lse = fa.fwd(qd, kd, vd, causal=causal, cu_seqlens=cud)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, deterministic=deterministic, cu_seqlens=cud,
                        tuning=tuning)
    assert fa.get_device_error() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


def _check_dense(grads, q, k, v, do, causal):
    ref = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), causal, q.shape[-1] ** -0.5)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        e = rel_fro(f64(g), r)
        assert e <= GRAD_RTOL, (name, e)


ATOMIC = [
    {"schedule": 0, "head_group": 1},
    {"schedule": 0, "head_group": 3, "reverse_blocks": 1},
    {"schedule": 1, "head_group": 1},
    {"schedule": 1, "head_group": 64, "reverse_blocks": 1},
    {"schedule": 1, "head_group": 2, "scores_first": 0},
    {"schedule": 0, "scores_first": 1, "reverse_blocks": 1},
]

DETERMINISTIC = [
    {"reverse_blocks": 0},
    {"reverse_blocks": 1},
    {"reverse_blocks": 1, "scores_first": 1},
    {"schedule": 0, "reverse_blocks": 1},
    {"schedule": 0, "head_group": 1, "reverse_blocks": 1},
    {"schedule": 1, "head_group": 3, "scores_first": 1},
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tuning", ATOMIC, ids=lambda t: ",".join("%s=%d" % kv for kv in t.items()))
def test_atomic_orders_match_oracle(fa, causal, tuning):
    # several key and query blocks per head, grouped heads, a ragged tail
    q, k, v, do = _inputs(2, 4, 2, 700, 700, seed=21)
    _check_dense(_grads(fa, q, k, v, do, causal, False, tuning), q, k, v, do, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tuning", DETERMINISTIC, ids=lambda t: ",".join("%s=%d" % kv for kv in t.items()))
def test_deterministic_orders_repeat_and_match_oracle(fa, causal, tuning):
    q, k, v, do = _inputs(2, 4, 2, 700, 700, seed=22)
    a = _grads(fa, q, k, v, do, causal, True, tuning)
    b = _grads(fa, q, k, v, do, causal, True, tuning)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    _check_dense(a, q, k, v, do, causal)


@pytest.mark.parametrize("tuning", [{"reverse_blocks": 0}, {"reverse_blocks": 1}], ids=["fwd", "rev"])
def test_deterministic_orders_sq_not_sk(fa, tuning):
    """Causal with Sq > Sk: the first query rows see no key (zero gradient
    rows), and the last query block is the only one every key block adds to."""
    q, k, v, do = _inputs(1, 2, 2, 520, 300, seed=23)
    a = _grads(fa, q, k, v, do, True, True, tuning)
    b = _grads(fa, q, k, v, do, True, True, tuning)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    _check_dense(a, q, k, v, do, True)


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("tuning", [{"reverse_blocks": 0}, {"reverse_blocks": 1}, {"scores_first": 0},
                                    {"scores_first": 1}], ids=["fwd", "rev", "wait_first", "scores_first"])
def test_packed_orders_match_oracle(fa, deterministic, tuning):
    """Packed sequences of mixed lengths (one of a single token, one ending
    one row past a block), grouped heads, causal."""
    lens = [300, 1, 700, 129, 1000]
    Hq, Hkv, D = 4, 2, 128
    cu = W.cu_seqlens_of(lens)
    T = int(cu[-1])
    q = W.randn_bf16((T, Hq, D), 2501)
    k = W.randn_bf16((T, Hkv, D), 2502)
    v = W.randn_bf16((T, Hkv, D), 2503)
    do = W.randn_bf16((T, Hq, D), 2504)
    a = _grads(fa, q, k, v, do, True, deterministic, tuning, cu=cu)
    if deterministic:
        b = _grads(fa, q, k, v, do, True, True, tuning, cu=cu)
        for x, y in zip(a, b):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    g = Hq // Hkv
    dq, dk, dv = (f64(t) for t in a)
    for s_ in range(len(lens)):
        lo, hi = int(cu[s_]), int(cu[s_ + 1])
        ref_dk = np.zeros((hi - lo, Hkv, D))
        ref_dv = np.zeros((hi - lo, Hkv, D))
        ref_dq = np.zeros((hi - lo, Hq, D))
        for h in range(Hq):
            hk = h // g
            gq, gk, gv = oracle.head_backward(f64(q[lo:hi, h]), f64(k[lo:hi, hk]), f64(v[lo:hi, hk]),
                                              f64(do[lo:hi, h]), True, D ** -0.5)
            ref_dq[:, h] = gq
            ref_dk[:, hk] += gk
            ref_dv[:, hk] += gv
        for name, got, ref in (("dq", dq[lo:hi], ref_dq), ("dk", dk[lo:hi], ref_dk), ("dv", dv[lo:hi], ref_dv)):
            if np.linalg.norm(ref) < 1e-9:
                assert np.max(np.abs(got)) <= 1e-3, (s_, name)
                continue
            e = rel_fro(got, ref)
            assert e <= GRAD_RTOL, (s_, name, e)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("group", [1, 3, 64])
def test_paired_kernel_head_groups(fa, causal, deterministic, group):
    """The paired-CTA kernel under every head grouping of its unit order
    (pairs of key blocks, longest first within a group)."""
    q, k, v, do = _inputs(2, 4, 2, 700, 700, seed=25)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=causal)
    runs = []
    for _ in range(2 if deterministic else 1):
        g = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, deterministic=deterministic, paired=True,
                   tuning={"head_group": group})
        assert fa.get_device_error() == 0
        runs.append(tuple(t.cpu() for t in g))
    if deterministic:
        for x, y in zip(*runs):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    _check_dense(runs[0], q, k, v, do, causal)
