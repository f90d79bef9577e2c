"""Backward pass in the packed variable-length layout (cu_seqlens), through
the C ABI, against the fp64 oracle's analytic gradients of each sequence:
every sequence is an independent attention problem over its own tokens
(causal mask aligned to its own start), and dK/dV of a key/value head sum
over its query-head group.  Relative Frobenius error <= 1e-2 per gradient.
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


def _packed(lens, Hq, Hkv, seed, D=128):
    cu = W.cu_seqlens_of(lens)
    T = int(cu[-1])
    q = W.randn_bf16((T, Hq, D), 100 * seed + 1)
    k = W.randn_bf16((T, Hkv, D), 100 * seed + 2)
    v = W.randn_bf16((T, Hkv, D), 100 * seed + 3)
    do = W.randn_bf16((T, Hq, D), 100 * seed + 4)
    return q, k, v, do, cu


def _gpu(fa, q, k, v, do, cu, causal, deterministic=False, tuning=None, poison=False):
    """poison: the gradient buffers start as NaN (a finiteness check then
    shows that every element was written)."""
    qd, kd, vd, dod, cud = (t.cuda() for t in (q, k, v, do, cu))
    o, lse = fa.fwd(qd, kd, vd, causal=causal, cu_seqlens=cud)
    outs = {}
    if poison:
        outs = {n: torch.full_like(t, float("nan")) for n, t in (("dq", qd), ("dk", kd), ("dv", vd))}
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, cu_seqlens=cud, deterministic=deterministic,
                        tuning=tuning, **outs)
    assert fa.get_device_error() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


def _reference(q, k, v, do, cu, causal, seqs=None, heads=None):
    """Per-sequence, per-head oracle gradients; dK/dV summed over each group."""
    Hq, Hkv = q.shape[1], k.shape[1]
    g = Hq // Hkv
    scale = q.shape[-1] ** -0.5
    out = {}
    seqs = range(len(cu) - 1) if seqs is None else seqs
    for b in seqs:
        s, e = int(cu[b]), int(cu[b + 1])
        if e == s:
            continue
        for h in (range(Hq) if heads is None else heads):
            hk = h // g
            gq, gk, gv = oracle.head_backward(f64(q[s:e, h]), f64(k[s:e, hk]), f64(v[s:e, hk]), f64(do[s:e, h]),
                                              causal, scale)
            out[(b, h)] = (gq, gk, gv)
    return out


def _check_full(grads, q, k, v, do, cu, causal):
    dq, dk, dv = (f64(t) for t in grads)
    Hq, Hkv = q.shape[1], k.shape[1]
    g = Hq // Hkv
    ref = _reference(q, k, v, do, cu, causal)
    rq, rk, rv = np.zeros(dq.shape), np.zeros(dk.shape), np.zeros(dv.shape)
    for (b, h), (gq, gk, gv) in ref.items():
        s, e = int(cu[b]), int(cu[b + 1])
        rq[s:e, h] = gq
        rk[s:e, h // g] += gk
        rv[s:e, h // g] += gv
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert np.all(np.isfinite(got)), name
        e = rel_fro(got, want)
        assert e <= GRAD_RTOL, (name, e)
        # every sequence on its own too (short ones are a tiny share of the norm)
        for b in range(len(cu) - 1):
            s, t = int(cu[b]), int(cu[b + 1])
            if t == s:
                continue
            w = want[s:t]
            if np.linalg.norm(w) < 1e-9:
                assert np.max(np.abs(got[s:t])) <= 1e-3, (name, b)
            else:
                assert rel_fro(got[s:t], w) <= GRAD_RTOL, (name, b, rel_fro(got[s:t], w))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lens,Hq,Hkv", [
    ([1, 130, 0, 513, 256, 77, 1000], 4, 2),   # ragged, an empty sequence, grouped heads
    ([63, 64, 65, 127, 128, 129], 2, 2),       # lengths around the 64-row and 128-key tiles
    ([700], 2, 1),                              # a single sequence
])
def test_packed_backward_matches_oracle(fa, causal, lens, Hq, Hkv):
    q, k, v, do, cu = _packed(lens, Hq, Hkv, seed=len(lens))
    _check_full(_gpu(fa, q, k, v, do, cu, causal), q, k, v, do, cu, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_backward_d64(fa, causal):
    q, k, v, do, cu = _packed([1, 130, 0, 513, 256, 77], 4, 2, seed=9, D=64)
    _check_full(_gpu(fa, q, k, v, do, cu, causal), q, k, v, do, cu, causal)


@pytest.mark.parametrize("tuning", [None, {"split_dq": 0}], ids=["default", "tickets"])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_deterministic_is_bitwise_repeatable(fa, causal, tuning):
    """Deterministic mode on packed sequences, by default (the split
    backward) and through the ticket-ordered fused kernel."""
    q, k, v, do, cu = _packed([300, 45, 900, 128], 4, 2, seed=5)
    a = _gpu(fa, q, k, v, do, cu, causal, deterministic=True, tuning=tuning)
    b = _gpu(fa, q, k, v, do, cu, causal, deterministic=True, tuning=tuning)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    _check_full(a, q, k, v, do, cu, causal)
    c = _gpu(fa, q, k, v, do, cu, causal)
    for x, y in zip(a, c):
        assert rel_fro(f64(x), f64(y)) <= 2e-3


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_split_dq_kernel(fa, D, causal):
    """The split backward on packed sequences (dK / dV from the main kernel
    without its dQ product, dQ from the query-tile kernel over each
    sequence's own keys), including empty, one-token and tile-boundary
    lengths: oracle parity and bitwise repeats."""
    q, k, v, do, cu = _packed([1, 130, 0, 513, 256, 77, 128, 129], 4, 2, seed=21, D=D)
    qd, kd, vd, dod, cud = (t.cuda() for t in (q, k, v, do, cu))
    o, lse = fa.fwd(qd, kd, vd, causal=causal, cu_seqlens=cud)
    runs = []
    for _ in range(2):
        g = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, cu_seqlens=cud, deterministic=True,
                   tuning={"split_dq": 1})
        assert fa.get_device_error() == 0
        runs.append(tuple(t.cpu() for t in g))
    for x, y in zip(*runs):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    _check_full(runs[0], q, k, v, do, cu, causal)


def test_packed_matches_dense_for_equal_lengths(fa):
    """Equal-length sequences packed back to back give the dense result."""
    B, S, H = 3, 384, 2
    q, k, v, do, cu = _packed([S] * B, H, H, seed=7)
    packed = _gpu(fa, q, k, v, do, cu, True)
    dense = [t.cuda().view(B, S, H, 128) for t in (q, k, v, do)]
    o, lse = fa.fwd(*dense[:3], causal=True)
    dd = fa.bwd(*dense[:3], o, lse, dense[3], causal=True)
    for x, y in zip(packed, dd):
        assert rel_fro(f64(x), f64(y.cpu().view(B * S, H, 128))) <= 2e-3


@pytest.mark.parametrize("deterministic", [False, True])
def test_varlen_gqa_config_sampled_sequences(fa, deterministic):
    """64 packed sequences (lengths 128..8192), Hq=32, Hkv=8, causal: whole
    (sequence, head) gradients of a few sequences compared with the oracle,
    atomic and deterministic (the split backward)."""
    w = W.varlen_gqa()
    (q, k, v, do), cu = W.make_inputs(w, with_grad=True)
    dq, dk, dv = _gpu(fa, q, k, v, do, cu, True, deterministic=deterministic, poison=True)
    for t in (dq, dk, dv):   # every element written (the buffers started as NaN)
        assert bool(torch.isfinite(t.float()).all())
    lens = np.diff(cu.numpy())
    seqs = [int(np.argmin(lens)), int(np.argmax(lens)), 17]
    g = w.Hq // w.Hkv
    for b in seqs:
        s, e = int(cu[b]), int(cu[b + 1])
        hk = 3
        ref = _reference(q, k, v, do, cu, True, seqs=[b], heads=range(hk * g, hk * g + g))
        rk = sum(ref[(b, h)][1] for h in range(hk * g, hk * g + g))
        rv = sum(ref[(b, h)][2] for h in range(hk * g, hk * g + g))
        for h in (hk * g, hk * g + g - 1):
            assert rel_fro(f64(dq[s:e, h]), ref[(b, h)][0]) <= GRAD_RTOL, (b, h)
        assert rel_fro(f64(dk[s:e, hk]), rk) <= GRAD_RTOL, b
        assert rel_fro(f64(dv[s:e, hk]), rv) <= GRAD_RTOL, b


def test_packed_bad_offsets_are_reported_not_computed(fa):
    """Decreasing offsets: FA_ERR_INVALID_ARG from the device, no output written."""
    cu = W.cu_seqlens_of([100, 200, 50]).cuda()
    cu[1] = 320          # 0, 320, 300, 350: the second sequence has negative length
    T = 350
    q = W.randn_bf16((T, 2, 128), 1).cuda()
    o = torch.zeros_like(q)
    lse = torch.zeros((2, T), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.full_like(q, 7.0) for _ in range(3))
    fa.bwd(q, q, q, o, lse, q, causal=True, cu_seqlens=cu, dq=dq, dk=dk, dv=dv)
    assert fa.get_device_error() == fa.binding.FA_ERR_INVALID_ARG
    assert fa.get_device_error() == 0
    for t in (dq, dk, dv):
        assert bool((t == 7.0).all())
