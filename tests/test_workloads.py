"""Host-side input generation and FLOP accounting (no GPU): the seeded
inputs every test and the benchmark share, and the counting rule the
throughput figures use (forward 4*B*Hq*Sq*Sk*D, half under a causal mask,
backward 2.5 times the forward), pinned to the workload table's figures."""

import pytest
import torch

from exact_attention_78_gb300 import flops as F
from exact_attention_78_gb300 import workloads as W


def test_inputs_are_seeded_and_reproducible():
    w = W.Workload("case", B=1, Hq=2, Hkv=1, Sq=65, Sk=33, D=64, causal=False, seed=5)
    (q1, k1, v1, do1), cu1 = W.make_inputs(w, with_grad=True)
    (q2, k2, v2, do2), _ = W.make_inputs(w, with_grad=True)
    assert cu1 is None
    for a, b in ((q1, q2), (k1, k2), (v1, v2), (do1, do2)):
        assert a.dtype == torch.bfloat16 and torch.equal(a, b)
    assert q1.shape == (1, 65, 2, 64) and k1.shape == (1, 33, 1, 64) and do1.shape == q1.shape
    w2 = W.Workload("case", B=1, Hq=2, Hkv=1, Sq=65, Sk=33, D=64, causal=False, seed=6)
    (q3, _, _), _ = W.make_inputs(w2)
    assert not torch.equal(q1, q3)
    # Q, K, V and dO are independent draws, not copies of one another
    assert not torch.equal(q1[:, :33, :1], k1)


def test_stress_variant_scales_q_exactly():
    base = W.Workload("case", B=1, Hq=1, Hkv=1, Sq=64, Sk=64, D=64, causal=False, seed=3)
    stress = W.Workload("case", B=1, Hq=1, Hkv=1, Sq=64, Sk=64, D=64, causal=False, seed=3, q_scale=4.0)
    (q, k, _), _ = W.make_inputs(base)
    (qs, ks, _), _ = W.make_inputs(stress)
    assert torch.equal(qs, q * 4) and torch.equal(ks, k)     # a power of two is exact in BF16


def test_varlen_workload_lengths_and_offsets():
    lens = W.varlen_lengths()
    assert len(lens) == 64 and lens == W.varlen_lengths()
    assert all(128 <= L <= 8192 for L in lens)
    cu = W.cu_seqlens_of(lens)
    assert cu.dtype == torch.int32 and int(cu[0]) == 0 and int(cu[-1]) == sum(lens)
    assert all(int(cu[i + 1]) - int(cu[i]) == lens[i] for i in range(64))
    w = W.varlen_gqa()
    assert w.packed and w.Hq == 32 and w.Hkv == 8 and w.D == 128 and w.causal
    assert list(w.seqlens) == lens
    # a small packed case: inputs [total, H, D] with the same offsets
    small = W.Workload("case", B=3, Hq=4, Hkv=2, Sq=0, Sk=0, D=64, causal=True, seed=1, seqlens=[5, 0, 70])
    (q, k, v), cu2 = W.make_inputs(small)
    assert cu2.tolist() == [0, 5, 5, 75] and q.shape == (75, 4, 64) and k.shape == (75, 2, 64)


@pytest.mark.parametrize("causal,gflop", [(False, 549.8), (True, 274.9)])
def test_dense_workload_flops(causal, gflop):
    """B=4, H=16, S=4096, D=128: 549.8 GFLOP forward, 274.9 causal."""
    assert F.fwd_flops(4, 16, 4096, 4096, 128, causal) / 1e9 == pytest.approx(gflop, abs=0.05)
    assert F.bwd_flops(4, 16, 4096, 4096, 128, causal) == 2.5 * F.fwd_flops(4, 16, 4096, 4096, 128, causal)


@pytest.mark.parametrize("S", [1024, 2048, 4096, 8192, 16384, 32768])
@pytest.mark.parametrize("D", [64, 128])
def test_sweep_flops_rule(S, D):
    """B * S = 32768, H = 16: forward 2,097,152 * S * D FLOP (non-causal)."""
    assert F.fwd_flops(32768 // S, 16, S, S, D, False) == 2_097_152 * S * D


def test_varlen_flops_sum_over_sequences():
    lens = [1, 130, 513]
    want = sum(F.fwd_flops(1, 32, L, L, 128, True) for L in lens)
    assert F.varlen_fwd_flops(lens, 32, 128, True) == want
    assert F.varlen_fwd_flops(lens, 32, 128, False) == 2 * want


def test_training_workload():
    w = W.train(deterministic=True)
    assert (w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.causal) == (2, 16, 16, 8192, 8192, 128, True)
    assert w.extra.get("deterministic") is True
    # backward 1,374 GFLOP (2.5 x the causal forward's 549.8)
    assert F.bwd_flops(2, 16, 8192, 8192, 128, True) / 1e9 == pytest.approx(1374.4, abs=0.1)
