"""Forward-pass parity on the GPU: the CUDA library (through its C ABI)
against the fp64 oracle on the same seeded BF16 inputs.

Small cases are compared element by element over whole tensors; they span
several 128-row tiles and 128-key blocks with ragged tails.  Full-size
workloads are compared on sampled rows computed one by one by the oracle.
"""

import numpy as np
import pytest
import torch

from exact_attention_78_gb300 import workloads as W

import oracle
from parity import LSE_ATOL, O_ATOL, check_forward_full, check_forward_sampled, f64, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_78_gb300 as fa_mod
    fa_mod.load_library(build_if_missing=True)
    return fa_mod


def _dense(B, Hq, Hkv, Sq, Sk, D, seed=0, q_scale=1.0):
    w = W.Workload("case", B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, D=D, causal=False, seed=seed, q_scale=q_scale)
    (q, k, v), _ = W.make_inputs(w)
    return q, k, v


def _run(fa, q, k, v, causal, cu=None, **kw):
    dev = [t.cuda() for t in (q, k, v)]
    cu_d = None if cu is None else cu.cuda()
    o, lse = fa.fwd(*dev, causal=causal, cu_seqlens=cu_d, **kw)
    assert fa.get_device_error() == 0
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_config(fa, causal):
    w = W.tiny(causal)
    (q, k, v), _ = W.make_inputs(w)
    o, lse = _run(fa, q, k, v, causal)
    check_forward_full(o, lse, q, k, v, causal, w.scale)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk", [
    (2, 3, 3, 700, 700),     # several tiles, ragged tail in both rows and keys
    (1, 4, 2, 384, 384),     # grouped-query heads, odd number of 128-row tiles
    (2, 2, 1, 129, 257),     # Sq < Sk: causal diagonal shifted right
    (1, 2, 2, 520, 300),     # Sq > Sk: causal leaves the first rows fully masked
    (1, 1, 1, 1, 1),         # one query, one key
    (1, 2, 2, 256, 1),       # a single key
])
def test_small_shapes_full_compare(fa, D, causal, B, Hq, Hkv, Sq, Sk):
    q, k, v = _dense(B, Hq, Hkv, Sq, Sk, D)
    o, lse = _run(fa, q, k, v, causal)
    check_forward_full(o, lse, q, k, v, causal, D ** -0.5)


def test_zero_queries_give_mean_of_visible_values(fa):
    """Closed form: Q = 0 -> O_i = mean of visible V rows, LSE_i = ln(#visible)."""
    q, k, v = _dense(1, 2, 2, 300, 300, 128)
    q = torch.zeros_like(q)
    o, lse = _run(fa, q, k, v, True)
    vf = f64(v)[0, :, 0]
    for i in (0, 1, 127, 128, 299):
        np.testing.assert_allclose(f64(o)[0, i, 0], vf[: i + 1].mean(axis=0), atol=O_ATOL)
        assert abs(float(lse[0, 0, i]) - np.log(i + 1)) <= LSE_ATOL


def test_causal_first_row_equals_first_value(fa):
    q, k, v = _dense(2, 2, 2, 256, 256, 64)
    o, _ = _run(fa, q, k, v, True)
    np.testing.assert_allclose(f64(o)[:, 0], f64(v)[:, 0], atol=8e-3)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_lazy_equals_eager_under_stress(fa, D, causal):
    """Q x 4 (logit std ~16): running maxima keep growing.  Lazy rescaling
    (threshold 8) is exact ("FlashAttention-4: Algorithm and Kernel
    Pipelining Co-Design ...", bullet "Lazy rescaling": skipping the rescale
    leaves the result unchanged), so it may differ from eager rescaling
    (threshold 0) only by rounding: the weights are rounded to BF16 at a
    different scale, and O is rounded to BF16 at the end.

    Pinned here, on whole tensors:
      * lazy and eager O differ by at most 2.5e-3 relative Frobenius (BF16
        output rounding alone is ~1.1e-3; measured 1.3-1.7e-3) -- six times
        tighter than the 1.5e-2 max-abs parity tolerance;
      * at least 90% of lazy O elements are within one BF16 ulp of eager O
        (measured 92-96%);
      * lazy is as accurate as eager against the fp64 oracle (relative
        Frobenius within 15%; measured ratio 1.05-1.08);
      * LSE agrees to 1e-5 (measured 1.9e-6).
    Both runs use the hardware exponential only, so that the comparison
    isolates the rescaling rule (the FMA polynomial's own error depends on
    its argument, which differs between the two rules; its accuracy has its
    own tests)."""
    q, k, v = _dense(1, 4, 4, 1024, 1024, D, seed=1, q_scale=4.0)
    o_l, lse_l = _run(fa, q, k, v, causal, rescale_threshold=8.0, emu_per_16=0)
    o_e, lse_e = _run(fa, q, k, v, causal, rescale_threshold=0.0, emu_per_16=0)
    check_forward_full(o_l, lse_l, q, k, v, causal, D ** -0.5)
    check_forward_full(o_e, lse_e, q, k, v, causal, D ** -0.5)
    o_ref, _ = oracle.attention_forward(f64(q), f64(k), f64(v), causal, D ** -0.5)
    assert rel_fro(f64(o_l), f64(o_e)) <= 2.5e-3
    ulps = (o_l.view(torch.int16).long() - o_e.view(torch.int16).long()).abs()
    assert float((ulps <= 1).float().mean()) >= 0.90
    assert rel_fro(f64(o_l), o_ref) <= 1.15 * rel_fro(f64(o_e), o_ref)
    assert float((lse_l - lse_e).abs().max()) <= 1e-5


@pytest.mark.parametrize("emu", [0, 2, 3, 4])
def test_exp2_emulation_fraction_keeps_parity(fa, emu):
    q, k, v = _dense(2, 2, 2, 640, 640, 128, seed=3)
    o, lse = _run(fa, q, k, v, True, emu_per_16=emu)
    check_forward_full(o, lse, q, k, v, True, 128 ** -0.5)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_split_p_and_ring_depth_change_no_bits(fa, D, causal):
    """P handed to the tensor cores in two halves (split_p = 1) or at once,
    and every K/V ring depth: the same products are issued in the same order,
    only their timing changes, so O and LSE are bitwise identical -- and
    match the oracle."""
    q, k, v = _dense(2, 3, 3, 700, 700, D, seed=5)
    base_o, base_l = _run(fa, q, k, v, causal, split_p=0)
    check_forward_full(base_o, base_l, q, k, v, causal, D ** -0.5)
    max_stages = 4 if D == 128 else 10
    for split in (0, 1):
        for stages in (2, 3, max_stages):
            o, lse = _run(fa, q, k, v, causal, split_p=split, kv_stages=stages)
            assert torch.equal(o.view(torch.int16), base_o.view(torch.int16)), (split, stages)
            assert torch.equal(lse, base_l), (split, stages)


@pytest.mark.parametrize("D", [64, 128])
def test_causal_head_groups_change_no_bits(fa, D):
    """Longest-first order within groups of 1, 4 or all (batch, head) pairs:
    each work unit computes the same thing wherever it runs."""
    q, k, v = _dense(2, 3, 3, 900, 900, D, seed=6)
    base_o, base_l = _run(fa, q, k, v, True, head_group=6)
    check_forward_full(base_o, base_l, q, k, v, True, D ** -0.5)
    for g in (1, 4, 100):
        o, lse = _run(fa, q, k, v, True, head_group=g)
        assert torch.equal(o.view(torch.int16), base_o.view(torch.int16)), g
        assert torch.equal(lse, base_l), g


@pytest.mark.parametrize("split_p", [0, 1])
def test_split_p_packed_lengths(fa, split_p):
    lens = [1, 130, 0, 513, 256, 77, 1000, 128, 129]
    cu = W.cu_seqlens_of(lens)
    T = int(cu[-1])
    q, k, v = W.randn_bf16((T, 4, 128), 31), W.randn_bf16((T, 2, 128), 32), W.randn_bf16((T, 2, 128), 33)
    for causal in (False, True):
        o, lse = _run(fa, q, k, v, causal, cu=cu, split_p=split_p)
        check_forward_full(o, lse, q, k, v, causal, 128 ** -0.5, cu=cu)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_variable_lengths(fa, causal):
    lens = [1, 130, 0, 513, 256, 77, 1000]
    cu = W.cu_seqlens_of(lens)
    T = int(cu[-1])
    q, k, v = W.randn_bf16((T, 4, 128), 11), W.randn_bf16((T, 2, 128), 12), W.randn_bf16((T, 2, 128), 13)
    o, lse = _run(fa, q, k, v, causal, cu=cu)
    check_forward_full(o, lse, q, k, v, causal, 128 ** -0.5, cu=cu)


def test_bad_offsets_are_reported_not_computed(fa):
    """cu_seqlens whose last entry differs from the row count: the kernel
    records FA_ERR_INVALID_ARG and writes nothing."""
    cu = W.cu_seqlens_of([100, 200]).cuda()
    cu[-1] = 250
    q = W.randn_bf16((300, 2, 64), 1).cuda()
    o = torch.full_like(q, 7.0)
    fa.fwd(q, q, q, causal=True, cu_seqlens=cu, out=o)
    assert fa.get_device_error() == fa.binding.FA_ERR_INVALID_ARG
    assert fa.get_device_error() == 0
    assert bool((o == 7.0).all())


def test_bounded_wait_reports_timeout_and_context_survives(fa):
    fa.wait_timeout_probe(20_000_000)          # 20 ms bound, nothing arrives
    assert fa.get_device_error() == fa.binding.FA_ERR_TIMEOUT
    assert fa.get_device_error() == 0
    q, k, v = _dense(1, 1, 1, 128, 128, 64)
    o, lse = _run(fa, q, k, v, False)
    check_forward_full(o, lse, q, k, v, False, 64 ** -0.5)


def test_exp2_emulation_within_one_bf16_ulp_of_hardware(fa):
    """The page's claim: after rounding to BF16 the FMA polynomial agrees with
    the hardware exponential within one ulp on at least 99% of inputs."""
    x = torch.cat([torch.linspace(-126.0, 8.0, 1 << 24),
                   torch.rand(1 << 20, generator=torch.Generator().manual_seed(5)) * 134.0 - 126.0])
    ye, yh = fa.exp2_probe(x.cuda())
    be = ye.cpu().to(torch.bfloat16).view(torch.int16).numpy().astype(np.int64)
    bh = yh.cpu().to(torch.bfloat16).view(torch.int16).numpy().astype(np.int64)
    ulp = np.abs(be - bh)
    assert np.mean(ulp <= 1) >= 0.99
    assert ulp.max() <= 2
    rel = np.abs(ye.cpu().double().numpy() / np.exp2(x.double().numpy()) - 1.0)
    assert rel.max() < 2.5e-4
    # integers are exact; a masked score (-inf) gives exactly zero
    n = torch.arange(-126, 9, dtype=torch.float32)
    ye_n, _ = fa.exp2_probe(n.cuda())
    assert torch.equal(ye_n.cpu(), torch.exp2(n))
    ye_m, yh_m = fa.exp2_probe(torch.tensor([-float("inf")], device="cuda"))
    assert float(ye_m) == 0.0 and float(yh_m) == 0.0


# ---------------------------------------------------------------- full size --

def _sampled(fa, w, heads, rows):
    """Full-size call in the benchmark's launch configuration.  O and LSE
    start as NaN, so the finiteness checks show that every row of every
    work unit was written (a unit skipped or dealt to no CTA would leave
    NaN); sampled rows are then compared with the oracle."""
    (q, k, v), cu = W.make_inputs(w)
    dev = [t.cuda() for t in (q, k, v)]
    cu_d = None if cu is None else cu.cuda()
    o_d = torch.full_like(dev[0], float("nan"))
    lse_shape = (w.Hq, q.shape[0]) if cu is not None else (w.B, w.Hq, w.Sq)
    lse_d = torch.full(lse_shape, float("nan"), device="cuda", dtype=torch.float32)
    o, lse = fa.fwd(*dev, causal=w.causal, cu_seqlens=cu_d, out=o_d, lse=lse_d)
    assert fa.get_device_error() == 0
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all()
    assert bool(torch.isfinite(lse).all())
    return check_forward_sampled(o, lse, q, k, v, w.causal, w.scale, heads, rows,
                                 cu_host=None if cu is None else cu.numpy())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("stress", [False, True])
def test_dense_config_sampled(fa, causal, stress):
    w = W.dense(causal=causal, stress=stress)
    rows = [0, 1, 127, 128, 255, 256, 1000, 2047, 2048, 3071, 4094, 4095]
    _sampled(fa, w, [(0, 0), (1, 7), (3, 15)], rows)


@pytest.mark.parametrize("S", list(W.SWEEP_S))
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_sweep_config_sampled(fa, S, D, causal):
    w = W.sweep(S, D, causal)
    rows = [0, 129, S // 2 - 1, S // 2, S - 257, S - 1]
    _sampled(fa, w, [(0, 0), (w.B - 1, 15)], rows)


def test_varlen_gqa_config_sampled(fa):
    w = W.varlen_gqa()
    rows = [0, 1, 255, 256, 1000, 4000, 8191]
    _sampled(fa, w, [(0, 0), (5, 31), (17, 9), (63, 20)], rows)
