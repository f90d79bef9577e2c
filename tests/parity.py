"""Helpers shared by the GPU parity tests: run the library, run the oracle on
the same BF16 inputs, compare with the tolerances the product promises.

Tolerances (against the fp64 oracle on the same BF16 inputs):
  forward  O max-abs <= 1.5e-2, LSE max-abs <= 1e-3;
  backward dQ, dK, dV relative Frobenius error <= 1e-2.
"""

import numpy as np
import torch

import oracle

O_ATOL = 1.5e-2
LSE_ATOL = 1e-3
GRAD_RTOL = 1e-2


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_forward_full(o, lse, q, k, v, causal, scale, cu=None):
    """Whole-tensor comparison (small cases)."""
    cu_np = None if cu is None else cu.cpu().numpy()
    o_ref, lse_ref = oracle.attention_forward(f64(q), f64(k), f64(v), causal, scale, cu_seqlens=cu_np)
    o_gpu, lse_gpu = f64(o), f64(lse)
    assert np.all(np.isfinite(o_gpu))
    err_o = np.max(np.abs(o_gpu - o_ref)) if o_ref.size else 0.0
    fin = np.isfinite(lse_ref)
    np.testing.assert_array_equal(np.isfinite(lse_gpu), fin)
    np.testing.assert_array_equal(lse_gpu[~fin], lse_ref[~fin])
    err_l = np.max(np.abs(lse_gpu[fin] - lse_ref[fin])) if fin.any() else 0.0
    assert err_o <= O_ATOL, err_o
    assert err_l <= LSE_ATOL, err_l
    return err_o, err_l


def check_forward_sampled(o, lse, q, k, v, causal, scale, heads, rows, cu_host=None):
    """Oracle rows computed one by one for the (batch-or-sequence, head) pairs
    in ``heads`` and the query rows ``rows`` (clipped to each sequence)."""
    Hq, Hkv = q.shape[-2], k.shape[-2]
    g = Hq // Hkv
    worst_o = worst_l = 0.0
    for b, h in heads:
        if cu_host is None:
            qh, kh, vh = q[b, :, h], k[b, :, h // g], v[b, :, h // g]
            oh, lh = o[b, :, h], lse[b, h]
        else:
            s0, s1 = int(cu_host[b]), int(cu_host[b + 1])
            qh, kh, vh = q[s0:s1, h], k[s0:s1, h // g], v[s0:s1, h // g]
            oh, lh = o[s0:s1, h], lse[h, s0:s1]
        r = np.array(sorted({int(x) for x in rows if 0 <= x < qh.shape[0]}), dtype=np.int64)
        if r.size == 0:
            continue
        o_ref, l_ref = oracle.head_forward(f64(qh), f64(kh), f64(vh), causal, scale, rows=r)
        o_g, l_g = f64(oh[torch.from_numpy(r)]), f64(lh[torch.from_numpy(r)])
        worst_o = max(worst_o, float(np.max(np.abs(o_g - o_ref))))
        worst_l = max(worst_l, float(np.max(np.abs(l_g - l_ref))))
    assert worst_o <= O_ATOL, worst_o
    assert worst_l <= LSE_ATOL, worst_l
    return worst_o, worst_l


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))
