"""Plain fp64 exact attention and its analytic gradients (test infrastructure).

This is the definition the GPU kernels must reproduce, written out directly:
the whole score matrix of a head is formed, the softmax subtracts the row
maximum explicitly, and nothing is tiled, fused or reordered.

Definition, from "FlashAttention-4: matrix throughput bottlenecks"
(lecompute.fr), section "Between the matrix products the kernel must produce
weights": scores compare queries with keys by a matrix product, softmax turns
each row of scores into positive weights that sum to one, and a second matrix
product combines the values with those weights.  The scaled form
O = softmax(scale * Q K^T [+ causal mask]) V with its per-row log-sum-exp, and
the backward pass producing dQ, dK and dV, follow "FlashAttention-4: Algorithm
and Kernel Pipelining Co-Design for Asymmetric Hardware Scaling"
(fdeinterviews.com summary), opening paragraph and bullet "Paired-CTA backward
pass".

Readings where the pages are silent (each is listed in the design notes):

* The log-sum-exp is in natural log: lse_i = m_i + ln(sum_j exp(s_ij - m_i)).
* The causal mask is aligned bottom-right: query i sees key j iff
  j <= i + (Sk - Sq).  With Sq == Sk this is the usual j <= i.
* A row that sees no key has O = 0 and lse = -inf, and zero gradients.
* Grouped-query heads: query head h reads key/value head h // (Hq // Hkv).
* Layouts: dense Q/O are [B, Sq, Hq, D] and K/V are [B, Sk, Hkv, D], lse is
  [B, Hq, Sq]; packed variable-length inputs are [total, H, D] with
  ``cu_seqlens`` of length B+1 and lse [Hq, total].
* The backward uses Delta_i = sum_d dO_id * O_id with the fp64 O recomputed
  here (the analytic gradient of L = sum(dO * O)).
"""

import numpy as np


def visible_mask(rows, Sq, Sk, causal):
    """Boolean [len(rows), Sk]: which keys each query row may attend to."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.arange(Sk, dtype=np.int64)
    if not causal:
        return np.ones((rows.size, Sk), dtype=bool)
    return cols[None, :] <= rows[:, None] + (Sk - Sq)


def _scores(q, k, causal, scale, rows):
    """Masked scaled scores s_ij = scale * q_i . k_j (-inf where not visible)."""
    Sq, Sk = q.shape[0], k.shape[0]
    if rows is None:
        rows = np.arange(Sq)
    rows = np.asarray(rows, dtype=np.int64)
    s = scale * (q[rows].astype(np.float64) @ k.astype(np.float64).T)
    return np.where(visible_mask(rows, Sq, Sk, causal), s, -np.inf), rows


def head_probabilities(q, k, causal, scale, rows=None):
    """Softmax weights of one head, with the row maximum subtracted.

    q: [Sq, D], k: [Sk, D].  Returns (p [R, Sk], lse [R]) for the query rows
    ``rows`` (all rows by default).  p rows sum to one; p is zero where masked.
    """
    s, _ = _scores(q, k, causal, scale, rows)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 on masked keys
    l = e.sum(axis=1)
    has = l > 0.0
    p = np.where(has[:, None], e / np.where(has, l, 1.0)[:, None], 0.0)
    lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    return p, lse


def head_forward(q, k, v, causal, scale, rows=None):
    """One head: O rows [R, Dv] and lse [R] (natural log)."""
    p, lse = head_probabilities(q, k, causal, scale, rows)
    return p @ v.astype(np.float64), lse


def head_backward(q, k, v, do, causal, scale):
    """Gradients of L = sum(dO * O) for one query head against one K/V head.

    Returns (dq [Sq, D], dk [Sk, D], dv [Sk, Dv]) in fp64.  With
    P the softmax weights, O = P V:  dV = P^T dO;  dP = dO V^T;
    Delta_i = sum_d dO_id O_id;  dS = P * (dP - Delta);  dQ = scale dS K;
    dK = scale dS^T Q.
    """
    q64, k64, v64, do64 = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    p, _ = head_probabilities(q64, k64, causal, scale)
    o = p @ v64
    dv = p.T @ do64
    dp = do64 @ v64.T
    delta = np.sum(do64 * o, axis=1)
    ds = p * (dp - delta[:, None])
    dq = scale * (ds @ k64)
    dk = scale * (ds.T @ q64)
    return dq, dk, dv


def _slices(B, S, cu_seqlens):
    """(batch index, token slice) per sequence for dense or packed layouts."""
    if cu_seqlens is None:
        return [(b, slice(None)) for b in range(B)]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return [(b, slice(int(cu[b]), int(cu[b + 1]))) for b in range(cu.size - 1)]


def _head_views(x, b, sl, h, packed):
    return x[sl, h, :] if packed else x[b, :, h, :]


def attention_forward(q, k, v, causal, scale, cu_seqlens=None):
    """Whole-tensor forward.  Returns (o fp64 in q's layout, lse fp64).

    Dense: q [B, Sq, Hq, D], k/v [B, Sk, Hkv, D] -> lse [B, Hq, Sq].
    Packed: q [total, Hq, D], k/v [total, Hkv, D], cu_seqlens [B+1]
    -> lse [Hq, total].
    """
    packed = cu_seqlens is not None
    Hq = q.shape[-2]
    Hkv = k.shape[-2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    g = Hq // Hkv
    o = np.zeros(q.shape[:-1] + (v.shape[-1],), dtype=np.float64)
    if packed:
        lse = np.full((Hq, q.shape[0]), -np.inf)
    else:
        lse = np.full((q.shape[0], Hq, q.shape[1]), -np.inf)
    for b, sl in _slices(q.shape[0], None, cu_seqlens):
        for h in range(Hq):
            qh = _head_views(q, b, sl, h, packed)
            kh = _head_views(k, b, sl, h // g, packed)
            vh = _head_views(v, b, sl, h // g, packed)
            oh, lh = head_forward(qh, kh, vh, causal, scale)
            if packed:
                o[sl, h, :] = oh
                lse[h, sl] = lh
            else:
                o[b, :, h, :] = oh
                lse[b, h, :] = lh
    return o, lse


def attention_backward(q, k, v, do, causal, scale, cu_seqlens=None):
    """Whole-tensor backward.  Returns (dq, dk, dv) fp64 in the input layouts.

    dK and dV of a key/value head sum the contributions of all query heads of
    its group.
    """
    packed = cu_seqlens is not None
    Hq = q.shape[-2]
    Hkv = k.shape[-2]
    g = Hq // Hkv
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    for b, sl in _slices(q.shape[0], None, cu_seqlens):
        for h in range(Hq):
            hk = h // g
            qh = _head_views(q, b, sl, h, packed)
            kh = _head_views(k, b, sl, hk, packed)
            vh = _head_views(v, b, sl, hk, packed)
            doh = _head_views(do, b, sl, h, packed)
            gq, gk, gv = head_backward(qh, kh, vh, doh, causal, scale)
            if packed:
                dq[sl, h, :] = gq
                dk[sl, hk, :] += gk
                dv[sl, hk, :] += gv
            else:
                dq[b, :, h, :] = gq
                dk[b, :, hk, :] += gk
                dv[b, :, hk, :] += gv
    return dq, dk, dv
