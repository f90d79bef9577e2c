"""Tiled online softmax with eager or lazy rescaling (test infrastructure).

Follows the steps the pages give, in their order, in fp64:

1. Keys are processed block by block; the score matrix is never formed whole
   ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
   Hardware Scaling", fdeinterviews.com summary, opening paragraph: tile queries
   and keys, compute softmax on the fly).
2. A running row maximum and row sum are kept; when the maximum changes, the
   accumulated output is rescaled (same page, bullet "Lazy rescaling", first
   sentence).
3. Lazy variant: the rescale happens only when the new block maximum exceeds
   the running maximum by more than 8 in log2 units (a factor of 256);
   otherwise the stale maximum is kept and the block's weights may reach 2^8.
   A final fix-up divides by the row sum taken at that same stale maximum, so
   the result is exact (same bullet; "FlashAttention-4: matrix throughput
   bottlenecks", lecompute.fr, section "Move some exponential work to different
   units", last paragraph: sums must share one scale, and final normalisation
   cannot repair an overflow -- the threshold keeps every weight <= 256).

Everything is carried in log2 units, x = s * scale * log2(e), as a kernel that
uses exp2 would; the log-sum-exp is returned in natural log.  The routine
exists to pin, independently of any GPU code, that lazy rescaling changes
nothing but the number of rescales.
"""

import numpy as np

LOG2E = 1.0 / np.log(2.0)


def tiled_forward(q, k, v, causal, scale, block_n=128, lazy=True, threshold=8.0):
    """One head, keys in blocks of ``block_n``.

    q: [Sq, D], k: [Sk, D], v: [Sk, Dv] (any float dtype; computed in fp64).
    Returns (o [Sq, Dv], lse [Sq], rescales) where ``rescales`` counts, over
    all rows and blocks, the times a row's accumulated output was multiplied
    by a factor < 1 (the first block of a row is not counted: nothing has
    been accumulated yet).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Sq, Sk = q.shape[0], k.shape[0]
    rows = np.arange(Sq)
    m_run = np.full(Sq, -np.inf)           # running max, log2 units
    l_run = np.zeros(Sq)                    # running row sum at m_run
    acc = np.zeros((Sq, v.shape[1]))        # running unnormalised output
    rescales = 0
    for j0 in range(0, Sk, block_n):
        cols = np.arange(j0, min(j0 + block_n, Sk))
        x = (q @ k[cols].T) * (scale * LOG2E)
        if causal:
            x = np.where(cols[None, :] <= rows[:, None] + (Sk - Sq), x, -np.inf)
        m_blk = x.max(axis=1)
        with np.errstate(invalid="ignore"):  # (-inf) - (-inf) on empty rows
            if lazy:
                grow = (m_blk - m_run > threshold) & np.isfinite(m_blk)
            else:
                grow = m_blk > m_run
            m_new = np.where(grow, m_blk, m_run)
            factor = np.where(grow, np.exp2(m_run - m_new), 1.0)  # 0 when m_run = -inf
        rescales += int(np.count_nonzero(grow & np.isfinite(m_run)))
        m_use = np.where(np.isfinite(m_new), m_new, 0.0)
        p = np.exp2(x - m_use[:, None])     # <= 2^threshold when lazy
        acc = acc * factor[:, None] + p @ v[cols]
        l_run = l_run * factor + p.sum(axis=1)
        m_run = m_new
    has = l_run > 0.0
    o = np.where(has[:, None], acc / np.where(has, l_run, 1.0)[:, None], 0.0)
    lse = np.where(has, (m_run + np.log2(np.where(has, l_run, 1.0))) / LOG2E, -np.inf)
    return o, lse, rescales
