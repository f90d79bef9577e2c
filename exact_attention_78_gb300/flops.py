"""FLOP and byte accounting used by the benchmark and the roofline report.

Conventions (one multiply-add counts as two FLOPs):

* forward FLOPs = 4 * B * Hq * Sq * Sk * D -- the two products Q K^T and P V,
  each 2 * Sq * Sk * D per head -- halved for a causal mask;
* backward FLOPs = 2.5 x forward -- five products of the same size
  (S = Q K^T recomputed, dP = dO V^T, dV = P^T dO, dK = dS^T Q, dQ = dS K).

The per-tile figures these reproduce are the 128 x 128 tile roofline of
"FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
Hardware Scaling" (fdeinterviews.com summary), paragraph on Blackwell's changed
balance: 1,024 tensor-core cycles for the forward tile and 2,560 for the
backward tile at 8,192 FLOP per SM per clock.
"""


def fwd_flops(B, Hq, Sq, Sk, D, causal):
    f = 4.0 * B * Hq * Sq * Sk * D
    return f / 2.0 if causal else f


def bwd_flops(B, Hq, Sq, Sk, D, causal):
    return 2.5 * fwd_flops(B, Hq, Sq, Sk, D, causal)


def varlen_fwd_flops(seqlens, Hq, D, causal):
    """Sum over packed sequences of the dense formula with Sq = Sk = L."""
    return sum(fwd_flops(1, Hq, L, L, D, causal) for L in seqlens)


def fwd_bytes(B, Hq, Hkv, Sq, Sk, D, elem=2):
    """Algorithmic HBM bytes of one forward call: read Q, K, V; write O, LSE."""
    return elem * B * D * (2 * Sq * Hq + 2 * Sk * Hkv) + 4 * B * Hq * Sq


def bwd_bytes(B, Hq, Hkv, Sq, Sk, D, elem=2):
    """Algorithmic HBM bytes of one backward call: read Q, K, V, O, dO, LSE;
    write dQ, dK, dV.  The fp32 dQ accumulator is scratch and not counted."""
    q_side = elem * B * Sq * Hq * D
    kv_side = elem * B * Sk * Hkv * D
    return 4 * q_side + 4 * kv_side + 4 * B * Hq * Sq
