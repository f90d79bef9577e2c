"""CPU oracle for exact attention: TEST INFRASTRUCTURE, not product code.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import anything from this package.  The CUDA library never
routes through it, and it shares no code, header, table or constant with the
CUDA path.

What it computes, and from which passage of the pages:

* ``attention``      -- the plain definition of scaled-dot-product attention in
  fp64: full score matrix, explicit max-subtracted softmax, weights times V,
  per-row log-sum-exp, and the analytic gradients.  Sources:
  "FlashAttention-4: matrix throughput bottlenecks" (lecompute.fr), section
  "Between the matrix products the kernel must produce weights" (scores = Q K^T,
  softmax rows positive and summing to one, second product with V), and
  "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
  Hardware Scaling" (fdeinterviews.com summary), opening paragraph (tiling,
  online softmax, never writing the full matrix) and bullet "Paired-CTA
  backward pass" (the backward produces dQ, dK, dV).
* ``online_softmax`` -- the tiled online-softmax recurrence with eager or lazy
  (threshold 8 in log2 units) rescaling and a final fix-up, from the same
  summary page, bullet "Lazy rescaling", and the lecompute.fr section "Move some
  exponential work to different units" (conditional rescale, final
  normalisation).
* ``exp2_emulation`` -- a float32 model of the software exponential: split x
  into integer and fraction, cubic polynomial on the fraction, add the integer
  to the exponent bits.  Summary page, bullet "Software exponentials".

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
invariants, library routines (scipy) or finite differences; none is "parity
unpinned".
"""

from .attention import (  # noqa: F401
    attention_forward,
    attention_backward,
    head_forward,
    head_backward,
    head_probabilities,
    visible_mask,
)
from .online_softmax import tiled_forward  # noqa: F401
from .exp2_emulation import (  # noqa: F401
    fit_cubic_exp2,
    emulated_exp2_f32,
    bf16_round_bits,
)
