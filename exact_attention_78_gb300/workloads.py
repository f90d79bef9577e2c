"""Seeded synthetic inputs and the named workload shapes.

This module only draws random numbers and describes shapes; it holds none of
the attention arithmetic.  Tests, the oracle checks and ``bench.py`` all take
their inputs from here, so the GPU path and the CPU oracle see the very same
BF16 values.

Inputs are i.i.d. N(0, 1) drawn in fp32 on the CPU from
``torch.Generator().manual_seed(seed)`` and rounded to BF16, in the layouts the
library uses: dense Q/dO [B, Sq, Hq, D], K/V [B, Sk, Hkv, D]; packed
variable-length [total, H, D] with int32 ``cu_seqlens`` of length B + 1.
"""

from dataclasses import dataclass, field
from typing import List, Optional

import torch


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    causal: bool
    seed: int = 0
    q_scale: float = 1.0          # multiply Q after rounding (stress: 4 -> logit std ~16)
    seqlens: Optional[List[int]] = None   # packed variable-length batch when set
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return self.D ** -0.5

    @property
    def packed(self) -> bool:
        return self.seqlens is not None

    def describe(self) -> dict:
        d = {"workload": self.name, "B": self.B, "Hq": self.Hq, "Hkv": self.Hkv,
             "Sq": self.Sq, "Sk": self.Sk, "D": self.D, "causal": self.causal,
             "seed": self.seed}
        if self.q_scale != 1.0:
            d["q_scale"] = self.q_scale
        if self.packed:
            d["total_tokens"] = int(sum(self.seqlens))
        return d


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def varlen_lengths(n: int = 64, lo: int = 128, hi: int = 8192, seed: int = 2) -> List[int]:
    """Sequence lengths drawn uniformly from [lo, hi] (inclusive), seeded."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=_gen(seed))]


def cu_seqlens_of(lengths: List[int]) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def randn_bf16(shape, seed: int) -> torch.Tensor:
    return torch.randn(*shape, generator=_gen(seed), dtype=torch.float32).to(torch.bfloat16)


def make_inputs(w: Workload, with_grad: bool = False):
    """Host BF16 tensors (q, k, v[, do]) and cu_seqlens (or None) for ``w``.

    Each tensor has its own seed derived from ``w.seed`` so that changing one
    shape does not change the others' values.
    """
    if w.packed:
        total = int(sum(w.seqlens))
        qs, ks = (total, w.Hq, w.D), (total, w.Hkv, w.D)
        cu = cu_seqlens_of(w.seqlens)
    else:
        qs, ks = (w.B, w.Sq, w.Hq, w.D), (w.B, w.Sk, w.Hkv, w.D)
        cu = None
    base = 1000 * w.seed
    q = randn_bf16(qs, base + 1)
    if w.q_scale != 1.0:
        q = (q.float() * w.q_scale).to(torch.bfloat16)
    k = randn_bf16(ks, base + 2)
    v = randn_bf16(ks, base + 3)
    out = [q, k, v]
    if with_grad:
        out.append(randn_bf16(qs, base + 4))
    return tuple(out), cu


def tiny(causal: bool = False) -> Workload:
    return Workload("tiny", B=1, Hq=2, Hkv=2, Sq=256, Sk=256, D=64, causal=causal)


def dense(causal: bool = False, stress: bool = False) -> Workload:
    return Workload("dense_stress" if stress else "dense", B=4, Hq=16, Hkv=16, Sq=4096,
                    Sk=4096, D=128, causal=causal, seed=1 if stress else 0,
                    q_scale=4.0 if stress else 1.0)


def sweep(S: int, D: int, causal: bool) -> Workload:
    return Workload(f"sweep_S{S}_D{D}", B=32768 // S, Hq=16, Hkv=16, Sq=S, Sk=S, D=D,
                    causal=causal)


def varlen_gqa() -> Workload:
    lens = varlen_lengths()
    return Workload("varlen_gqa", B=len(lens), Hq=32, Hkv=8, Sq=max(lens), Sk=max(lens),
                    D=128, causal=True, seqlens=lens)


def train(deterministic: bool = False) -> Workload:
    return Workload("train", B=2, Hq=16, Hkv=16, Sq=8192, Sk=8192, D=128, causal=True,
                    extra={"deterministic": deterministic})


SWEEP_S = (1024, 2048, 4096, 8192, 16384, 32768)
