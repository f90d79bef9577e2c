"""The FLOP accounting used by the benchmark reproduces the pages' tile roofline.

The golden values are printed on the pages (cited in the fixture); the
accounting under test is ``exact_attention_78_gb300.flops``.
"""

import json
import os

from exact_attention_78_gb300 import flops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "roofline_tile.json")


def _g():
    with open(GOLDEN) as f:
        return json.load(f)


def test_forward_tile_mma_and_exp_cycles():
    g = _g()
    t, r = g["tile"], g["per_sm_per_clock"]
    f = flops.fwd_flops(1, 1, t["M"], t["N"], t["D"], causal=False)
    assert f / r["bf16_mma_ops"] == g["forward_tile_cycles"]["mma"]
    assert t["M"] * t["N"] / r["exp_ops"] == g["forward_tile_cycles"]["exp"]


def test_backward_tile_is_five_products():
    g = _g()
    t, r = g["tile"], g["per_sm_per_clock"]
    f = flops.bwd_flops(1, 1, t["M"], t["N"], t["D"], causal=False)
    assert f / r["bf16_mma_ops"] == g["backward_tile_cycles"]["mma"]
    assert f == 5 * 2 * t["M"] * t["N"] * t["D"]
    b = g["backward_tile_cycles"]
    assert round(100 * (b["smem"] - b["mma"]) / b["mma"]) == b["smem_over_mma_percent"]
    # the SMEM figure is a whole number of 128-byte transactions per tile step
    assert b["smem"] * r["smem_bytes"] == 425984


def test_causal_halves_and_varlen_sums():
    assert flops.fwd_flops(2, 3, 64, 64, 32, True) * 2 == flops.fwd_flops(2, 3, 64, 64, 32, False)
    assert flops.varlen_fwd_flops([64, 32], 3, 32, False) == (
        flops.fwd_flops(1, 3, 64, 64, 32, False) + flops.fwd_flops(1, 3, 32, 32, 32, False))


def test_lazy_threshold_and_headline():
    g = _g()
    assert 2 ** g["lazy_rescale"]["threshold_log2"] == g["lazy_rescale"]["factor"]
    implied_peak = g["headline"]["fwd_tflops"] / g["headline"]["fraction_of_peak"]
    assert 2200 < implied_peak < 2300     # B200 dense BF16, ~2.27 PFLOP/s
