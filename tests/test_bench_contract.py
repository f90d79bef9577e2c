"""The benchmark's reference arm (the CPU oracle) runs without a GPU, so its
JSON line can be checked here against the benchmark contract: one line,
the contract's keys, and the values the driver computes its ratio from.
Also the pieces of the GPU arm that need no device: the per-step FLOP
count and the traffic lookup's source hashing."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_attention_78_gb300 import workloads as W  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "1", "--B", "1", "--H", "2", "--S", "256", "--D", "64"],
                         capture_output=True, text=True, timeout=300, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["unit"] == "TFLOPS"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "dense" and d["config"]["D"] == 64


def test_step_flops_follow_the_counting_rule():
    """Forward 4*B*Hq*Sq*Sk*D (half under a causal mask), backward 2.5x."""
    w = W.Workload("dense", B=4, Hq=16, Hkv=16, Sq=4096, Sk=4096, D=128, causal=False)
    fwd = 4 * 4 * 16 * 4096 * 4096 * 128
    assert bench.fwd_flops_of(w) == fwd
    assert bench.step_flops(w, True) == 3.5 * fwd
    wc = W.Workload("dense_causal", B=4, Hq=16, Hkv=16, Sq=4096, Sk=4096, D=128, causal=True)
    assert bench.fwd_flops_of(wc) == fwd / 2


def test_traffic_record_ignores_comments_only():
    src = "int a; // note\n/* block\n comment */ int  b;\n"
    assert bench.code_only(src) == bench.code_only("int a;\nint b;")
    assert bench.code_only(src) != bench.code_only("int a; int c;")
