"""Forward-pass tuning sweep: measures the knobs of ``fa_fwd_tuning`` per
configuration, the data behind the library's per-configuration defaults.

    python -m exact_attention_78_gb300.tune sweep [split_emu|stages|group|all]
        one JSON line per (knobs, configuration): forward TFLOPS over the
        sequence-length sweep (B * S = 32768 tokens, H = 16, D = 64 / 128,
        causal and not), CUDA events, 3 warm-up and 20 timed calls per cell.

    python -m exact_attention_78_gb300.tune profile
        for each table entry (B = 8, H = 16, S = 4096; D, mask, split_p,
        emu_per_16) two untimed calls, then one call inside an NVTX range
        named "prof", so that ``ncu --nvtx --nvtx-include "prof/"`` captures
        exactly one launch per entry.

Inputs are i.i.d. N(0, 1) BF16 drawn on the device (timing only; parity is
the tests' business).  Every call goes through the library's C ABI.
"""

import json
import sys

import torch

from . import binding as fa

SWEEP_S = (1024, 2048, 4096, 8192, 16384, 32768)
TOKENS = 32768
HEADS = 16


class _Inputs:
    """Q, K, V, O of TOKENS x HEADS x D elements, reshaped per configuration."""

    def __init__(self):
        self.buf = {}
        self.lse = torch.empty(TOKENS * HEADS, device="cuda", dtype=torch.float32)

    def get(self, S, D):
        if D not in self.buf:
            n = TOKENS * HEADS * D
            g = torch.Generator(device="cuda")
            g.manual_seed(0)
            self.buf[D] = [torch.randn(n, device="cuda", generator=g).to(torch.bfloat16) for _ in range(3)]
            self.buf[D].append(torch.empty(n, device="cuda", dtype=torch.bfloat16))
        B = TOKENS // S
        q, k, v, o = (t.view(B, S, HEADS, D) for t in self.buf[D])
        return q, k, v, o, self.lse.view(B, HEADS, S)


def fwd_tflops(inputs, S, D, causal, iters=20, **knobs):
    q, k, v, o, lse = inputs.get(S, D)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        fa.fwd(q, k, v, causal=causal, out=o, lse=lse, **knobs)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        fa.fwd(q, k, v, causal=causal, out=o, lse=lse, **knobs)
    e1.record(stream)
    torch.cuda.synchronize()
    if fa.get_device_error() != 0:
        raise RuntimeError("device error during the sweep")
    ms = e0.elapsed_time(e1) / iters
    flops = 4.0 * (TOKENS // S) * HEADS * S * S * D * (0.5 if causal else 1.0)
    return flops / (ms * 1e-3) / 1e12, ms


def sweep(which="all"):
    inputs = _Inputs()

    def emit(tag, S, D, causal, **knobs):
        tf, ms = fwd_tflops(inputs, S, D, causal, **knobs)
        print(json.dumps({"sweep": tag, "S": S, "D": D, "causal": causal, **knobs, "tflops": round(tf, 1),
                          "ms": round(ms, 4)}), flush=True)

    if which in ("all", "split_emu"):
        for D in (128, 64):
            for causal in (False, True):
                for S in SWEEP_S:
                    for split in (0, 1):
                        for emu in (0, 2, 4):
                            emit("split_emu", S, D, causal, split_p=split, emu_per_16=emu)
    if which in ("all", "stages"):
        for D, stages in ((128, (2, 3, 4)), (64, (4, 6, 8, 10))):
            for causal in (False, True):
                for S in (1024, 4096, 16384):
                    for st in stages:
                        emit("stages", S, D, causal, kv_stages=st, split_p=1)
    if which in ("all", "group"):
        for S in (1024, 4096):
            bh = HEADS * TOKENS // S
            for g in sorted({bh, 8, 32}):
                emit("group", S, 128, True, head_group=g)


def profile():
    S, B = 4096, 8
    for D in (128, 64):
        n = B * S * HEADS * D
        g = torch.Generator(device="cuda")
        g.manual_seed(0)
        q, k, v = (torch.randn(n, device="cuda", generator=g).to(torch.bfloat16).view(B, S, HEADS, D)
                   for _ in range(3))
        o = torch.empty_like(q)
        lse = torch.empty(B, HEADS, S, device="cuda")
        for causal in (False, True):
            for split in (0, 1):
                for emu in (0, 2, 4):
                    knobs = dict(split_p=split, emu_per_16=emu)
                    for _ in range(2):
                        fa.fwd(q, k, v, causal=causal, out=o, lse=lse, **knobs)
                    torch.cuda.synchronize()
                    torch.cuda.nvtx.range_push("prof")
                    fa.fwd(q, k, v, causal=causal, out=o, lse=lse, **knobs)
                    torch.cuda.nvtx.range_pop()
                    torch.cuda.synchronize()
                    print(json.dumps({"D": D, "causal": causal, **knobs}), flush=True)
        del q, k, v, o


def main(argv):
    fa.load_library(build_if_missing=True)
    torch.cuda.set_device(0)
    mode = argv[1] if len(argv) > 1 else "sweep"
    if mode == "sweep":
        sweep(argv[2] if len(argv) > 2 else "all")
    elif mode == "profile":
        profile()
    else:
        raise SystemExit("usage: python -m exact_attention_78_gb300.tune [sweep [split_emu|stages|group|all] | profile]")


if __name__ == "__main__":
    main(sys.argv)
