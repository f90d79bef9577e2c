"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic BF16
input: the forward call (O, LSE) followed, once built, by the backward call
(dQ, dK, dV) on the same tensors.  Default workload: dense B=4, H=16,
S=4096, D=128 (non-causal; --causal for the masked variant).

Prints ONE JSON line (rank 0).  `value` is whole-job TFLOPS
(forward 4*B*Hq*Sq*Sk*D, halved when causal; backward 2.5x that) over all
ranks, timed with CUDA events on the launching stream with inputs resident in
HBM; `e2e` times the same steps through the public API from pinned host
buffers, including host->device and device->host copies.

--impl reference times the CPU oracle (fp64 numpy) on a bounded sample of the
same workload instead: the pages ship no code to run, so the oracle is the
reference arm.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from exact_attention_78_gb300 import flops as F  # noqa: E402
from exact_attention_78_gb300 import replicas  # noqa: E402
from exact_attention_78_gb300 import workloads as W  # noqa: E402

METRIC = "attention fwd/bwd TFLOPS on 1 GB300, BF16 D=128 S=1K–32K; % of BF16 peak"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="dense", choices=["dense", "train", "varlen"],
                    help="dense: B,H,S,D below; train: B=2 H=16 S=8192 D=128 causal; "
                         "varlen: 64 packed sequences, Hq=32 Hkv=8, D=128, causal")
    ap.add_argument("--deterministic", action="store_true", help="deterministic dQ order in the backward")
    ap.add_argument("--paired", action="store_true",
                    help="backward main kernel on CTA pairs (paired tcgen05 MMAs) instead of single CTAs")
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--fwd-only", action="store_true", help="time the forward call alone")
    ap.add_argument("--B", type=int, default=4)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--S", type=int, default=4096)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--emu", type=int, default=None, help="exp2 emulation: entries of every 16 on FMA")
    ap.add_argument("--fwd-tune", default="",
                    help="forward knobs as name=value,... (split_p, kv_stages, head_group); "
                         "default: the library's per-configuration choice")
    ap.add_argument("--bwd-tune", default="",
                    help="backward knobs as name=value,... (schedule, head_group, reverse_blocks, scores_first); "
                         "default: the library's per-call choice")
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="repeat the block of --steps timed steps until the blocks together last this long "
                         "(so that clock samples see the GPU under load); the median block is reported")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline sample")
    return ap.parse_args()


def dist_env():
    return replicas.rank_env()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                      "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                     timeout=5).stdout.strip()
                if out:
                    self.samples.append([x.strip() for x in out.split(",")])
            except Exception:
                pass
            self._stop.wait(0.1)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._t.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [v for v in (num(s[1]) for s in self.samples) if v is not None]
        mx = [v for v in (num(s[2]) for s in self.samples) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if len(s) > 4 + i and s[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


def code_only(src):
    """Source text with comments and whitespace runs removed, so that a
    comment edit does not retire a traffic record taken on the same code."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def measured_traffic(kernel, w):
    """DRAM bytes per launch of `kernel` from the committed ncu record, if it
    was taken on this workload and the kernel sources are unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        recs = json.load(f).get(kernel)
    if not recs or w.packed:
        return None
    if isinstance(recs, dict):
        recs = [recs]
    sha = source_sha(kernel)
    want = "dense B=%d Hq=Hkv=%d S=%d D=%d %s" % (w.B, w.Hq, w.Sq, w.D, "causal" if w.causal else "non-causal")
    for rec in recs:
        if rec["source_sha"] == sha and rec["workload"] == want:
            return rec["dram_read_bytes"] + rec["dram_write_bytes"]
    return None


# The sources each kernel is compiled from (a traffic record holds only while
# they are unchanged, comments and whitespace aside).
KERNEL_SOURCES = {
    "bwd_kernel": ["fa_bwd.cu", "ptx.cuh", "softmax_math.cuh", "exp2_poly.h", "fa_internal.h"],
    "bwd_pair_kernel": ["fa_bwd_pair.cu", "ptx.cuh", "softmax_math.cuh", "exp2_poly.h", "fa_internal.h"],
    "fwd_kernel": ["fa_fwd.cu", "q_sched.cuh", "ptx.cuh", "softmax_math.cuh", "exp2_poly.h", "fa_internal.h"],
    "dq_kernel": ["fa_bwd_dq.cu", "q_sched.cuh", "ptx.cuh", "softmax_math.cuh", "exp2_poly.h", "fa_internal.h"],
}


def source_sha(kernel):
    import hashlib
    csrc = os.path.join(ROOT, "exact_attention_78_gb300", "csrc")
    m = hashlib.sha256()
    for fn in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, fn)) as f:
            m.update(code_only(f.read()).encode())
    return m.hexdigest()[:16]


def workload(args):
    if args.workload == "train":
        return W.train(args.deterministic)
    if args.workload == "varlen":
        return W.varlen_gqa()
    return W.Workload("dense_causal" if args.causal else "dense", B=args.B, Hq=args.H, Hkv=args.H, Sq=args.S,
                      Sk=args.S, D=args.D, causal=args.causal)


def fwd_flops_of(w):
    if w.packed:
        return F.varlen_fwd_flops(w.seqlens, w.Hq, w.D, w.causal)
    return F.fwd_flops(w.B, w.Hq, w.Sq, w.Sk, w.D, w.causal)


def step_flops(w, with_bwd):
    return fwd_flops_of(w) * (3.5 if with_bwd else 1.0)


# --------------------------------------------------------------- oracle arm --

def oracle_sample(w, seconds=15.0, with_bwd=True):
    """Times the fp64 oracle on whole heads of the workload until about
    `seconds` have passed (at least one head); returns (TFLOPS, description,
    threads, seconds per head)."""
    import oracle
    one = W.Workload("s", B=1, Hq=1, Hkv=1, Sq=w.Sq, Sk=w.Sk, D=w.D, causal=w.causal)
    (q, k, v, do), _ = W.make_inputs(one, with_grad=True)

    def f64(t):
        return t.float().numpy().astype(np.float64)[0, :, 0]

    qh, kh, vh, doh = f64(q), f64(k), f64(v), f64(do)
    per_head = F.fwd_flops(1, 1, w.Sq, w.Sk, w.D, w.causal)
    if with_bwd:
        per_head += F.bwd_flops(1, 1, w.Sq, w.Sk, w.D, w.causal)
    t0 = time.perf_counter()
    heads = 0
    while True:
        oracle.head_forward(qh, kh, vh, w.causal, w.scale)
        if with_bwd:
            oracle.head_backward(qh, kh, vh, doh, w.causal, w.scale)
        heads += 1
        if time.perf_counter() - t0 >= seconds or heads >= w.B * w.Hq:
            break
    dt = time.perf_counter() - t0
    try:
        threads = len(os.sched_getaffinity(0))
    except AttributeError:
        threads = os.cpu_count()
    desc = "%d of %d (b,h) heads, %s, S=%d D=%d, numpy fp64 (BLAS threads = affinity)" % (
        heads, w.B * w.Hq, "fwd+bwd" if with_bwd else "fwd", w.Sq, w.D)
    return heads * per_head / dt / 1e12, desc, threads, dt / heads


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    w = workload(args)
    with_bwd = not args.fwd_only
    for _ in range(args.warmup):
        oracle_sample(w, seconds=0.0, with_bwd=with_bwd)
    vals, per_head = [], []
    desc = threads = None
    for _ in range(args.steps):
        v, desc, threads, sph = oracle_sample(w, seconds=0.0, with_bwd=with_bwd)
        vals.append(v)
        per_head.append(sph)
    val = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(per_head) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {**w.describe(), "step": "fwd+bwd" if with_bwd else "fwd",
                       "sample": "one (b,h) head of the workload per step"},
            "cpu_baseline": {"value": val, "unit": "TFLOPS", "cores": threads, "kind": "oracle", "sample": desc},
            "e2e": {"value": val, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm --

def run_gpu(args):
    import exact_attention_78_gb300 as fa
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        replicas.init("nccl", device=torch.device("cuda", local))
    # rank 0 builds the library if it is missing or stale; the others load
    # it once rank 0 is done
    if rank == 0:
        fa.load_library(build_if_missing=True)
    if ws > 1:
        replicas.barrier()
    fa.load_library()
    w = workload(args)
    (q, k, v, do), cu = W.make_inputs(w, with_grad=True)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    cud = None if cu is None else cu.cuda()
    o = torch.empty_like(qd)
    lse_shape = (w.Hq, qd.shape[0]) if w.packed else (w.B, w.Hq, w.Sq)
    lse = torch.empty(lse_shape, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    det = bool(w.extra.get("deterministic", args.deterministic))
    paired = True if args.paired else None
    tuning = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in args.bwd_tune.split(",") if kv} or None
    fwd_knobs = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in args.fwd_tune.split(",") if kv}
    if args.emu is not None:
        fwd_knobs["emu_per_16"] = args.emu

    have_bwd = not args.fwd_only
    ws_buf = dq = dk = dv = None
    if have_bwd:
        # an unsupported backward configuration raises here: the step is
        # never silently reduced to the forward
        if w.packed:
            rows = qd.shape[0]
            need = fa.bwd_workspace_size(w.B, w.Hq, w.Hkv, rows, rows, w.D, det, total_q=rows)
        else:
            need = fa.bwd_workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, det)
        ws_buf = torch.empty(need, dtype=torch.uint8, device="cuda")
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        fa.fwd(qd, kd, vd, causal=w.causal, cu_seqlens=cud, out=o, lse=lse, **fwd_knobs)
        fa.bwd(qd, kd, vd, o, lse, dod, causal=w.causal, deterministic=det, workspace=ws_buf, dq=dq, dk=dk,
               dv=dv, paired=paired, cu_seqlens=cud, tuning=tuning)
    torch.cuda.synchronize()

    ev_f0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_f1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_b1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    fwd_times, bwd_times = [], []

    def step(i=None):
        if i is not None:
            ev_f0[i].record(stream)
        fa.fwd(qd, kd, vd, causal=w.causal, cu_seqlens=cud, out=o, lse=lse, **fwd_knobs)
        if i is not None:
            ev_f1[i].record(stream)
        if have_bwd:
            fa.bwd(qd, kd, vd, o, lse, dod, causal=w.causal, deterministic=det, workspace=ws_buf, dq=dq, dk=dk,
                   dv=dv, paired=paired, cu_seqlens=cud, tuning=tuning)
        if i is not None:
            ev_b1[i].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    st = fa.get_device_error()
    if st != 0:
        raise RuntimeError("device error during warm-up: %s" % fa.status_string(st))

    def barrier():
        torch.cuda.synchronize()
        replicas.barrier()
        torch.cuda.synchronize()

    # Timed region: blocks of exactly `steps` steps, each bracketed by a
    # barrier and a device synchronisation on both sides and timed with CUDA
    # events on the launching stream.  A block of a few milliseconds is too
    # short for clock samples taken every 100 ms to see the GPU under load,
    # so blocks repeat until together they last --min-timed-s; the median
    # block (max over ranks) is reported, and the per-call times average
    # over every timed step.
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    block_ms = []
    max_blocks = 1000
    with ClockSampler(local) as clocks:
        while True:
            barrier()
            start.record(stream)
            for i in range(args.steps):
                step(i)
            end.record(stream)
            torch.cuda.synchronize()
            barrier()
            block_ms.append(replicas.max_over_ranks(start.elapsed_time(end), device="cuda"))
            fwd_times += [ev_f0[i].elapsed_time(ev_f1[i]) for i in range(args.steps)]
            if have_bwd:
                bwd_times += [ev_f1[i].elapsed_time(ev_b1[i]) for i in range(args.steps)]
            # every rank takes the same decision (block times are already the max over ranks)
            if sum(block_ms) >= args.min_timed_s * 1e3 or len(block_ms) >= max_blocks:
                break
    if fa.get_device_error() != 0:
        raise RuntimeError("device error in timed region")
    elapsed_ms = statistics.median(block_ms)
    fwd_ms = statistics.mean(fwd_times)
    bwd_ms = statistics.mean(bwd_times) if have_bwd else 0.0

    flops_step = step_flops(w, have_bwd)
    ms_step = elapsed_ms / args.steps
    value = ws * flops_step / (ms_step * 1e-3) / 1e12

    # end to end through the public API: every step copies its own inputs in
    # from pinned host memory and reads its own results (O, LSE and, with the
    # backward, dQ, dK, dV) back to pinned host memory, all inside the timed
    # region.  Two sets of device buffers and one stream per copy direction
    # let step i + 1's inputs arrive, and step i - 1's results leave, while
    # step i computes (the host link is full duplex).
    e2e = None
    if not args.no_e2e:
        host_in = [t.pin_memory() for t in ((q, k, v, do) if have_bwd else (q, k, v))]
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        hg = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (qd, kd, vd)] if have_bwd else []
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = ho.numel() * 2 + hl.numel() * 4 + sum(t.numel() * 2 for t in hg)
        sets = []
        for _ in range(2):
            ins = [torch.empty_like(t) for t in ((qd, kd, vd, dod) if have_bwd else (qd, kd, vd))]
            grads = [torch.empty_like(t) for t in (qd, kd, vd)] if have_bwd else []
            sets.append((ins, torch.empty_like(o), torch.empty_like(lse), grads))
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        copied = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        read = [torch.cuda.Event() for _ in range(2)]

        def e2e_issue(i):
            bset = i % 2
            ins, oo, ll, gg = sets[bset]
            if i >= 2:
                s_in.wait_event(computed[bset])      # step i - 2 has consumed this set's inputs
            with torch.cuda.stream(s_in):
                for dst, src in zip(ins, host_in):
                    dst.copy_(src, non_blocking=True)
                copied[bset].record(s_in)
            stream.wait_event(copied[bset])
            if i >= 2:
                stream.wait_event(read[bset])        # step i - 2's results have left
            fa.fwd(ins[0], ins[1], ins[2], causal=w.causal, cu_seqlens=cud, out=oo, lse=ll, stream=stream,
                   **fwd_knobs)
            if have_bwd:
                fa.bwd(ins[0], ins[1], ins[2], oo, ll, ins[3], causal=w.causal, deterministic=det, workspace=ws_buf,
                       dq=gg[0], dk=gg[1], dv=gg[2], paired=paired, cu_seqlens=cud, stream=stream, tuning=tuning)
            computed[bset].record(stream)
            s_out.wait_event(computed[bset])
            with torch.cuda.stream(s_out):
                ho.copy_(oo, non_blocking=True)
                hl.copy_(ll, non_blocking=True)
                for hgt, g in zip(hg, gg):
                    hgt.copy_(g, non_blocking=True)
                read[bset].record(s_out)

        for i in range(2):
            e2e_issue(i)
        torch.cuda.synchronize()
        barrier()
        n_e2e = max(3, args.steps // 4)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(n_e2e):
            e2e_issue(i)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = replicas.max_over_ranks(e0.elapsed_time(e1) / n_e2e, device="cuda")
        e2e = {"value": ws * flops_step / (e_ms * 1e-3) / 1e12, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "pipeline": "double-buffered: next step's inputs in and previous step's results out during compute"}

    if rank != 0:
        replicas.finalize()
        return

    pk, pk_kind = peaks()
    # dominant kernel: the longer of the forward kernel and the backward call
    if have_bwd and bwd_ms > fwd_ms:
        dom, dom_ms, dom_flops = "bwd", bwd_ms, 2.5 * fwd_flops_of(w)
    else:
        dom, dom_ms, dom_flops = "fwd", fwd_ms, fwd_flops_of(w)
    kname = "bwd_pair_kernel" if (dom == "bwd" and args.paired) else dom + "_kernel"
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    # Denominator: the burst BF16 peak (a dense GEMM timed for milliseconds
    # at full clock), because each call here runs for milliseconds; the
    # fraction of the sustained (seconds-long, power-capped) figure is given
    # beside it for context.
    peak = float(pk["bf16_tflops"])
    sustained = pk.get("bf16_tflops_sustained")
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": measured_traffic(kname, w), "kernel": kname,
                "timed": ("the whole backward call (its pre, main and post kernels), CUDA events on its stream"
                          if dom == "bwd" else "the forward call (one kernel), CUDA events on its stream"),
                "peak_kind": "%s burst bf16 (bf16_tflops)" % pk_kind,
                "frac_of_sustained": achieved / float(sustained) if sustained else None}

    cpu = None
    if not args.no_cpu:
        cpu_v, cpu_desc, cpu_threads, _ = oracle_sample(w, seconds=12.0, with_bwd=have_bwd)
        cpu = {"value": cpu_v, "unit": "TFLOPS", "cores": cpu_threads, "kind": "oracle", "sample": cpu_desc}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**w.describe(), "step": "fwd+bwd" if have_bwd else "fwd", "deterministic": det,
                   "bwd_kernel": "paired CTAs" if args.paired else "single CTA",
                   **({"bwd_tuning": tuning} if tuning else {}),
                   **({"fwd_tuning": fwd_knobs} if fwd_knobs else {}),
                   "l2": "inputs larger than L2 (Q,K,V,O %d MiB each)" % (qd.numel() * 2 >> 20),
                   "parallelism": "replicas" if ws > 1 else "single"},
        "fwd_tflops": fwd_flops_of(w) / (fwd_ms * 1e-3) / 1e12,
        "fwd_ms": fwd_ms,
        "bwd_tflops": (2.5 * fwd_flops_of(w) / (bwd_ms * 1e-3) / 1e12 if have_bwd else None),
        "bwd_ms": bwd_ms if have_bwd else None,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        # per timed step (every block): the forward kernel; the backward's
        # pre, main and post kernels (packed layout: plus the offset-checking
        # plan kernel)
        "gpu_launches": len(block_ms) * args.steps * (1 + ((4 if w.packed else 3) if have_bwd else 0)),
        "timed_blocks": {"blocks": len(block_ms), "steps_per_block": args.steps,
                         "block_ms_min": min(block_ms), "block_ms_median": elapsed_ms,
                         "block_ms_max": max(block_ms), "total_s": sum(block_ms) / 1e3},
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    replicas.finalize()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
