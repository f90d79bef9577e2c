"""fa_bwd_noalloc: the backward pass for callers that may not allocate device
memory (a serving runtime or framework allocator that owns the whole GPU, or a
code path where an allocation would stall the device).  It takes its scratch
from a buffer built into the library instead of a caller workspace.

Checked through the C ABI against fa_bwd (caller-provided workspace) on the
same inputs, on two calls in a row: the built-in buffer keeps the previous
call's contents, so the second call also shows that the entry point clears
what must start at zero.  This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

from exact_attention_78_gb300 import workloads as W

from parity import GRAD_RTOL, f64, rel_fro

pytestmark = pytest.mark.gpu

FA_ERR_WORKSPACE = 5
STATIC_SCRATCH_BYTES = 64 << 20


def _call_noalloc(lib, q, k, v, o, lse, do, dq, dk, dv, causal, deterministic):
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.fa_bwd_noalloc(p(q), p(k), p(v), p(o), p(lse), p(do), p(dq), p(dk), p(dv), B, Hq, Hkv, Sq, Sk, D,
                              int(causal), D ** -0.5, None, int(deterministic),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("deterministic", [False, True])
def test_noalloc_backward_matches_fa_bwd_twice(deterministic):
    import exact_attention_78_gb300 as fa
    lib = fa.load_library(build_if_missing=True)
    w = W.Workload("noalloc", B=2, Hq=4, Hkv=2, Sq=700, Sk=700, D=128, causal=True, seed=21)
    assert fa.bwd_workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, deterministic) <= STATIC_SCRATCH_BYTES
    (q, k, v, do), _ = W.make_inputs(w, with_grad=True)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=True)
    ref = fa.bwd(qd, kd, vd, o, lse, dod, causal=True, deterministic=deterministic)
    assert fa.get_device_error() == 0
    for call in range(2):
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        st = _call_noalloc(lib, qd, kd, vd, o, lse, dod, dq, dk, dv, True, deterministic)
        assert st == 0, (call, st)
        assert fa.get_device_error() == 0
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            e = rel_fro(f64(g), f64(r))
            assert e <= GRAD_RTOL, (call, name, e)
            if deterministic:
                assert torch.equal(g.view(torch.int16), r.view(torch.int16)), (call, name)


@pytest.mark.parametrize("deterministic", [False, True])
def test_noalloc_packed_backward_matches_fa_bwd_twice(deterministic):
    """Packed variable-length layout with grouped heads: here the built-in
    buffer also holds the per-sequence tables and the work order that the
    first kernel writes, so two calls in a row show that none of the earlier
    call's contents leaks into the next."""
    import exact_attention_78_gb300 as fa
    lib = fa.load_library(build_if_missing=True)
    lens = [300, 1, 700, 129, 0, 256]
    cu = W.cu_seqlens_of(lens)
    T = int(cu[-1])
    Hq, Hkv, D = 4, 2, 128
    assert fa.bwd_workspace_size(len(lens), Hq, Hkv, T, T, D, deterministic, total_q=T) <= STATIC_SCRATCH_BYTES
    q, k, v, do = (W.randn_bf16((T, h, D), 40 + i).cuda() for i, h in enumerate((Hq, Hkv, Hkv, Hq)))
    cud = cu.cuda()
    o, lse = fa.fwd(q, k, v, causal=True, cu_seqlens=cud)
    ref = fa.bwd(q, k, v, o, lse, do, causal=True, deterministic=deterministic, cu_seqlens=cud)
    assert fa.get_device_error() == 0
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    for call in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = lib.fa_bwd_noalloc(p(q), p(k), p(v), p(o), p(lse), p(do), p(dq), p(dk), p(dv), len(lens), Hq, Hkv,
                                T, T, D, 1, D ** -0.5, p(cud), int(deterministic),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, (call, st)
        assert fa.get_device_error() == 0
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            e = rel_fro(f64(g), f64(r))
            assert e <= GRAD_RTOL, (call, name, e)
            if deterministic:
                assert torch.equal(g.view(torch.int16), r.view(torch.int16)), (call, name)


def test_noalloc_rejects_problems_larger_than_its_buffer():
    import exact_attention_78_gb300 as fa
    lib = fa.load_library(build_if_missing=True)
    # B=1, Hq=16, S=16384, D=128 needs a 128 MiB dQ accumulator
    assert fa.bwd_workspace_size(1, 16, 16, 16384, 16384, 128) > STATIC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")   # never touched: rejected before launch
    p = ctypes.c_void_p(t.data_ptr())
    st = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 16, 16, 16384, 16384, 128, 1, 128 ** -0.5, None, 0,
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == FA_ERR_WORKSPACE
