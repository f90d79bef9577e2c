"""ctypes binding of the C ABI (include/fa.h, include/fa_diag.h).

Argument marshalling only: torch tensors supply device memory and the current
CUDA stream; every step of the computation runs in the library's kernels.
There is no fallback: if the shared library is missing, every call raises.
"""

import ctypes
import os

import torch

from . import build as _build

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_WORKSPACE = range(6)
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA",
                4: "FA_ERR_TIMEOUT", 5: "FA_ERR_WORKSPACE"}


class FAError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s" % (where, STATUS_NAMES.get(status, status)))


class FwdTuning(ctypes.Structure):
    _fields_ = [("rescale_threshold", ctypes.c_float), ("emu_per_16", ctypes.c_int), ("split_p", ctypes.c_int),
                ("kv_stages", ctypes.c_int), ("head_group", ctypes.c_int)]


class BwdTuning(ctypes.Structure):
    _fields_ = [("paired", ctypes.c_int), ("schedule", ctypes.c_int), ("head_group", ctypes.c_int),
                ("reverse_blocks", ctypes.c_int), ("scores_first", ctypes.c_int), ("split_dq", ctypes.c_int)]


_LIB = None
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

_SIGNATURES = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp]),
    "fa_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp,
                       ctypes.POINTER(FwdTuning), _vp]),
    "fa_fwd_default_tuning": (FwdTuning, []),
    "fa_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_int), _i, _i]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _i,
                    _vp, _sz, _vp]),
    "fa_bwd_default_tuning": (BwdTuning, []),
    "fa_bwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _i,
                       _vp, _sz, ctypes.POINTER(BwdTuning), _vp]),
    "fa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp,
                            _i, _vp]),
    "fa_get_device_error": (_i, [_vp]),
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_diag_exp2": (_i, [_vp, _vp, _vp, ctypes.c_longlong, _vp]),
    "fa_diag_wait_timeout": (_i, [ctypes.c_ulonglong, _vp]),
}


def lib_path():
    return _build.LIB


def load_library(build_if_missing=False):
    """Loads the in-tree shared library; raises if absent.  With
    build_if_missing, (re)builds it first when it is absent or older than a
    source file."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise RuntimeError("CUDA library %s is not built; run exact_attention_78_gb300.build.build()"
                               % _build.LIB)
        _build.build()
    lib = ctypes.CDLL(_build.LIB)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(status, where):
    if status != FA_OK:
        raise FAError(status, where)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_bf16(name, t):
    if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA bfloat16 tensor" % name)


def _check_out(name, t, shape, dtype, device):
    """A caller-supplied output buffer: the library writes shape x dtype
    elements at its address, so anything else is refused here."""
    if (not t.is_cuda or t.device != device or t.dtype != dtype or not t.is_contiguous()
            or tuple(t.shape) != tuple(shape)):
        raise ValueError("%s must be a contiguous %s tensor of shape %s on %s" % (name, dtype, tuple(shape), device))


def _check_same_device(device, **tensors):
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError("%s is on %s, q on %s" % (name, t.device, device))


def _dims(q, k, cu_seqlens):
    """(B, Hq, Hkv, Sq, Sk, D) as the C ABI wants them."""
    if cu_seqlens is None:
        if q.dim() != 4 or k.dim() != 4:
            raise ValueError("dense q/k/v are [B, S, H, D]")
        B, Sq, Hq, D = q.shape
        Sk, Hkv = k.shape[1], k.shape[2]
    else:
        if q.dim() != 3 or k.dim() != 3:
            raise ValueError("packed q/k/v are [total, H, D]")
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or not cu_seqlens.is_contiguous():
            raise ValueError("cu_seqlens must be a contiguous CUDA int32 tensor")
        B = cu_seqlens.numel() - 1
        Sq, Hq, D = q.shape
        Sk, Hkv = k.shape[0], k.shape[1]
    return B, Hq, Hkv, Sq, Sk, D


def fwd(q, k, v, causal=False, scale=None, cu_seqlens=None, out=None, lse=None, rescale_threshold=None,
        emu_per_16=None, split_p=None, kv_stages=None, head_group=None, stream=None):
    """O, LSE = attention(q, k, v).  Dense [B,S,H,D] or packed [total,H,D].
    rescale_threshold, emu_per_16, split_p, kv_stages and head_group override
    the library's per-configuration choices (fa_fwd_tuning)."""
    lib = load_library()
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_bf16(n, t)
    _check_same_device(q.device, k=k, v=v, cu_seqlens=cu_seqlens)
    B, Hq, Hkv, Sq, Sk, D = _dims(q, k, cu_seqlens)
    if scale is None:
        scale = D ** -0.5
    lse_shape = (Hq, Sq) if cu_seqlens is not None else (B, Hq, Sq)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_out("out", out, q.shape, torch.bfloat16, q.device)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    else:
        _check_out("lse", lse, lse_shape, torch.float32, q.device)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D, int(bool(causal)),
            float(scale), _ptr(cu_seqlens)]
    with torch.cuda.device(q.device):   # the library launches on the current device
        knobs = {"emu_per_16": emu_per_16, "split_p": split_p, "kv_stages": kv_stages, "head_group": head_group}
        if rescale_threshold is None and all(x is None for x in knobs.values()):
            st = lib.fa_fwd(*args, _stream(stream))
        else:
            t = lib.fa_fwd_default_tuning()
            if rescale_threshold is not None:
                t.rescale_threshold = float(rescale_threshold)
            for name, val in knobs.items():
                if val is not None:
                    setattr(t, name, int(val))
            st = lib.fa_fwd_ex(*args, ctypes.byref(t), _stream(stream))
    _check(st, "fa_fwd")
    return out, lse


def bwd_workspace_size(B, Hq, Hkv, Sq, Sk, D, deterministic=False, total_q=0, cu_seqlens_host=None):
    """Workspace bytes of fa_bwd.  Packed layout: total_q = packed row count
    (= Sq = Sk); cu_seqlens_host, if given, is a host sequence of B + 1 offsets."""
    offs = None
    if cu_seqlens_host is not None:
        vals = [int(x) for x in cu_seqlens_host]
        offs = (ctypes.c_int * len(vals))(*vals)
    return int(load_library().fa_bwd_workspace_size(B, Hq, Hkv, Sq, Sk, D, offs, int(total_q),
                                                    int(bool(deterministic))))


def bwd(q, k, v, o, lse, do, causal=False, scale=None, deterministic=False, workspace=None, dq=None, dk=None,
        dv=None, paired=None, cu_seqlens=None, stream=None, tuning=None):
    """dQ, dK, dV of attention(q, k, v) given O, LSE and dO.  Dense [B,S,H,D]
    or packed [total,H,D] with cu_seqlens (LSE [Hq, total]).  paired=True runs
    the main kernel on CTA pairs (paired tcgen05 MMAs; dense only).  tuning:
    a dict of fa_bwd_tuning fields (schedule, head_group, reverse_blocks,
    scores_first, split_dq) overriding the per-call defaults."""
    unknown = set(tuning or {}) - {f[0] for f in BwdTuning._fields_}
    if unknown:
        raise KeyError("unknown backward tuning field(s): %s" % ", ".join(sorted(unknown)))
    lib = load_library()
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check_bf16(n, t)
    _check_same_device(q.device, k=k, v=v, o=o, lse=lse, do=do, cu_seqlens=cu_seqlens)
    B, Hq, Hkv, Sq, Sk, D = _dims(q, k, cu_seqlens)
    if tuple(o.shape) != tuple(q.shape) or tuple(do.shape) != tuple(q.shape):
        raise ValueError("o and do must have q's shape %s" % (tuple(q.shape),))
    if tuple(v.shape) != tuple(k.shape):
        raise ValueError("v must have k's shape %s" % (tuple(k.shape),))
    lse_shape = (Hq, Sq) if cu_seqlens is not None else (B, Hq, Sq)
    if not lse.is_cuda or lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != lse_shape:
        raise ValueError("lse must be a contiguous CUDA float32 tensor of shape %s" % (lse_shape,))
    if scale is None:
        scale = D ** -0.5
    need = bwd_workspace_size(B, Hq, Hkv, Sq, Sk, D, deterministic, total_q=Sq if cu_seqlens is not None else 0)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    elif not workspace.is_cuda or workspace.device != q.device or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on %s" % q.device)
    for name, t, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t is not None:
            _check_out(name, t, like.shape, torch.bfloat16, q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq,
            Sk, D, int(bool(causal)), float(scale), _ptr(cu_seqlens), int(bool(deterministic)), _ptr(workspace),
            workspace.numel() * workspace.element_size()]
    with torch.cuda.device(q.device):   # the library launches on the current device
        if paired is None and not tuning:
            st = lib.fa_bwd(*args, _stream(stream))
        else:
            t = lib.fa_bwd_default_tuning()
            if paired is not None:
                t.paired = int(bool(paired))
            for name, val in (tuning or {}).items():
                setattr(t, name, int(val))
            st = lib.fa_bwd_ex(*args, ctypes.byref(t), _stream(stream))
    _check(st, "fa_bwd")
    return dq, dk, dv


def get_device_error(stream=None):
    """Synchronises and returns (and clears) the library's device error status."""
    return int(load_library().fa_get_device_error(_stream(stream)))


def status_string(status):
    return load_library().fa_status_string(int(status)).decode()


def exp2_probe(x, stream=None):
    """(2^x by the FMA polynomial, 2^x by the hardware unit) for a CUDA float32 tensor."""
    lib = load_library()
    if not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA float32 tensor")
    ye, yh = torch.empty_like(x), torch.empty_like(x)
    _check(lib.fa_diag_exp2(_ptr(x), _ptr(ye), _ptr(yh), x.numel(), _stream(stream)), "fa_diag_exp2")
    return ye, yh


def wait_timeout_probe(limit_ns, stream=None):
    _check(load_library().fa_diag_wait_timeout(int(limit_ns), _stream(stream)), "fa_diag_wait_timeout")
