"""The C-ABI shared library on the host, without a GPU: it builds, loads,
exports every function the public headers declare, and rejects bad
arguments synchronously before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import exact_attention_78_gb300 as fa
    return fa.load_library(build_if_missing=True)


def _declared():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        with open(os.path.join(ROOT, "include", h)) as f:
            text = f.read()
        names += re.findall(r"^FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text, flags=re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_get_device_error", "fa_status_string",
            "fa_fwd_ex", "fa_diag_exp2", "fa_diag_wait_timeout"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in enumerate(["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA",
                                 "FA_ERR_TIMEOUT", "FA_ERR_WORKSPACE"]):
        assert lib.fa_status_string(code).decode() == name
    assert lib.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"


# Pointers that are never dereferenced: validation rejects every call below
# before any CUDA call is made.
A = ctypes.c_void_p(1 << 20)          # 16-byte aligned fake address
MIS = ctypes.c_void_p((1 << 20) + 8)  # misaligned


def _fwd(lib, q=A, k=A, v=A, o=A, lse=A, B=1, Hq=2, Hkv=2, Sq=128, Sk=128, D=128, causal=0, scale=0.125,
         cu=None):
    return lib.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, cu, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(lse=None), 1), (dict(o=MIS), 1), (dict(k=MIS), 1),
    (dict(B=0), 1), (dict(Sq=0), 1), (dict(Sk=-3), 1), (dict(Hq=3, Hkv=2), 1),
    (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1),
    (dict(causal=2), 1), (dict(D=96), 2), (dict(D=256), 2),
    (dict(cu=ctypes.c_void_p(A.value), Sq=100, Sk=120), 1),
    (dict(cu=ctypes.c_void_p(A.value + 2)), 1),
    (dict(cu=ctypes.c_void_p(A.value), B=2000), 2),
])
def test_forward_rejects_bad_arguments(lib, kw, status):
    assert _fwd(lib, **kw) == status


def test_forward_tuning_validation(lib):
    from exact_attention_78_gb300.binding import FwdTuning
    t = lib.fa_fwd_default_tuning()
    assert t.rescale_threshold == 8.0 and t.emu_per_16 == -1 and t.split_p == -1 and t.kv_stages == -1
    assert t.head_group == -1
    for thr, emu, split, stages in ((-1.0, 0, -1, -1), (17.0, 0, -1, -1), (8.0, 1, -1, -1), (8.0, 5, -1, -1),
                                    (float("nan"), 0, -1, -1), (8.0, 0, 2, -1), (8.0, 0, 0, 1), (8.0, 0, 0, 5)):
        bad = FwdTuning(thr, emu, split, stages, -1)
        assert lib.fa_fwd_ex(A, A, A, A, A, 1, 2, 2, 128, 128, 128, 0, 0.125, None, ctypes.byref(bad), None) == 1
    # D = 64 allows a deeper ring than D = 128
    bad = FwdTuning(8.0, 0, 0, 11, -1)
    assert lib.fa_fwd_ex(A, A, A, A, A, 1, 2, 2, 128, 128, 64, 0, 0.125, None, ctypes.byref(bad), None) == 1


def _ws(lib, B, Hq, Hkv, Sq, Sk, D, det, total_q=0, offs=None):
    arr = None if offs is None else (ctypes.c_int * len(offs))(*offs)
    return lib.fa_bwd_workspace_size(B, Hq, Hkv, Sq, Sk, D, arr, total_q, det)


def test_workspace_size(lib):
    n = _ws(lib, 2, 16, 16, 8192, 8192, 128, 0)
    acc = 2 * 8192 * 16 * 128 * 4
    rows = 2 * 16 * 8192 * 4
    assert n == acc + 2 * rows + 256                # + the scheduler's work counter
    det = _ws(lib, 2, 16, 16, 8192, 8192, 128, 1)
    assert det == n + 2 * 16 * 128 * 2 * 4      # two tickets (feature halves) per 64-row query block
    # ragged rows: the per-row terms are padded to a multiple of 64 rows
    r = _ws(lib, 1, 2, 2, 100, 100, 128, 0)
    assert r == (1 * 100 * 2 * 128 * 4 + 255) // 256 * 256 + 2 * (1 * 2 * 128 * 4) + 256
    assert _ws(lib, 2, 16, 16, 8192, 8192, 96, 0) == 0
    # D = 64: the accumulator halves, the row terms do not
    assert _ws(lib, 2, 16, 16, 8192, 8192, 64, 0) == acc // 2 + 2 * rows + 256
    assert _ws(lib, 2, 15, 4, 8192, 8192, 128, 0) == 0
    assert _ws(lib, 2, 16, 16, 8192, 8192, 128, 3) == 0


def test_packed_workspace_size(lib):
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    B, H, total = 3, 4, 1000
    pad = (total + 63) // 64 * 64 + 64 * B          # row terms per head: every sequence rounded up to 64
    order = (total // 128 + B) * 2 * 8                # unit order table: (key block, kv head) entries of 8 B
    want = al(total * H * 128 * 4) + 2 * al(H * pad * 4) + al((2 * B + 4) * 4) + al(order) + 256
    assert _ws(lib, B, H, 2, total, total, 128, 0, total_q=total) == want
    assert _ws(lib, B, H, 2, total, total, 128, 1, total_q=total) == want + al(H * (pad // 64) * 2 * 4)
    assert _ws(lib, B, H, 2, total, total, 128, 0, total_q=total, offs=[0, 10, 700, 1000]) == want
    assert _ws(lib, B, H, 2, total, total, 128, 0, total_q=total, offs=[0, 10, 5, 1000]) == 0     # decreasing
    assert _ws(lib, B, H, 2, total, total, 128, 0, total_q=total, offs=[0, 10, 700, 999]) == 0    # last != total
    assert _ws(lib, B, H, 2, total, 999, 128, 0, total_q=total) == 0                              # Sk != total
    assert _ws(lib, 1025, H, 2, total, total, 128, 0, total_q=total) == 0                         # too many sequences


def test_backward_rejects_bad_arguments(lib):
    def call(ws=A, ws_bytes=1 << 40, cu=None, det=0, D=128, dq=A):
        return lib.fa_bwd(A, A, A, A, A, A, dq, A, A, 1, 2, 2, 128, 128, D, 0, 0.125, cu, det, ws, ws_bytes, None)
    assert call(dq=None) == 1
    assert call(dq=MIS) == 1
    assert call(det=2) == 1
    assert call(D=80) == 2
    assert call(cu=ctypes.c_void_p(A.value + 2)) == 1      # offsets must be 4-byte aligned
    assert call(ws=None) == 5
    assert call(ws=ctypes.c_void_p(A.value + 16)) == 5
    assert call(ws_bytes=100) == 5


def test_backward_tuning_validation(lib):
    from exact_attention_78_gb300.binding import BwdTuning
    d = lib.fa_bwd_default_tuning()
    assert d.paired == 0
    assert (d.schedule, d.head_group, d.reverse_blocks, d.scores_first, d.split_dq) == (-1, -1, -1, -1, -1)
    # one knob out of range at a time, on top of the defaults (only rejected
    # calls are made: the pointers are not device memory)
    bad_values = {"paired": (2, 7), "schedule": (2,), "head_group": (0,), "reverse_blocks": (2,),
                  "scores_first": (3,), "split_dq": (2,)}
    for name, vals in bad_values.items():
        for val in vals:
            bad = lib.fa_bwd_default_tuning()
            setattr(bad, name, val)
            assert lib.fa_bwd_ex(A, A, A, A, A, A, A, A, A, 1, 2, 2, 128, 128, 128, 0, 0.125, None, 0, A, 1 << 40,
                                 ctypes.byref(bad), None) == 1, (name, val)
    assert len(BwdTuning._fields_) == 6


def test_binding_rejects_unknown_backward_knob():
    import torch
    import exact_attention_78_gb300 as fa
    x = torch.zeros(1, 128, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(KeyError):
        fa.bwd(x, x, x, x, torch.zeros(1, 2, 128), x, tuning={"no_such_knob": 1})


def test_diag_argument_checks(lib):
    assert lib.fa_diag_exp2(None, None, None, -1, None) == 1
    assert lib.fa_diag_exp2(None, None, None, 10, None) == 1
    assert lib.fa_diag_exp2(None, None, None, 0, None) == 0
    assert lib.fa_diag_wait_timeout(0, None) == 1
    assert lib.fa_diag_wait_timeout(20_000_000_000, None) == 1


def test_python_binding_fails_loudly_without_cuda_tensors():
    import torch
    import exact_attention_78_gb300 as fa
    x = torch.zeros(1, 128, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd(x, x, x)


def test_headers_compile_as_c99_and_link(lib, tmp_path):
    """The public headers are plain C: a C99 program (strict, warnings as
    errors) includes both, links the shared library, and its struct sizes
    match the Python binding's."""
    import shutil
    import subprocess
    from exact_attention_78_gb300 import binding
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    so = binding.lib_path()
    exe = str(tmp_path / "abi_consumer")
    subprocess.run([gcc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "abi_consumer.c"), "-o", exe, "-L", os.path.dirname(so),
                    "-l:" + os.path.basename(so), "-Wl,-rpath," + os.path.dirname(so)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=60).stdout
    sizes = dict(line.rsplit(" ", 1) for line in out.splitlines() if line.startswith("sizeof"))
    assert int(sizes["sizeof fa_fwd_tuning"]) == ctypes.sizeof(binding.FwdTuning)
    assert int(sizes["sizeof fa_bwd_tuning"]) == ctypes.sizeof(binding.BwdTuning)
    assert "status FA_ERR_WORKSPACE" in out
