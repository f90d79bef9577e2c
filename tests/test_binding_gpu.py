"""The Python binding refuses caller-supplied buffers the library would write
out of bounds (wrong shape, dtype or layout), sizes a workspace in bytes
whatever its element type, and launches on the tensors' own device."""

import pytest
import torch

from exact_attention_78_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_78_gb300 as fa_mod
    fa_mod.load_library(build_if_missing=True)
    return fa_mod


def _qkv(B=1, H=2, S=256, D=128):
    w = W.Workload("case", B=B, Hq=H, Hkv=H, Sq=S, Sk=S, D=D, causal=False, seed=31)
    (q, k, v, do), _ = W.make_inputs(w, with_grad=True)
    return tuple(t.cuda() for t in (q, k, v, do))


def test_forward_output_buffers_are_checked(fa):
    q, k, v, _ = _qkv()
    with pytest.raises(ValueError):
        fa.fwd(q, k, v, out=torch.empty(1, 128, 2, 128, dtype=torch.bfloat16, device="cuda"))   # too short
    with pytest.raises(ValueError):
        fa.fwd(q, k, v, out=torch.empty_like(q, dtype=torch.float16))
    with pytest.raises(ValueError):
        fa.fwd(q, k, v, lse=torch.empty(1, 2, 256, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        fa.fwd(q, k, v, lse=torch.empty(1, 256, 2, dtype=torch.float32, device="cuda").transpose(1, 2))
    o, lse = fa.fwd(q, k, v, out=torch.empty_like(q), lse=torch.empty(1, 2, 256, device="cuda"))
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_backward_buffers_are_checked(fa):
    q, k, v, do = _qkv()
    o, lse = fa.fwd(q, k, v)
    with pytest.raises(ValueError):
        fa.bwd(q, k, v, o, lse, do, dq=torch.empty(1, 255, 2, 128, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        fa.bwd(q, k, v, o, lse.reshape(2, 256), do)
    with pytest.raises(ValueError):
        fa.bwd(q, k, v, o[:, :128], lse, do)


def test_workspace_is_sized_in_bytes(fa):
    """A float32 workspace of exactly the needed bytes is accepted, and one
    element short is refused by the library (FA_ERR_WORKSPACE)."""
    q, k, v, do = _qkv()
    o, lse = fa.fwd(q, k, v)
    need = fa.bwd_workspace_size(1, 2, 2, 256, 256, 128)
    assert need % 4 == 0
    ref = fa.bwd(q, k, v, o, lse, do)
    got = fa.bwd(q, k, v, o, lse, do, workspace=torch.empty(need // 4, dtype=torch.float32, device="cuda"))
    for a, b in zip(ref, got):
        assert (a.float() - b.float()).abs().max().item() <= 1e-2
    with pytest.raises(fa.FAError) as e:
        fa.bwd(q, k, v, o, lse, do, workspace=torch.empty(need // 4 - 1, dtype=torch.float32, device="cuda"))
    assert e.value.status == 5


@pytest.mark.parametrize("D", [64, 128])
def test_gradients_into_16_byte_aligned_buffers(fa, D):
    """dK and dV rows are written with 32-byte stores when both buffers are
    32-byte aligned and with 16-byte stores otherwise (the ABI asks for 16).
    In deterministic mode the two paths must give the same bits."""
    q, k, v, do = _qkv(B=1, H=2, S=300, D=D)
    o, lse = fa.fwd(q, k, v, causal=True)
    ref = fa.bwd(q, k, v, o, lse, do, causal=True, deterministic=True)

    def offset_like(t):
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
        view = buf[8:].view(t.shape)            # 16 bytes past a 512-byte-aligned allocation
        assert view.data_ptr() % 32 == 16
        return view

    dq, dk, dv = offset_like(q), offset_like(k), offset_like(v)
    got = fa.bwd(q, k, v, o, lse, do, causal=True, deterministic=True, dq=dq, dk=dk, dv=dv)
    assert fa.get_device_error() == 0
    for a, b in zip(ref, got):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_output_into_16_byte_aligned_buffer(fa, D, causal):
    """O rows are written with 32-byte stores when O is 32-byte aligned and
    with 16-byte stores otherwise (the ABI asks for 16): same bits."""
    q, k, v, _ = _qkv(B=2, H=2, S=300, D=D)
    ref_o, ref_l = fa.fwd(q, k, v, causal=causal)
    buf = torch.empty(q.numel() + 8, dtype=q.dtype, device=q.device)
    o = buf[8:].view(q.shape)                  # 16 bytes past a 512-byte-aligned allocation
    assert o.data_ptr() % 32 == 16
    got_o, got_l = fa.fwd(q, k, v, causal=causal, out=o)
    assert fa.get_device_error() == 0
    assert torch.equal(ref_o.view(torch.int16), got_o.view(torch.int16))
    assert torch.equal(ref_l, got_l)
