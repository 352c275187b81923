"""The fused MLP entry point for callers that cannot allocate device memory.

wl_mlp_geglu_fused_noalloc runs the same MLP as wl_mlp_geglu_fused but keeps
its workspace in a scratch array built into libwl.so, so a caller that may not
call cudaMalloc (a host callback, an allocator hook, a process with a fixed
device-memory budget) can still use it.  These tests call it through the C ABI
and check it against the workspace entry point, twice in a row (the scratch
keeps the previous call's contents), plus the size limit.  This file is
collected last so a stop-at-first-failure run has already run everything else.
"""
import ctypes as C

import pytest
import torch

import wl_synth
from tests.parity import TOL

pytestmark = pytest.mark.gpu


def _case(seed, T, hidden, inter, r):
    g = wl_synth.make_generator(seed)
    x = wl_synth.draw_x(g, T, hidden)
    ths = [wl_synth.draw_theta(g, hidden, inter, r), wl_synth.draw_theta(g, hidden, inter, r),
           wl_synth.draw_theta(g, inter, hidden, r)]
    return x, ths


def _call_noalloc(wl, x, ths, y, ydt_code, r):
    T, hidden = x.shape
    inter = ths[0].W0.shape[0]
    ps = [wl._proj(th, inp, r, n) for th, inp, n in
          zip(ths, (hidden, hidden, inter), ("gate", "up", "down"))]
    st = wl.lib().wl_mlp_geglu_fused_noalloc(
        C.c_void_p(x.data_ptr()), ps[0], ps[1], ps[2], C.c_void_p(y.data_ptr()),
        T, hidden, inter, r, ydt_code, C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


@pytest.mark.parametrize("ydt,code", [(torch.bfloat16, 0), (torch.float32, 1)])
@pytest.mark.parametrize("T,r", [(1, 4), (3, 32)])
def test_noalloc_matches_workspace_entry_point(wl, gpu, ydt, code, T, r):
    x, ths = _case(90 + T + r, T, 1152, 6912, r)
    xg = x.to(gpu)
    tg = [t.to(gpu) for t in ths]
    ref = wl.wl_mlp_geglu_fused(xg, *tg, ydt=ydt).float()
    rms = ref.pow(2).mean().sqrt().item()
    for _ in range(2):  # two calls in a row through the shared scratch
        y = torch.full((T, 1152), float("nan"), dtype=ydt, device=gpu)
        st = _call_noalloc(wl, xg, tg, y, code, r)
        assert st == wl.WL_OK, wl.wl_last_error()
        assert wl.wl_device_status() == wl.WL_OK
        err = (y.float() - ref).abs().max().item()
        assert err <= TOL[ydt] * rms, err


@pytest.mark.parametrize("ydt,code", [(torch.bfloat16, 0), (torch.float32, 1)])
@pytest.mark.parametrize("T", [16, 48])
def test_noalloc_many_tokens_after_a_decode_call(wl, gpu, ydt, code, T):
    """T > 8 takes the tensor-core MLP, whose workspace (fp32 g and u, then
    the bf16 hi and lo parts of h) is laid out differently from the decode
    path's; a decode-shape call first leaves its own data in the scratch.
    48 tokens is close to the largest T the 4 MiB scratch holds for these
    shapes with fp32 outputs."""
    r = 16
    xd, thd = _case(70, 1, 1152, 6912, r)
    yd = torch.empty(1, 1152, dtype=ydt, device=gpu)
    assert _call_noalloc(wl, xd.to(gpu), [t.to(gpu) for t in thd], yd, code, r) == wl.WL_OK
    x, ths = _case(80 + T, T, 1152, 6912, r)
    xg = x.to(gpu)
    tg = [t.to(gpu) for t in ths]
    ref = wl.wl_mlp_geglu_fused(xg, *tg, ydt=ydt).float()
    rms = ref.pow(2).mean().sqrt().item()
    y = torch.full((T, 1152), float("nan"), dtype=ydt, device=gpu)
    st = _call_noalloc(wl, xg, tg, y, code, r)
    assert st == wl.WL_OK, wl.wl_last_error()
    assert wl.wl_device_status() == wl.WL_OK
    err = (y.float() - ref).abs().max().item()
    assert err <= TOL[ydt] * rms, err


def test_noalloc_python_wrapper(wl, gpu):
    x, ths = _case(5, 2, 1152, 6912, 4)
    xg = x.to(gpu)
    tg = [t.to(gpu) for t in ths]
    ref = wl.wl_mlp_geglu_fused(xg, *tg).float()
    y = torch.full((2, 1152), float("nan"), dtype=torch.bfloat16, device=gpu)
    out = wl.wl_mlp_geglu_fused_noalloc(xg, *tg, y=y)
    assert out is y
    torch.cuda.synchronize()
    rms = ref.pow(2).mean().sqrt().item()
    assert (y.float() - ref).abs().max().item() <= TOL[torch.bfloat16] * rms


def test_noalloc_rejects_sizes_beyond_scratch(wl, gpu):
    hidden, inter, r = 5376, 21504 * 8, 128
    need = wl.wl_mlp_workspace_bytes(1, hidden, inter, r)
    assert need > 4 << 20
    x = torch.zeros(1, hidden, dtype=torch.bfloat16, device=gpu)
    y = torch.zeros(1, hidden, dtype=torch.bfloat16, device=gpu)
    P = wl._Proj(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), inter)
    Pd = wl._Proj(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), hidden)
    st = wl.lib().wl_mlp_geglu_fused_noalloc(C.c_void_p(x.data_ptr()), P, P, Pd,
                                             C.c_void_p(y.data_ptr()), 1, hidden, inter, r, 0, None)
    assert st == wl.WL_ERR_UNSUPPORTED
    assert "built-in scratch" in wl.wl_last_error()
