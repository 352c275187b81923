"""The one-launch layer stack (wl_stack_create / wl_stack_decode): every
output of every layer against the oracle on the bf16 input that projection
received (parity is per projection: chaining bf16 activations through many
layers is not part of the contract), repeat launches bit-identical, and the
limits reported as WL_ERR_UNSUPPORTED.  1..4 tokens and 5..32 tokens run
different kernels; both are covered, at ragged small shapes and at the
Gemma-3-1B layer (32 tokens: the batched-decode case with 32 requests)."""
import numpy as np
import pytest
import torch

import wl_synth
from tests.parity import assert_parity, bf16_ulp

pytestmark = pytest.mark.gpu

GEMMA = dict(hidden=1152, q=1024, kv=256, inter=6912)


def _layers(L, shapes, r, seed, dev, G=None, kind="random"):
    from rank_weight_reconstruction_wl_gb300.stack import build_layers

    return build_layers(L, G or L, 1, shapes, r, seed=seed, device=dev, kind=kind)


def _check_layers(orc, layers, stk, x):
    cpu = lambda t: t.detach().cpu()
    tc = lambda t: wl_synth.Theta(cpu(t.W0), cpu(t.s), cpu(t.U), cpu(t.V))
    xin = cpu(x)
    for l, th in enumerate(layers):
        o = stk.outs[l]
        for name, t in (("yq", th.q), ("yk", th.k), ("yv", th.v)):
            assert_parity(o[name], orc.linear(xin, tc(t)), torch.bfloat16, f"layer {l} {name}")
        assert_parity(o["yo"], orc.linear(cpu(o["yq"]), tc(th.o)), torch.bfloat16, f"layer {l} o")
        ref = orc.mlp_geglu(cpu(o["yo"]), tc(th.gate), tc(th.up), tc(th.down))
        assert_parity(o["ym"], ref, torch.bfloat16, f"layer {l} mlp")
        xin = cpu(o["ym"])


@pytest.mark.parametrize("shapes,L,T,r", [
    (dict(hidden=128, q=64, kv=64, inter=192), 3, 1, 4),
    (dict(hidden=128, q=64, kv=40, inter=192), 2, 3, 5),
    (dict(hidden=256, q=128, kv=72, inter=320), 3, 4, 0),
    (dict(hidden=192, q=256, kv=64, inter=640), 2, 2, 32),
    (dict(hidden=64, q=64, kv=16, inter=64), 2, 1, 8),
    (dict(hidden=128, q=64, kv=40, inter=192), 2, 5, 5),
    (dict(hidden=256, q=128, kv=72, inter=320), 3, 8, 0),
    (dict(hidden=128, q=64, kv=64, inter=192), 2, 12, 16),
    (dict(hidden=192, q=256, kv=64, inter=640), 2, 17, 32),
    (dict(hidden=128, q=64, kv=24, inter=256), 3, 32, 4),
    (dict(hidden=64, q=64, kv=16, inter=64), 2, 32, 1),
])
def test_stack_kernel_small(wl, orc, gpu, shapes, L, T, r):
    layers = _layers(L, shapes, r, seed=11 + T + r, dev=gpu)
    stk = wl.WLStack(layers, T, device=gpu)
    g = torch.Generator(device=gpu)
    g.manual_seed(5)
    x = torch.randn(T, shapes["hidden"], generator=g, device=gpu).to(torch.bfloat16)
    stk.decode(x)
    torch.cuda.synchronize()
    assert wl.wl_device_status() == wl.WL_OK, wl.wl_last_error()
    _check_layers(orc, layers, stk, x)


@pytest.mark.parametrize("L,G,T,r", [(3, 3, 1, 4), (2, 1, 4, 32), (2, 2, 2, 16),
                                     (3, 3, 32, 4), (2, 1, 32, 4), (2, 2, 32, 16), (3, 1, 32, 32),
                                     (2, 2, 16, 32), (2, 1, 7, 4)])
def test_stack_kernel_gemma(wl, orc, gpu, L, G, T, r):
    layers = _layers(L, GEMMA, r, seed=21 + r, dev=gpu, G=G)
    stk = wl.WLStack(layers, T, device=gpu)
    g = torch.Generator(device=gpu)
    g.manual_seed(6)
    x = torch.randn(T, GEMMA["hidden"], generator=g, device=gpu).to(torch.bfloat16)
    stk.decode(x)
    torch.cuda.synchronize()
    assert wl.wl_device_status() == wl.WL_OK, wl.wl_last_error()
    _check_layers(orc, layers, stk, x)


@pytest.mark.parametrize("T,r", [(1, 4), (4, 32), (32, 4), (32, 32)])
def test_stack_kernel_delta_dominant(wl, orc, gpu, T, r):
    """U, V drawn ten times larger than the default, so that the rank-r term
    (x V) U^T outweighs the W0 term in every projection: the kernels' z = x V
    and U z paths are then checked well inside the tolerance, not at a few
    per cent of it."""
    layers = _layers(2, GEMMA, r, seed=40 + T + r, dev=gpu, kind="delta")
    cpu = lambda t: t.detach().cpu()
    th = layers[0].q
    g = torch.Generator(device=gpu)
    g.manual_seed(8)
    x = torch.randn(T, GEMMA["hidden"], generator=g, device=gpu).to(torch.bfloat16)
    full = orc.linear(cpu(x), wl_synth.Theta(cpu(th.W0), cpu(th.s), cpu(th.U), cpu(th.V)))
    w0only = orc.linear(cpu(x), wl_synth.Theta(cpu(th.W0), cpu(th.s), 0 * cpu(th.U), 0 * cpu(th.V)))
    rms = lambda a: float(np.sqrt(np.mean(a ** 2)))
    assert rms(full - w0only) > 1.5 * rms(w0only)
    stk = wl.WLStack(layers, T, device=gpu)
    stk.decode(x)
    torch.cuda.synchronize()
    assert wl.wl_device_status() == wl.WL_OK, wl.wl_last_error()
    _check_layers(orc, layers, stk, x)


@pytest.mark.parametrize("T", [1, 32])
def test_stack_kernel_repeat_identical(wl, gpu, T):
    layers = _layers(4, GEMMA, 4, seed=3, dev=gpu)
    stk = wl.WLStack(layers, T, device=gpu)
    x = torch.randn(T, GEMMA["hidden"], device=gpu).to(torch.bfloat16)
    stk.decode(x)
    first = [{k: v.clone() for k, v in o.items()} for o in stk.outs]
    s = torch.cuda.Stream(gpu)
    for _ in range(10):
        stk.decode(x, stream=s)
    s.synchronize()
    assert wl.wl_device_status(s) == wl.WL_OK, wl.wl_last_error()
    for a, b in zip(first, stk.outs):
        for k in a:
            assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("T", [1, 32])
def test_stack_kernel_matches_per_call_path(wl, gpu, T):
    """The one-launch stack and the per-projection calls on the same inputs."""
    layers = _layers(2, GEMMA, 4, seed=4, dev=gpu)
    stk = wl.WLStack(layers, T, device=gpu)
    x = torch.randn(T, GEMMA["hidden"], device=gpu).to(torch.bfloat16)
    stk.decode(x)
    torch.cuda.synchronize()
    th = layers[0]
    yq, yk, yv = wl.wl_qkv_fused(x, th.q, th.k, th.v)
    yo = wl.wl_linear(stk.outs[0]["yq"], th.o.W0, th.o.s, th.o.U, th.o.V)
    ym = wl.wl_mlp_geglu_fused(stk.outs[0]["yo"], th.gate, th.up, th.down)
    torch.cuda.synchronize()
    for a, b in ((yq, "yq"), (yk, "yk"), (yv, "yv"), (yo, "yo"), (ym, "ym")):
        # both are bf16 roundings of fp32 values within 1e-2 rms of the exact
        # result: they may differ by that twice plus one bf16 step
        ref = a.double().cpu().numpy()
        y = stk.outs[0][b].double().cpu().numpy()
        rms = float(np.sqrt(np.mean(ref ** 2)))
        d = np.abs(y - ref) - bf16_ulp(np.maximum(np.abs(y), np.abs(ref)))
        assert d.max() <= 2e-2 * rms, (b, d.max(), rms)


@pytest.mark.parametrize("T,r,hidden", [(33, 4, 128), (1, 33, 128), (1, 4, 96), (32, 33, 128), (16, 4, 96)])
def test_stack_kernel_limits(wl, gpu, T, r, hidden):
    shapes = dict(hidden=hidden, q=64, kv=64, inter=128)
    layers = _layers(1, shapes, r, seed=1, dev=gpu)
    with pytest.raises(wl.WLError) as ei:
        wl.WLStack(layers, T, device=gpu)
    assert ei.value.status == wl.WL_ERR_UNSUPPORTED
