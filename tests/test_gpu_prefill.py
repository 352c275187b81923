"""GPU parity of the tensor-core (tcgen05) path that wl_linear and
wl_qkv_fused take for more than 64 tokens, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import wl_synth
from tests.parity import SHAPES_1B, assert_canaries, assert_parity, guarded_empty

pytestmark = pytest.mark.gpu

YDT = [torch.bfloat16, torch.float32]


def _run(wl, x, th, ydt, dev):
    buf, y, pad = guarded_empty((x.shape[0], th.out), ydt, dev)
    tg = th.to(dev)
    wl.wl_linear(x.to(dev), tg.W0, tg.s, tg.U if th.r else None, tg.V if th.r else None, y=y, ydt=ydt)
    torch.cuda.synchronize()
    assert wl.wl_device_status() == wl.WL_OK, wl.wl_last_error()
    assert_canaries(buf, pad)
    return y


@pytest.mark.parametrize("T", [65, 128, 200])
@pytest.mark.parametrize("n_in,out", [(64, 16), (520, 300), (1152, 256), (136, 513)])
@pytest.mark.parametrize("r", [0, 4, 8, 16, 33, 64, 128])
def test_prefill_ragged(wl, orc, gpu, T, n_in, out, r):
    ydt = torch.float32 if (T + r) % 2 else torch.bfloat16
    x, th = wl_synth.linear_case(3000 + T + r, T, n_in, out, r)
    y = _run(wl, x, th, ydt, gpu)
    assert_parity(y, orc.linear(x, th), ydt, f"T={T} in={n_in} out={out} r={r}")


@pytest.mark.parametrize("ydt", YDT)
@pytest.mark.parametrize("kind", ["random", "degenerate"])
def test_prefill_degenerate_and_random(wl, orc, gpu, ydt, kind):
    x, th = wl_synth.linear_case(1, 256, 1152, 1024, 32, kind=kind)
    y = _run(wl, x, th, ydt, gpu)
    assert_parity(y, orc.linear(x, th), ydt, kind)


@pytest.mark.parametrize("fam", sorted(SHAPES_1B))
@pytest.mark.parametrize("r", [16, 32])
def test_prefill_gemma_T2048_sampled(wl, orc, gpu, fam, r):
    """T = 2048 at the Gemma-1B shapes: 64 sampled tokens, all outputs."""
    n_in, out = SHAPES_1B[fam]
    x, th = wl_synth.linear_case(2, 2048, n_in, out, r)
    for ydt in YDT:
        y = _run(wl, x, th, ydt, gpu)
        tok = np.sort(np.random.default_rng(r).choice(2048, 64, replace=False))
        ref = orc.linear_sel(x, th, tok=tok)
        assert_parity(y[torch.as_tensor(tok, device=gpu)], ref, ydt, fam)


def test_prefill_qkv_fused(wl, orc, gpu):
    g = wl_synth.make_generator(5)
    T = 300
    x = wl_synth.draw_x(g, T, 1152)
    ths = [wl_synth.draw_theta(g, 1152, o, 16) for o in (1024, 256, 256)]
    ys = wl.wl_qkv_fused(x.to(gpu), *[t.to(gpu) for t in ths], ydt=torch.float32)
    torch.cuda.synchronize()
    for y, th in zip(ys, ths):
        assert_parity(y, orc.linear(x, th), torch.float32)


def test_prefill_matches_decode_rows(wl, gpu):
    """Rows of a 128-token tensor-core result agree with 8-token decode calls."""
    x, th = wl_synth.linear_case(4, 128, 1152, 512, 8)
    yp = _run(wl, x, th, torch.float32, gpu).cpu()
    for t0 in range(0, 128, 32):
        yd = _run(wl, x[t0:t0 + 8], th, torch.float32, gpu).cpu()
        d = (yd - yp[t0:t0 + 8]).abs().max().item()
        assert d <= 1e-5 * yp.abs().max().item()


def _mlp_case(seed, T, hidden, inter, r):
    g = wl_synth.make_generator(seed)
    x = wl_synth.draw_x(g, T, hidden)
    ths = [wl_synth.draw_theta(g, hidden, inter, r), wl_synth.draw_theta(g, hidden, inter, r),
           wl_synth.draw_theta(g, inter, hidden, r)]
    return x, ths


@pytest.mark.parametrize("T", [9, 65, 200])
@pytest.mark.parametrize("hidden,inter,r", [(64, 136, 3), (264, 520, 0), (128, 1000, 33), (128, 1000, 16), (64, 136, 8)])
def test_prefill_mlp_small(wl, orc, gpu, T, hidden, inter, r):
    x, ths = _mlp_case(T * 7 + r, T, hidden, inter, r)
    ref = orc.mlp_geglu(x, *ths)
    for ydt in YDT:
        buf, y, pad = guarded_empty((T, hidden), ydt, gpu)
        wl.wl_mlp_geglu_fused(x.to(gpu), *[t.to(gpu) for t in ths], y=y, ydt=ydt)
        assert wl.wl_device_status() == wl.WL_OK, wl.wl_last_error()
        assert_canaries(buf, pad)
        assert_parity(y, ref, ydt, f"mlp T={T}")


@pytest.mark.parametrize("r", [16, 32])
def test_prefill_mlp_gemma_T2048_sampled(wl, orc, gpu, r):
    x, ths = _mlp_case(r, 2048, 1152, 6912, r)
    tok = np.sort(np.random.default_rng(r).choice(2048, 48, replace=False))
    ref = orc.mlp_geglu(x, *ths, tok=tok)
    for ydt in YDT:
        y = wl.wl_mlp_geglu_fused(x.to(gpu), *[t.to(gpu) for t in ths], ydt=ydt)
        assert wl.wl_device_status() == wl.WL_OK
        assert_parity(y[torch.as_tensor(tok, device=gpu)], ref, ydt, "mlp T=2048")
