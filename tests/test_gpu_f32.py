"""GPU parity of the fp32 encoding (wl_linear_f32, wl_qkv_fused_f32) against
the oracle's fp64 evaluation of the fp32 values ("Serve and generate with
weightless", "Supported encodings and devices": the architectures also
support float32).  Tolerances as for bf16 inputs: 1e-4 rms(y_ref) for fp32
outputs, 1e-2 rms for bf16 outputs (after the final cast)."""
import numpy as np
import pytest
import torch

import wl_synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


def _to(th, dev):
    return wl_synth.Theta(th.W0.to(dev), th.s.to(dev), th.U.to(dev), th.V.to(dev))


@pytest.mark.parametrize("T,n_in,out,r", [
    (1, 8, 1, 0), (1, 72, 40, 1), (3, 1152, 1024, 4), (5, 136, 200, 5), (16, 264, 96, 32),
    (17, 512, 130, 16), (64, 1152, 256, 128), (200, 200, 72, 33), (7, 6912, 1152, 4),
    # the few-token form at each of its z widths: T x r up to 64
    (1, 5376, 4096, 64), (2, 1152, 1536, 32), (8, 1024, 1152, 8), (4, 2056, 300, 16), (1, 16, 9, 3),
    # the 128 x 128 tiled form at each of its z widths, ragged T, out and K
    (40, 128, 72, 0), (33, 1024, 200, 24), (130, 264, 260, 64),
])
@pytest.mark.parametrize("ydt", [torch.float32, torch.bfloat16])
def test_f32_linear_ragged(wl, orc, gpu, T, n_in, out, r, ydt):
    x, th = wl_synth.linear_case_f32(T * 13 + r, T, n_in, out, r)
    ref = orc.linear_f32(x, th)
    tg = _to(th, gpu)
    U = tg.U if r > 0 else None
    V = tg.V if r > 0 else None
    y = wl.wl_linear(x.to(gpu), tg.W0, tg.s, U, V, ydt=ydt)
    torch.cuda.synchronize()
    assert_parity(y, ref, ydt, f"fp32 linear T={T} {n_in}->{out} r={r}")


@pytest.mark.parametrize("kind", ["degenerate", "delta"])
def test_f32_special_cases(wl, orc, gpu, kind):
    x, th = wl_synth.linear_case_f32(9, 4, 1152, 1024, 8, kind=kind)
    tg = _to(th, gpu)
    y = wl.wl_linear(x.to(gpu), tg.W0, tg.s, tg.U, tg.V, ydt=torch.float32)
    ref = orc.linear_f32(x, th)
    if kind == "degenerate":
        # U = V = 0, s = 1: x W0^T (library matmul in float64)
        np.testing.assert_allclose(ref, (x.double() @ th.W0.double().T).numpy(), rtol=0, atol=1e-9)
    assert_parity(y, ref, torch.float32, kind)


@pytest.mark.parametrize("T", [1, 5, 96])
def test_f32_qkv_fused(wl, orc, gpu, T):
    g = wl_synth.make_generator(31 + T)
    x = wl_synth.draw_x_f32(g, T, 1152)
    ths = [wl_synth.draw_theta_f32(g, 1152, o, 16) for o in (1024, 256, 256)]
    tg = [_to(t, gpu) for t in ths]
    ys = wl.wl_qkv_fused(x.to(gpu), *tg, ydt=torch.float32)
    torch.cuda.synchronize()
    for y, t, n in zip(ys, ths, "qkv"):
        assert_parity(y, orc.linear_f32(x, t), torch.float32, f"qkv {n}")
    # the same as three single calls, within accumulation order
    for y, t in zip(ys, tg):
        y1 = wl.wl_linear(x.to(gpu), t.W0, t.s, t.U, t.V, ydt=torch.float32)
        ref = y1.double().cpu().numpy()
        assert np.max(np.abs(y.double().cpu().numpy() - ref)) <= 1e-5 * np.sqrt(np.mean(ref ** 2))


def test_f32_gemma_prefill_rows(wl, orc, gpu):
    """Gemma-3-1B q projection at T=2048 (fp32 output), every output checked."""
    x, th = wl_synth.linear_case_f32(4, 2048, 1152, 1024, 16)
    tg = _to(th, gpu)
    y = wl.wl_linear(x.to(gpu), tg.W0, tg.s, tg.U, tg.V, ydt=torch.float32)
    assert_parity(y, orc.linear_f32(x, th), torch.float32, "q T=2048")
