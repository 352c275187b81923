"""GPU parity of wl_mlp_geglu_fused (against the oracle's fp64 GeGLU MLP) and
of wl_materialize (bit-exact against the oracle's fixed-order fp32 value)."""
import numpy as np
import pytest
import torch

import wl_synth
from tests.parity import SHAPES_1B, assert_canaries, assert_parity, guarded_empty

pytestmark = pytest.mark.gpu


def _mlp_case(seed, T, hidden, inter, r, kind="random"):
    g = wl_synth.make_generator(seed)
    x = wl_synth.draw_x(g, T, hidden)
    tg = wl_synth.draw_theta(g, hidden, inter, r, kind)
    tu = wl_synth.draw_theta(g, hidden, inter, r, kind)
    td = wl_synth.draw_theta(g, inter, hidden, r, kind)
    return x, tg, tu, td


def _run_mlp(wl, x, tg, tu, td, ydt, dev):
    T, hidden = x.shape
    buf, y, pad = guarded_empty((T, hidden), ydt, dev)
    wl.wl_mlp_geglu_fused(x.to(dev), tg.to(dev), tu.to(dev), td.to(dev), y=y, ydt=ydt)
    assert wl.wl_device_status() == wl.WL_OK
    assert_canaries(buf, pad)
    return y


@pytest.mark.parametrize("T", [1, 3, 8, 11])
@pytest.mark.parametrize("hidden,inter,r", [(64, 136, 3), (264, 520, 0), (128, 1000, 33)])
def test_mlp_small(wl, orc, gpu, T, hidden, inter, r):
    x, tg, tu, td = _mlp_case(T + r, T, hidden, inter, r)
    ref = orc.mlp_geglu(x, tg, tu, td)
    for ydt in (torch.bfloat16, torch.float32):
        assert_parity(_run_mlp(wl, x, tg, tu, td, ydt, gpu), ref, ydt, f"T={T}")


@pytest.mark.parametrize("r", [4, 32])
@pytest.mark.parametrize("T", [1, 4])
def test_mlp_gemma_decode(wl, orc, gpu, r, T):
    x, tg, tu, td = _mlp_case(40 + r, T, 1152, 6912, r)
    ref = orc.mlp_geglu(x, tg, tu, td)
    for ydt in (torch.bfloat16, torch.float32):
        assert_parity(_run_mlp(wl, x, tg, tu, td, ydt, gpu), ref, ydt)


def test_mlp_degenerate(wl, orc, gpu):
    x, tg, tu, td = _mlp_case(7, 2, 1152, 6912, 4, kind="degenerate")
    ref = orc.mlp_geglu(x, tg, tu, td)
    assert_parity(_run_mlp(wl, x, tg, tu, td, torch.float32, gpu), ref, torch.float32)


def test_mlp_repeated_calls_share_workspace(wl, gpu):
    """The workspace barrier words are left at zero: calls can follow each other."""
    x, tg, tu, td = _mlp_case(8, 1, 1152, 6912, 4)
    ys = [_run_mlp(wl, x, tg, tu, td, torch.float32, gpu) for _ in range(3)]
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])


def test_mlp_large_set_sampled(wl, orc, gpu):
    """hidden 5376, inter 21504, r=64, T=1: the oracle computes a sample of y."""
    x, tg, tu, td = _mlp_case(9, 1, 5376, 21504, 64)
    y = _run_mlp(wl, x, tg, tu, td, torch.bfloat16, gpu)
    cols = np.sort(np.random.default_rng(1).choice(5376, 128, replace=False))
    ref = orc.mlp_geglu(x, tg, tu, td, col=cols)
    assert_parity(y[:, torch.as_tensor(cols, device=gpu)], ref, torch.bfloat16)


# -------------------------------------------------------------- materialize
def _mat_check(wl, orc, th, dev):
    tg = th.to(dev)
    for dt in (torch.float32, torch.bfloat16):
        buf, w, pad = guarded_empty((th.out, th.inp), dt, dev)
        wl.wl_materialize(tg.W0, tg.s, tg.U if th.r else None, tg.V if th.r else None,
                          dt=dt, out=w)
        torch.cuda.synchronize()
        assert_canaries(buf, pad)
        if dt == torch.float32:
            want = orc.materialize_f32(th)
            got = w.cpu().numpy()
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        else:
            want = orc.materialize_bf16(th)
            got = wl_synth.bf16_bits(w)
            assert np.array_equal(got, want)


@pytest.mark.parametrize("r", [0, 1, 3, 32, 33, 128])
def test_materialize_ragged_bitexact(wl, orc, gpu, r):
    _, th = wl_synth.linear_case(50 + r, 1, 264, 70, r)
    _mat_check(wl, orc, th, gpu)


@pytest.mark.parametrize("fam", sorted(SHAPES_1B))
def test_materialize_gemma_shapes_bitexact(wl, orc, gpu, fam):
    n_in, out = SHAPES_1B[fam]
    _, th = wl_synth.linear_case(60, 1, n_in, out, 32)
    _mat_check(wl, orc, th, gpu)


def test_materialize_passthrough_is_original(wl, gpu):
    _, th = wl_synth.linear_case(0, 1, 1152, 1024, 16, kind="passthrough")
    tg = th.to(gpu)
    w = wl.wl_materialize(tg.W0, tg.s, tg.U, tg.V, dt=torch.bfloat16)
    assert torch.equal(w.cpu().view(torch.int16), th.W0.view(torch.int16))
    w32 = wl.wl_materialize(tg.W0, tg.s, tg.U, tg.V, dt=torch.float32)
    assert torch.equal(w32.cpu(), th.W0.float())
