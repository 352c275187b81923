"""The precompute path ("Serve and generate with weightless", fast path):
W_eff materialised once (bf16) and run as a dense projection of rank 0,
against the oracle of the original bundle (one bf16 rounding of W_eff stays
inside the bf16 bar)."""
import pytest
import torch

import wl_synth
from tests.parity import SHAPES_1B, assert_parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fam", ["q", "o", "gate", "down"])
@pytest.mark.parametrize("T", [1, 300])
def test_materialized_dense_projection(wl, orc, gpu, fam, T):
    n_in, out = SHAPES_1B[fam]
    x, th = wl_synth.linear_case(70 + T, T, n_in, out, 16)
    tg = th.to(gpu)
    w = wl.wl_materialize(tg.W0, tg.s, tg.U, tg.V, dt=torch.bfloat16)
    y = wl.wl_linear(x.to(gpu), w, torch.ones(out, device=gpu), None, None)
    torch.cuda.synchronize()
    assert_parity(y, orc.linear(x, th), torch.bfloat16, f"{fam} T={T}")


def test_materialized_stack(wl, orc, gpu):
    """Two Gemma-1B layers through the stack kernel with materialised weights."""
    from rank_weight_reconstruction_wl_gb300.stack import build_layers, materialize_layers

    shapes = dict(hidden=1152, q=1024, kv=256, inter=6912)
    layers = build_layers(2, 2, 1, shapes, 4, seed=31, device=gpu)
    dense = materialize_layers(layers)
    stk = wl.WLStack(dense, 1, device=gpu)
    x = torch.randn(1, 1152, generator=torch.Generator(device=gpu).manual_seed(2), device=gpu).to(torch.bfloat16)
    stk.decode(x)
    torch.cuda.synchronize()
    assert wl.wl_device_status() == wl.WL_OK
    cpu = lambda t: t.detach().cpu()
    tc = lambda t: wl_synth.Theta(cpu(t.W0), cpu(t.s), cpu(t.U), cpu(t.V))
    xin = cpu(x)
    for l, th in enumerate(layers):
        o = stk.outs[l]
        assert_parity(o["yq"], orc.linear(xin, tc(th.q)), torch.bfloat16, f"layer {l} q")
        assert_parity(o["yo"], orc.linear(cpu(o["yq"]), tc(th.o)), torch.bfloat16, f"layer {l} o")
        ref = orc.mlp_geglu(cpu(o["yo"]), tc(th.gate), tc(th.up), tc(th.down))
        assert_parity(o["ym"], ref, torch.bfloat16, f"layer {l} mlp")
        xin = cpu(o["ym"])
