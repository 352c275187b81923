"""The analytic compression ratio ("What weightless inference costs",
Compression) against the bytes of actual bundles: W0 shared per band, s, U,
V per layer (CPU only)."""
import pytest
import torch

from rank_weight_reconstruction_wl_gb300.metrics import (compression_ratio, dense_bytes, projection_dims,
                                                         theta_bytes)

SMALL = dict(hidden=64, q=32, kv=16, inter=96)


def _counted(layers):
    seen, total = set(), 0
    for th in layers:
        for fam in projection_dims(SMALL):
            t = getattr(th, fam)
            if t.W0.data_ptr() not in seen:
                seen.add(t.W0.data_ptr())
                total += t.W0.numel() * t.W0.element_size()
            for x in (t.s, t.U, t.V):
                total += x.numel() * x.element_size()
    return total


@pytest.mark.parametrize("L,G", [(6, 1), (6, 2), (6, 3), (6, 6), (5, 2)])
@pytest.mark.parametrize("r", [0, 4])
def test_theta_bytes_match_bundles(L, G, r):
    from rank_weight_reconstruction_wl_gb300.stack import build_layers

    layers = build_layers(L, G, 1, SMALL, r, seed=3, device="cpu")
    assert theta_bytes(SMALL, L, G, r) == _counted(layers)
    dense = sum(getattr(layers[0], f).W0.numel() * 2 for f in projection_dims(SMALL)) * L
    assert dense_bytes(SMALL, L) == dense


def test_passthrough_and_trends():
    L = 26
    gemma = dict(hidden=1152, q=1024, kv=256, inter=6912)
    outs = sum(o for _, o in projection_dims(gemma).values())
    mats = sum(o * i for i, o in projection_dims(gemma).values())
    # G = L, r = 0: one W0 per layer plus the fp32 scale vectors
    assert compression_ratio(gemma, L, L, 0) == pytest.approx(1 + 4 * outs / (2 * mats), rel=1e-15)
    # fewer shared blocks and lower rank shrink the bundle
    assert compression_ratio(gemma, L, 1, 4) < compression_ratio(gemma, L, 2, 4) < compression_ratio(gemma, L, 26, 4)
    assert compression_ratio(gemma, L, 1, 4) < compression_ratio(gemma, L, 1, 32)
    with pytest.raises(ValueError):
        theta_bytes(gemma, L, 0, 4)
