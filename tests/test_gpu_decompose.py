"""GPU decomposition (wl_decompose_band) against the decomposition oracle
(oracle/decompose.py) on the same bf16 weights.

What is unique is compared directly: W0 (the band mean, bit-exact for two
layers, whose fp32 sum is exact; within one bf16 step otherwise), s (fp32
least squares), and, where the residual has a clear spectral gap (a planted
rank-r residual), the delta U V^T.  Without a gap the rank-r subspace is not
unique; there the reconstruction must be near the Eckart-Young optimum that
the oracle attains.  The passthrough point (one layer per band) must be
exact: W0 = W, s = 1, U = V = 0 ("Set the fast path on NVIDIA").
"""
import numpy as np
import pytest
import torch

import wl_synth
from tests.parity import bf16_ulp

pytestmark = pytest.mark.gpu


def _f64(t):
    return t.detach().double().cpu().numpy()


def _planted(seed, out, inp, r, n=2):
    """n bf16 weights B + c_l D (c = +1, -1, ...) with D of rank r and the rows
    of B orthogonal to D's row space (the oracle pins' construction)."""
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((inp, r))
    P = rng.standard_normal((out, r))
    Dm = P @ Q.T / np.sqrt(inp)
    Braw = rng.standard_normal((out, inp)) / np.sqrt(inp)
    B = Braw - Braw @ (Q @ np.linalg.solve(Q.T @ Q, Q.T))
    cs = [1.0, -1.0, 0.5, -0.5][:n]
    return [torch.from_numpy(B + c * Dm).to(torch.bfloat16) for c in cs]


@pytest.mark.parametrize("r", [0, 4])
def test_passthrough_exact(wl, gpu, r):
    g = wl_synth.make_generator(3)
    Ws = [wl_synth.draw_theta(g, 200, 72, 0).W0.to(gpu) for _ in range(3)]
    res = wl.decompose(Ws, 3, r)
    torch.cuda.synchronize()
    assert wl.wl_device_status() == wl.WL_OK
    for W, (W0, s, U, V) in zip(Ws, res):
        assert torch.equal(W0, W)
        assert torch.equal(s, torch.ones_like(s))
        assert not U.float().abs().sum() and not V.float().abs().sum()


@pytest.mark.parametrize("out,inp,r,n", [(96, 160, 4, 2), (130, 72, 8, 2), (256, 512, 16, 3), (6912, 1152, 16, 2),
                                         # k = r + p of 48 and 108: the wider Gram forms
                                         (160, 256, 40, 2), (300, 264, 100, 2)])
def test_planted_residual_matches_oracle(wl, orc, gpu, out, inp, r, n):
    from oracle import decompose as D

    Ws = _planted(out + inp + r, out, inp, r, n)
    W0r, sr, Ur, Vr = D.decompose_band(Ws, r)
    W0, s, U, V = wl.wl_decompose_band([W.to(gpu) for W in Ws], r, p=8, iters=4, seed=1)
    torch.cuda.synchronize()
    assert wl.wl_device_status() == wl.WL_OK
    w0 = _f64(W0)
    if n == 2:
        assert np.array_equal(w0, W0r)
    else:
        assert np.all(np.abs(w0 - W0r) <= bf16_ulp(np.abs(W0r)))
    for l in range(n):
        assert np.max(np.abs(_f64(s[l]) - sr[l]) / np.maximum(np.abs(sr[l]), 1e-30)) <= 1e-5
        dg = _f64(U[l]) @ _f64(V[l]).T
        dr = Ur[l] @ Vr[l].T
        assert np.linalg.norm(dg - dr) <= 1e-2 * np.linalg.norm(dr), l
        eg = D.rel_frobenius(Ws[l], W0, s[l], U[l], V[l])
        er = D.rel_frobenius(Ws[l], W0r, sr[l], Ur[l], Vr[l])
        assert abs(eg - er) <= 1e-3, (eg, er)


@pytest.mark.parametrize("out,inp,r", [(256, 512, 8), (1024, 1152, 32)])
def test_flat_spectrum_near_optimal(wl, orc, gpu, out, inp, r):
    """Random weights: no gap, so the subspace is not unique; the residual
    left by the GPU's rank-r delta must be within 5 % of the truncated SVD's
    (Eckart-Young) residual, and never below it beyond bf16 rounding."""
    from oracle import decompose as D

    g = wl_synth.make_generator(out + r)
    Ws = [wl_synth.draw_theta(g, inp, out, 0).W0 for _ in range(2)]
    W0r, sr, Ur, Vr = D.decompose_band(Ws, r)
    W0, s, U, V = wl.wl_decompose_band([W.to(gpu) for W in Ws], r, p=8, iters=4, seed=2)
    torch.cuda.synchronize()
    for l in range(2):
        eg = D.rel_frobenius(Ws[l], W0, s[l], U[l], V[l])
        er = D.rel_frobenius(Ws[l], W0r, sr[l], Ur[l], Vr[l])
        assert eg <= 1.05 * er, (eg, er)
        assert eg >= 0.99 * er, (eg, er)


def test_bands_share_w0(wl, gpu):
    g = wl_synth.make_generator(9)
    Ws = [wl_synth.draw_theta(g, 64, 48, 0).W0.to(gpu) for _ in range(5)]
    res = wl.decompose(Ws, 2, 4)
    for l in range(5):
        for m in range(5):
            same_band = wl.wl_band_of_layer(l, 5, 2) == wl.wl_band_of_layer(m, 5, 2)
            assert (res[l][0].data_ptr() == res[m][0].data_ptr()) == same_band


def test_limits(wl, gpu):
    W = torch.zeros(16, 24, dtype=torch.bfloat16, device=gpu)
    with pytest.raises(wl.WLError):
        wl.wl_decompose_band([W], 17)  # r > min(out, in)
    with pytest.raises(wl.WLError):
        wl.wl_decompose_band([W], 4, p=200)  # r + p > 160
