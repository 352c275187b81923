"""Pins for the decomposition oracle (oracle/decompose.py): against what the
pages fix (the passthrough point reproduces the original weights exactly and
its relative Frobenius error is 0: "Set the fast path on NVIDIA", "What
weightless inference costs") and against mathematics (an exactly planted
rank-r residual is recovered; the truncated SVD attains the Eckart-Young
error; the least-squares scale satisfies its normal equations; the error
does not grow with the rank).  None compares the oracle with itself or with
the CUDA library.  Planted mistakes in a copy of the oracle must fail a pin.
"""
import numpy as np
import pytest
import torch

import wl_synth


def _weights(seed, L, out, inp):
    g = wl_synth.make_generator(seed)
    return [wl_synth.draw_theta(g, inp, out, 0).W0 for _ in range(L)]


def test_passthrough_reproduces_weights_exactly(orc):
    from oracle import decompose as D

    L, out, inp, r = 3, 40, 64, 4
    Ws = _weights(1, L, out, inp)
    for band in D.band_members(L, L):
        assert len(band) == 1
        W = Ws[band[0]]
        W0, ss, Us, Vs = D.decompose_band([W], r)
        assert np.array_equal(W0, W.double().numpy())
        assert np.array_equal(ss[0], np.ones(out))
        assert not Us[0].any() and not Vs[0].any()
        assert D.rel_frobenius(W, W0, ss[0], Us[0], Vs[0]) == 0.0


def _planted(seed, out, inp, r):
    """W1 = B + D, W2 = B - D with D of rank r and every row of B orthogonal
    to D's row space: band mean B, scales 1, residuals +D and -D."""
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((inp, r))
    P = rng.standard_normal((out, r))
    Dm = P @ Q.T / np.sqrt(inp)
    Braw = rng.standard_normal((out, inp)) / np.sqrt(inp)
    proj = Q @ np.linalg.solve(Q.T @ Q, Q.T)
    B = Braw - Braw @ proj
    return B, Dm, [B + Dm, B - Dm]


@pytest.mark.parametrize("out,inp,r", [(48, 80, 3), (96, 64, 8), (30, 200, 1)])
def test_planted_rank_r_residual_recovered(orc, out, inp, r):
    from oracle import decompose as D

    B, Dm, Ws = _planted(out + inp + r, out, inp, r)
    W0, ss, Us, Vs = D.decompose_band(Ws, r, store=False)
    assert np.max(np.abs(W0 - B)) <= 1e-14 * np.max(np.abs(B))
    for W, s, U, V, sign in zip(Ws, ss, Us, Vs, (1, -1)):
        assert np.max(np.abs(s - 1.0)) <= 1e-12
        assert np.max(np.abs(U @ V.T - sign * Dm)) <= 1e-12 * np.max(np.abs(Dm))
        assert D.rel_frobenius(W, W0, s, U, V) <= 1e-12


@pytest.mark.parametrize("r", [1, 3, 8])
def test_truncation_attains_eckart_young_error(orc, r):
    from oracle import decompose as D

    rng = np.random.default_rng(r)
    R = rng.standard_normal((37, 53))
    U, V, S = D.truncated_svd(R, r)
    err2 = np.linalg.norm(R - U @ V.T) ** 2
    assert abs(err2 - np.sum(S[r:] ** 2)) <= 1e-10 * np.sum(S ** 2)
    # the split is even: U and V carry the same column norms
    assert np.allclose(np.linalg.norm(U, axis=0), np.linalg.norm(V, axis=0), rtol=1e-12)


def test_row_scale_normal_equations(orc):
    from oracle import decompose as D

    rng = np.random.default_rng(5)
    W0 = rng.standard_normal((20, 33))
    W = 0.7 * W0 + 0.3 * rng.standard_normal((20, 33))
    s = D.row_scale(W, W0)
    resid = W - s[:, None] * W0
    assert np.max(np.abs(np.einsum("oi,oi->o", resid, W0))) <= 1e-12 * np.max(np.abs(W0)) ** 2 * 33
    assert np.allclose(D.row_scale(2.5 * W0, W0), 2.5, rtol=1e-14, atol=0)
    W0z = W0.copy()
    W0z[3] = 0.0
    assert D.row_scale(W, W0z)[3] == 1.0


def test_error_non_increasing_in_rank_and_zero_at_full_rank(orc):
    from oracle import decompose as D

    Ws = _weights(7, 3, 24, 40)
    prev = np.inf
    for r in (0, 1, 2, 4, 8, 24):
        W0, ss, Us, Vs = D.decompose_band(Ws, r, store=False)
        e = max(D.rel_frobenius(W, W0, s, U, V) for W, s, U, V in zip(Ws, ss, Us, Vs))
        assert e <= prev + 1e-15
        prev = e
    assert prev <= 1e-12  # rank min(out, in) reconstructs every layer


def test_bands_partition_layers(orc):
    from oracle import decompose as D

    for L in (1, 5, 26):
        for G in range(1, L + 1):
            bands = D.band_members(L, G)
            assert sorted(l for b in bands for l in b) == list(range(L))
            sizes = [len(b) for b in bands]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1


# ------------------------------------------------ planted mistakes -------
@pytest.mark.parametrize("mutant", ["no_sqrt_split", "first_layer_as_mean", "scale_ignored", "smallest_values"])
def test_planted_mistakes_fail_a_pin(orc, monkeypatch, mutant):
    from oracle import decompose as D

    if mutant == "no_sqrt_split":
        def bad(R, r):
            Uf, S, Vt = np.linalg.svd(D._f64(R), full_matrices=False)
            return Uf[:, :r] * S[None, :r], Vt[:r].T * S[None, :r], S
        monkeypatch.setattr(D, "truncated_svd", bad)
    elif mutant == "first_layer_as_mean":
        monkeypatch.setattr(D, "band_mean", lambda Ws: D._f64(Ws[0]))
    elif mutant == "scale_ignored":
        monkeypatch.setattr(D, "row_scale", lambda W, W0: np.ones(D._f64(W).shape[0]))
    else:
        def bad(R, r):
            Uf, S, Vt = np.linalg.svd(D._f64(R), full_matrices=False)
            sq = np.sqrt(S[-r:])
            return Uf[:, -r:] * sq, Vt[-r:].T * sq, S
        monkeypatch.setattr(D, "truncated_svd", bad)
    failed = 0
    for test in (lambda: test_planted_rank_r_residual_recovered(orc, 48, 80, 3),
                 lambda: test_truncation_attains_eckart_young_error(orc, 3),
                 lambda: test_row_scale_normal_equations(orc)):
        try:
            test()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"{mutant} passed every pin"
