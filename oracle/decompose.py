"""Decomposition of dense projection weights into theta bundles, in fp64 --
TEST INFRASTRUCTURE (see the package docstring: only tests, smoke() and the
bench's CPU legs may use it).

The pages describe the decomposition only through its results: the weight
adapter "auto-decomposes" a checkpoint into the theta bundle ("Serve and
generate with weightless", "How the custom architecture loads"); the bundle is
a shared W0 per band of G layers, a per-row scale s and a rank-r delta U V^T
(overview); at the passthrough point G = num_layers "each reconstructed weight
equals the original" ("Set the fast path on NVIDIA"); and fidelity is
relative_frobenius_error = ||W - (diag(s) W0 + U V^T)||_F / ||W||_F ("What
weightless inference costs", "Reconstruction fidelity").  The steps below are
the plainest reading that reaches those results:

  1. W0 of a band = the mean of the band's weights, stored as bf16 (round to
     nearest even), since the bundle stores W0 as bf16;
  2. s of a layer = the per-row least-squares scale against the stored W0,
     s[o] = <W[o], W0[o]> / <W0[o], W0[o]> (1 where the W0 row is zero),
     stored as fp32;
  3. U, V of a layer = the rank-r truncated SVD of the residual
     R = W - diag(s) W0 (Eckart-Young: the best rank-r approximation in the
     Frobenius norm), split evenly: U = U_r sqrt(S_r), V = V_r sqrt(S_r),
     stored as bf16.

At G = L every band holds one layer: W0 = W exactly, s = 1 exactly, R = 0
and U = V = 0, so the reconstruction is exact (the pages' passthrough point).
np.linalg.svd (LAPACK) is the library step of (3).
"""
from __future__ import annotations

import numpy as np
import torch


def _f64(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        return a.detach().to(torch.float64).cpu().numpy()
    return np.asarray(a, dtype=np.float64)


def _bf16(a: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (to nearest even), returned as fp64."""
    from . import f64_to_bf16, bf16_bits_to_f64

    return bf16_bits_to_f64(f64_to_bf16(np.ascontiguousarray(a, dtype=np.float64)))


def band_mean(Ws) -> np.ndarray:
    """Step 1 before storage: the mean of the band's weights (fp64)."""
    M = np.zeros_like(_f64(Ws[0]))
    for W in Ws:
        M += _f64(W)
    return M / len(Ws)


def row_scale(W, W0) -> np.ndarray:
    """Step 2 before storage: per-row least-squares scale of W against W0."""
    W, W0 = _f64(W), _f64(W0)
    num = np.einsum("oi,oi->o", W, W0)
    den = np.einsum("oi,oi->o", W0, W0)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), 1.0)


def truncated_svd(R, r: int):
    """Step 3 before storage: U = U_r sqrt(S_r), V = V_r sqrt(S_r)."""
    R = _f64(R)
    out, inp = R.shape
    if r == 0:
        return np.zeros((out, 0)), np.zeros((inp, 0)), np.linalg.svd(R, compute_uv=False)
    Uf, S, Vt = np.linalg.svd(R, full_matrices=False)
    k = min(r, S.size)
    sq = np.sqrt(S[:k])
    U = np.zeros((out, r))
    V = np.zeros((inp, r))
    U[:, :k] = Uf[:, :k] * sq[None, :]
    V[:, :k] = Vt[:k, :].T * sq[None, :]
    return U, V, S


def decompose_band(Ws, r: int, store: bool = True):
    """Theta of one band: the band's weights Ws (list of [out, in]) ->
    (W0, [s_l], [U_l], [V_l]).  store=True rounds W0, U, V to bf16 and s to
    fp32 as the bundle stores them (values returned as fp64 arrays);
    store=False keeps every step in fp64."""
    M = band_mean(Ws)
    W0 = _bf16(M) if store else M
    ss, Us, Vs = [], [], []
    for W in Ws:
        s = row_scale(W, W0)
        if store:
            s = s.astype(np.float32).astype(np.float64)
        R = _f64(W) - s[:, None] * W0
        U, V, _ = truncated_svd(R, r)
        if store:
            U, V = _bf16(U), _bf16(V)
        ss.append(s)
        Us.append(U)
        Vs.append(V)
    return W0, ss, Us, Vs


def band_members(L: int, G: int):
    """Layers of each of the G bands: layer l belongs to band floor(l G / L)."""
    from . import band_of_layer

    bands = [[] for _ in range(G)]
    for l in range(L):
        bands[band_of_layer(l, L, G)].append(l)
    return bands


def reconstruct(W0, s, U, V) -> np.ndarray:
    """diag(s) W0 + U V^T in fp64."""
    return _f64(s)[:, None] * _f64(W0) + _f64(U) @ _f64(V).T


def rel_frobenius(W, W0, s, U, V) -> float:
    """||W - (diag(s) W0 + U V^T)||_F / ||W||_F in fp64."""
    W = _f64(W)
    return float(np.linalg.norm(W - reconstruct(W0, s, U, V)) / np.linalg.norm(W))
