"""Pins for the fp64 CPU oracle: checks against what the pages and mathematics
fix, never against the oracle itself and never against the CUDA library.

Sources (documentation pages of the weightless framework):
* "In-kernel reconstruction", formula section: per-element expansion of y.
* "In-kernel reconstruction", "The GEMM path": s*(x W0^T) + (x V) U^T.
* "Serve and generate with weightless", "Set the fast path on NVIDIA":
  W_eff = s*W0 + U V^T; passthrough reproduces the original weight.
* "What weightless inference costs", "Reconstruction fidelity":
  relative_frobenius_error.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import wl_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_golden(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            d[k] = [float(a) for a in v]
    return d


def _bf(vals, shape):
    return torch.tensor(vals, dtype=torch.float32).reshape(shape).to(torch.bfloat16)


def _golden_case():
    g = _load_golden("linear_tiny.txt")
    T, n_in, out, r = (int(g[k][0]) for k in ("T", "in", "out", "r"))
    x = _bf(g["x"], (T, n_in))
    th = wl_synth.Theta(_bf(g["W0"], (out, n_in)), torch.tensor(g["s"], dtype=torch.float32),
                        _bf(g["U"], (out, r)), _bf(g["V"], (n_in, r)))
    return g, x, th


def f64(t):
    return t.detach().double().cpu().numpy()


# ------------------------------------------------------------ golden -------
def test_golden_linear_exact(orc):
    g, x, th = _golden_case()
    y = orc.linear(x, th)
    assert np.array_equal(y.reshape(-1), np.array(g["y"]))
    yf = orc.linear_factored(x, th)
    assert np.array_equal(yf.reshape(-1), np.array(g["y"]))


def test_golden_weff_and_materialize(orc):
    g, x, th = _golden_case()
    assert np.array_equal(orc.weff(th).reshape(-1), np.array(g["W_eff"]))
    assert np.array_equal(orc.materialize_f32(th).reshape(-1).astype(np.float64),
                          np.array(g["W_eff"]))
    want_bits = wl_synth.bf16_bits(torch.tensor(g["W_eff"]).to(torch.bfloat16))
    assert np.array_equal(orc.materialize_bf16(th).reshape(-1), want_bits)


def test_golden_rel_frobenius(orc):
    g, x, th = _golden_case()
    W = np.array(g["W_eff"]).reshape(th.out, th.inp)
    assert orc.rel_frobenius(W, th) == 0.0
    o, i = (int(a) for a in g["rel_frob_E_at"])
    W[o, i] += 1.0
    assert orc.rel_frobenius(W, th) == pytest.approx(g["rel_frob_E_value"][0], rel=1e-15)


# ------------------------------------------------------- brute force -------
def _brute(x, th):
    """Per-element expansion, pure Python floats (fp64), as on the page."""
    X, W0, U, V = f64(x), f64(th.W0), f64(th.U), f64(th.V)
    s = th.s.double().numpy()
    T, n_in = X.shape
    out, r = U.shape
    y = [[0.0] * out for _ in range(T)]
    for t in range(T):
        for o in range(out):
            a = 0.0
            for i in range(n_in):
                a += float(W0[o, i]) * float(X[t, i])
            d = 0.0
            for k in range(r):
                vx = 0.0
                for i in range(n_in):
                    vx += float(V[i, k]) * float(X[t, i])
                d += float(U[o, k]) * vx
            y[t][o] = float(s[o]) * a + d
    return np.array(y)


@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("n_in,out", [(8, 8), (24, 16), (8, 16)])
@pytest.mark.parametrize("r", [0, 1, 3])
def test_brute_force_tiny(orc, T, n_in, out, r):
    x, th = wl_synth.linear_case(100 + T * 7 + r, T, n_in, out, r)
    y = orc.linear(x, th)
    yb = _brute(x, th)
    scale = np.sqrt(np.mean(yb ** 2)) + 1e-300
    assert np.max(np.abs(y - yb)) <= 1e-13 * scale


# ---------------------------------------------- fp32-encoded bundles -------
# "Serve and generate with weightless", "Supported encodings and devices": the
# architectures also support float32.  The fp32 entry converts every operand
# to fp64 exactly; it is pinned like the bf16 one and tied to it.
@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("n_in,out", [(8, 8), (24, 16)])
@pytest.mark.parametrize("r", [0, 1, 3])
def test_f32_brute_force_tiny(orc, T, n_in, out, r):
    x, th = wl_synth.linear_case_f32(200 + T * 7 + r, T, n_in, out, r)
    y = orc.linear_f32(x, th)
    yb = _brute(x, th)
    scale = np.sqrt(np.mean(yb ** 2)) + 1e-300
    assert np.max(np.abs(y - yb)) <= 1e-13 * scale


def test_f32_degenerate_matches_torch_matmul(orc):
    x, th = wl_synth.linear_case_f32(1, 4, 1152, 256, 4, kind="degenerate")
    y = orc.linear_f32(x, th)
    ref = (x.double() @ th.W0.double().T).numpy()
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.sqrt(np.mean(ref ** 2))


def test_f32_matches_gemm_path_float64(orc):
    """The GEMM-path form s*(x W0^T) + (x V) U^T in torch float64."""
    x, th = wl_synth.linear_case_f32(2, 5, 320, 96, 7)
    y = orc.linear_f32(x, th)
    X, W0, s, U, V = (t.double() for t in (x, th.W0, th.s, th.U, th.V))
    ref = (s[None, :] * (X @ W0.T) + (X @ V) @ U.T).numpy()
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.sqrt(np.mean(ref ** 2))


def test_f32_equals_bf16_entry_on_bf16_values(orc):
    """fp32 operands that are bf16 values give exactly the bf16 entry's result
    (same fp64 values, same order)."""
    x, th = wl_synth.linear_case(3, 3, 64, 40, 5)
    th32 = wl_synth.Theta(th.W0.float(), th.s, th.U.float(), th.V.float())
    assert np.array_equal(orc.linear_f32(x.float(), th32), orc.linear(x, th))


# --------------------------------------------- two independent forms -------
@pytest.mark.parametrize("T,n_in,out,r", [(1, 40, 24, 8), (5, 64, 48, 16), (3, 1152, 64, 4),
                                          (2, 24, 200, 3)])
def test_explicit_equals_factored(orc, T, n_in, out, r):
    x, th = wl_synth.linear_case(7, T, n_in, out, r)
    y = orc.linear(x, th)
    yf = orc.linear_factored(x, th)
    scale = np.sqrt(np.mean(yf ** 2))
    assert np.max(np.abs(y - yf)) <= 1e-12 * scale


def test_degenerate_matches_torch_matmul(orc):
    """U = V = 0, s = 1: y must equal x W0^T (library matmul in float64)."""
    x, th = wl_synth.linear_case(0, 4, 1152, 1024, 4, kind="degenerate")
    y = orc.linear(x, th)
    ref = (x.double() @ th.W0.double().T).numpy()
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.sqrt(np.mean(ref ** 2))


def test_random_matches_torch_float64(orc):
    """Library routine restatement of the GEMM path in float64."""
    x, th = wl_synth.linear_case(0, 4, 1152, 1024, 4)
    y = orc.linear(x, th)
    X, W0, U, V = (t.double() for t in (x, th.W0, th.U, th.V))
    ref = (th.s.double()[None, :] * (X @ W0.T) + (X @ V) @ U.T).numpy()
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.sqrt(np.mean(ref ** 2))


# ------------------------------------------------------- closed forms -------
def test_one_hot_gives_weff_column(orc):
    n_in, out, r = 48, 40, 5
    _, th = wl_synth.linear_case(3, 1, n_in, out, r)
    for i in (0, 17, n_in - 1):
        x = torch.zeros(1, n_in, dtype=torch.bfloat16)
        x[0, i] = 1.0
        y = orc.linear(x, th)[0]
        want = (th.s.double() * th.W0.double()[:, i]
                + th.U.double() @ th.V.double()[i, :]).numpy()
        assert np.max(np.abs(y - want)) <= 1e-15


def test_w0_zero_gives_low_rank_only(orc):
    x, th = wl_synth.linear_case(4, 3, 64, 32, 6)
    th.W0 = torch.zeros_like(th.W0)
    y = orc.linear(x, th)
    ref = ((x.double() @ th.V.double()) @ th.U.double().T).numpy()
    assert np.max(np.abs(y - ref)) <= 1e-13 * np.sqrt(np.mean(ref ** 2))


def test_uv_zero_gives_scaled_w0_term(orc):
    x, th = wl_synth.linear_case(5, 3, 64, 32, 6)
    th.U = torch.zeros_like(th.U)
    th.V = torch.zeros_like(th.V)
    y = orc.linear(x, th)
    ref = (th.s.double()[None, :] * (x.double() @ th.W0.double().T)).numpy()
    assert np.max(np.abs(y - ref)) <= 1e-13 * np.sqrt(np.mean(ref ** 2))


def test_linearity_in_x_and_s(orc):
    x, th = wl_synth.linear_case(6, 3, 64, 32, 6)
    y1 = orc.linear(x, th)
    y2 = orc.linear((x.float() * 2).to(torch.bfloat16), th)
    assert np.array_equal(y2, 2 * y1)          # scaling by 2 is exact
    th0 = wl_synth.Theta(th.W0, th.s, torch.zeros_like(th.U), torch.zeros_like(th.V))
    th2 = wl_synth.Theta(th.W0, th.s * 2, th.U, th.V)
    # only the W0 term scales with s
    d = orc.linear(x, th2) - y1
    assert np.max(np.abs(d - orc.linear(x, th0))) <= 1e-13 * np.sqrt(np.mean(y1 ** 2))


def test_token_rows_independent(orc):
    """Row t of a T-token result equals the 1-token result on that row."""
    x, th = wl_synth.linear_case(8, 6, 96, 40, 4)
    y = orc.linear(x, th)
    for t in range(6):
        assert np.array_equal(orc.linear(x[t:t + 1], th)[0], y[t])
    sel = orc.linear_sel(x, th, tok=[5, 1], col=[39, 0, 7])
    assert np.array_equal(sel, y[np.ix_([5, 1], [39, 0, 7])])


# ------------------------------------------------------------- gelu --------
def test_gelu_tanh_matches_torch(orc):
    v = np.concatenate([np.linspace(-8, 8, 161), [0.0, 1e-8, -1e-8, 30.0, -30.0]])
    want = torch.nn.functional.gelu(torch.tensor(v, dtype=torch.float64),
                                    approximate="tanh").numpy()
    got = np.array([orc.gelu_tanh(a) for a in v])
    assert np.max(np.abs(got - want)) <= 1e-15
    assert orc.gelu_tanh(0.0) == 0.0
    assert orc.gelu_tanh(30.0) == 30.0
    assert abs(orc.gelu_tanh(-30.0)) < 1e-300 or orc.gelu_tanh(-30.0) == 0.0


# ------------------------------------------------------------- MLP ---------
def test_mlp_equals_composition(orc):
    T, hidden, inter, r = 3, 64, 96, 4
    g = wl_synth.make_generator(11)
    x = wl_synth.draw_x(g, T, hidden)
    tg = wl_synth.draw_theta(g, hidden, inter, r)
    tu = wl_synth.draw_theta(g, hidden, inter, r)
    td = wl_synth.draw_theta(g, inter, hidden, r)
    y, h = orc.mlp_geglu(x, tg, tu, td, want_h=True)
    # composition from torch float64 pieces
    def weff(th):
        return th.s.double()[:, None] * th.W0.double() + th.U.double() @ th.V.double().T
    X = x.double()
    gg = X @ weff(tg).T
    uu = X @ weff(tu).T
    hh = torch.nn.functional.gelu(gg, approximate="tanh") * uu
    yy = hh @ weff(td).T
    assert np.max(np.abs(h - hh.numpy())) <= 1e-13 * hh.abs().max().item()
    assert np.max(np.abs(y - yy.numpy())) <= 1e-12 * yy.abs().max().item()
    ys = orc.mlp_geglu(x, tg, tu, td, tok=[2, 0], col=[5, 63])
    assert np.array_equal(ys, y[np.ix_([2, 0], [5, 63])])


# ------------------------------------------------------- materialize -------
def _round_f32(q: Fraction) -> float:
    """Exact rational -> nearest fp32 (ties to even); normal range only."""
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    assert -126 <= e <= 127
    m = a / Fraction(2) ** (e - 23)          # in [2^23, 2^24)
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * float(Fraction(fl) * Fraction(2) ** (e - 23))


def test_round_f32_helper_against_numpy():
    rng = np.random.default_rng(0)
    for v in rng.standard_normal(200):
        assert _round_f32(Fraction(float(v))) == float(np.float32(v))


def test_materialize_f32_fixed_order(orc):
    """Every element recomputed with exact rationals: d = fma chain over k
    ascending, then fl32(s*W0) and fl32(w + d)."""
    n_in, out, r = 32, 24, 16
    _, th = wl_synth.linear_case(9, 1, n_in, out, r)
    got = orc.materialize_f32(th)
    W0, U, V = f64(th.W0), f64(th.U), f64(th.V)
    s = th.s.numpy()
    for o in range(out):
        for i in range(n_in):
            d = 0.0
            for k in range(r):
                d = _round_f32(Fraction(float(U[o, k])) * Fraction(float(V[i, k])) + Fraction(d))
            w = np.float32(s[o]) * np.float32(W0[o, i])
            w = np.float32(w + np.float32(d))
            assert got[o, i] == w, (o, i)


def test_f32_to_bf16_matches_torch(orc):
    rng = np.random.default_rng(2)
    a = rng.standard_normal(4096).astype(np.float32)
    # exact ties and their neighbours
    ties = (np.arange(256, dtype=np.uint32) << 16 | 0x8000).view(np.float32) * 1.0
    a = np.concatenate([a, ties.astype(np.float32), np.float32([0.0, -0.0, 1e-30, 3.4e38])])
    want = wl_synth.bf16_bits(torch.from_numpy(a).to(torch.bfloat16))
    assert np.array_equal(orc.f32_to_bf16(a), want)


def test_materialize_passthrough_bit_exact(orc):
    """G = num_layers: W0 is the original weight, s = 1, U = V = 0, so the
    reconstructed weight must equal the original exactly."""
    _, th = wl_synth.linear_case(0, 1, 1152, 256, 4, kind="passthrough")
    assert np.array_equal(orc.materialize_bf16(th), wl_synth.bf16_bits(th.W0))
    assert np.array_equal(orc.materialize_f32(th), th.W0.float().numpy())
    W = th.W0.double().numpy()
    assert orc.rel_frobenius(W, th) == 0.0
    assert np.array_equal(orc.weff(th), W)


def test_materialize_close_to_fp64(orc):
    _, th = wl_synth.linear_case(12, 1, 256, 128, 32)
    w32 = orc.materialize_f32(th).astype(np.float64)
    w64 = orc.weff(th)
    assert np.max(np.abs(w32 - w64)) <= 2 ** -22 * np.abs(w64).max()


def test_rel_frobenius_closed_form(orc):
    _, th = wl_synth.linear_case(13, 1, 64, 48, 4)
    W = (th.s.double()[:, None] * th.W0.double() + th.U.double() @ th.V.double().T).numpy()
    rng = np.random.default_rng(3)
    E = 1e-3 * rng.standard_normal(W.shape)
    got = orc.rel_frobenius(W + E, th)
    want = np.linalg.norm(E) / np.linalg.norm(W + E)
    assert got == pytest.approx(want, rel=1e-9)


# -------------------------------------------------------- band select ------
def test_band_of_layer(orc):
    L = 26
    assert [orc.band_of_layer(l, L, L) for l in range(L)] == list(range(L))
    assert [orc.band_of_layer(l, L, 1) for l in range(L)] == [0] * L
    for G in (2, 3, 5, 13):
        b = [orc.band_of_layer(l, L, G) for l in range(L)]
        assert b[0] == 0 and b[-1] == G - 1
        assert all(b2 - b1 in (0, 1) for b1, b2 in zip(b, b[1:]))
        sizes = np.bincount(b)
        assert sizes.max() - sizes.min() <= 1
    assert orc.band_of_layer(26, 26, 1) == -1
    assert orc.band_of_layer(0, 26, 27) == -1
    assert orc.band_of_layer(-1, 26, 1) == -1


def _round_bf16_exact(v: float) -> float:
    """Exact rational rounding of a double to 8 significant bits (RNE)."""
    q = Fraction(v)
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    m = a / Fraction(2) ** (e - 7)             # in [2^7, 2^8)
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * float(Fraction(fl) * Fraction(2) ** (e - 7))


def test_f64_to_bf16_exact_rounding(orc):
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-6, 6, 3000),
                        [0.0, -0.0, 1.0, -1.0]])
    # exact midpoints between bf16 neighbours (ties) and one ulp of fp64 off them
    base = (np.arange(1, 200, dtype=np.float64) / 128.0) * 4.0
    mids = base + 2.0 ** -6 * 0.5 * (base / 4.0 >= 1) + 0.0
    v = np.concatenate([v, mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf)])
    got = orc.round_bf16(v)
    want = np.array([_round_bf16_exact(float(a)) for a in v])
    assert np.array_equal(got, want)


def test_f64_to_bf16_agrees_with_torch_on_fp32_values(orc):
    rng = np.random.default_rng(5)
    a32 = rng.standard_normal(5000).astype(np.float32)
    want = wl_synth.bf16_bits(torch.from_numpy(a32).to(torch.bfloat16))
    assert np.array_equal(orc.f64_to_bf16(a32.astype(np.float64)), want)


def test_bf16_error_measure():
    """The bf16 parity measure: correctly rounded outputs score 0, a one-step
    flip next to a rounding midpoint scores about the distance to it, and an
    output two steps off scores about one and a half steps."""
    from tests.parity import bf16_ulp
    import torch as _t
    ref = np.array([1.0 + 2 ** -9, 3.0, 2.0 + 2 ** -7 + 1e-9])
    y_ok = _t.tensor([1.0, 3.0, 2.0 + 2 ** -6]).to(_t.bfloat16)
    yv = y_ok.double().numpy()
    assert np.array_equal(bf16_ulp(np.array([1.0, 3.0, 2.0])), np.array([2 ** -7, 2 ** -6, 2 ** -6]))
    d = np.maximum(0.0, np.abs(yv - ref) - 0.5 * bf16_ulp(yv))
    assert np.max(d) < 1e-8
    y_flip = np.array([1.0, 3.0, 2.0])          # the other side of the midpoint
    d = np.maximum(0.0, np.abs(y_flip - ref) - 0.5 * bf16_ulp(y_flip))
    assert d[2] < 2e-9
    y_bad = np.array([1.0 + 2 * 2 ** -7, 3.0, 2.0])
    d = np.maximum(0.0, np.abs(y_bad - ref) - 0.5 * bf16_ulp(y_bad))
    assert abs(d[0] - (2 * 2 ** -7 - 2 ** -9 - 2 ** -8)) < 1e-12
