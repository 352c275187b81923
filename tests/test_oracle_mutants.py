"""The pins must be strong enough to catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/wl_oracle.c (CPU only:
a dropped term, a wrong sign, a transposed or wrong index, a wrong constant,
a changed rounding or summation order), builds it with the oracle's own gcc
flags, runs every pin in tests/test_oracle_pins.py against it, and requires at
least one pin to fail.
"""
import inspect
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "wl_oracle.c")

MUTANTS = {
    "drop_delta": ("w += bf(U[o * r + k]) * bf(V[i * r + k]);", "w += 0.0;"),
    "delta_sign": ("w += bf(U[o * r + k]) * bf(V[i * r + k]);",
                   "w -= bf(U[o * r + k]) * bf(V[i * r + k]);"),
    "V_transposed": ("w += bf(U[o * r + k]) * bf(V[i * r + k]);",
                     "w += bf(U[o * r + k]) * bf(V[k * in + i]);"),
    "U_row0": ("w += bf(U[o * r + k]) * bf(V[i * r + k]);", "w += bf(U[k]) * bf(V[i * r + k]);"),
    "drop_s": ("double w = (double)s[o] * bf(W0[o * in + i]);", "double w = bf(W0[o * in + i]);"),
    "s_on_delta": ("row[i] = w;", "row[i] = w + (s[o] - 1.0) * (w - (double)s[o] * bf(W0[o * in + i]));"),
    "x_token0": ("acc += bf(x[t * in + i]) * row[i];", "acc += bf(x[i]) * row[i];"),
    "gelu_const": ("0.044715", "0.04715"),
    "gelu_on_up": ("h[a] = orc_gelu_tanh(g[a]) * u[a];", "h[a] = g[a] * orc_gelu_tanh(u[a]);"),
    # (an unfused d + U*V chain is an equivalent mutant: a bf16 x bf16 product
    # is exact in fp32, so it is not listed)
    "mat_fused_final": ("float w = s[o] * bf_f32(W0[o * in + i]);\n            if (r > 0) w = w + d;\n            Weff[o * in + i] = w;",
                        "float w = fmaf(s[o], bf_f32(W0[o * in + i]), d);\n            Weff[o * in + i] = w;"),
    "mat_k_descending": ("for (int64_t k = 0; k < r; ++k)\n                d = fmaf(bf_f32(U[o * r + k]), bf_f32(V[i * r + k]), d);",
                         "for (int64_t k = r - 1; k >= 0; --k)\n                d = fmaf(bf_f32(U[o * r + k]), bf_f32(V[i * r + k]), d);"),
    "bf16_ties_away": ("u += 0x7fffu + lsb;", "u += 0x8000u;"),
    "f64_bf16_truncate": ("u += (1ull << 44) - 1ull + lsb;", "u += 0ull;"),
    "band_round": ("return (l * G) / L;", "return (l * G + L - 1) / L;"),
    "frob_no_sqrt": ("return sqrt(num) / sqrt(den);", "return num / den;"),
}


def _pin_functions():
    fns = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = list(inspect.signature(fn).parameters)
        marks = getattr(fn, "pytestmark", [])
        grids = [m.args for m in marks if m.name == "parametrize"]
        if not grids:
            fns.append((name, fn, [{}]))
            continue
        combos = [{}]
        for argnames, values in grids:
            names = [a.strip() for a in argnames.split(",")]
            new = []
            for c in combos:
                for v in values:
                    v = v if len(names) > 1 else (v,)
                    new.append({**c, **dict(zip(names, v))})
            combos = new
        fns.append((name, fn, combos))
    return fns


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path, orc):
    old, new = MUTANTS[mutant]
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {mutant} no longer in the oracle"
    msrc = src.replace(old, new)
    cfile = tmp_path / "mut.c"
    cfile.write_text(msrc)
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(cfile), "-o", str(so), "-lm"], check=True)
    caught = []
    prev = oracle._swap_library(str(so))
    try:
        for name, fn, combos in _pin_functions():
            for kw in combos:
                args = {k: v for k, v in kw.items()}
                if "orc" in inspect.signature(fn).parameters:
                    args["orc"] = oracle
                try:
                    fn(**args)
                except AssertionError:
                    caught.append(name)
                    break
    finally:
        oracle._swap_library(None)
    assert caught, f"no pin caught mutant {mutant}"
