"""Seeded synthetic inputs for the weightless linear projection.

Both the CUDA library's tests/benchmark and the CPU oracle draw their inputs
from here, so the same bits feed both sides.  This module holds none of the
method's arithmetic: it only draws random numbers and rounds them to bf16.

Recipe (value distributions of the theta bundle on the "Serve and generate
with weightless" page: a W0 block, a per-row scale s and a rank-r delta U, V):

* generator: ``torch.Generator(device).manual_seed(seed)``;
* draws are fp32 ``randn`` in the order x, then per projection W0, s, U, V;
* x ~ N(0, 1), W0 ~ N(0, 1/in), s = 1 + 0.1 N(0, 1) (kept fp32),
  U, V ~ N(0, 0.02^2) (0.02 read as the standard deviation);
* bf16 tensors are rounded from fp32 with round-to-nearest-even.

``kind`` selects the special cases of the method:

* ``"random"``       the distributions above;
* ``"degenerate"``   s = 1, U = V = 0 (the map reduces to x W0^T);
* ``"passthrough"``  same values as degenerate: W0 plays the original weight
  W ~ N(0, 1/in), so the reconstructed weight equals the original exactly;
* ``"delta"``        U, V ~ N(0, 0.2^2) (ten times the default): the rank-r
  term (x V) U^T then outweighs the W0 term, so a test of it is not hidden
  under the W0 term's share of the tolerance.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = [
    "Theta",
    "make_generator",
    "draw_x",
    "draw_theta",
    "linear_case",
    "linear_case_f32",
    "draw_x_f32",
    "draw_theta_f32",
    "layer_case",
    "GEMMA_1B",
    "LARGE_SET",
]

# Projection shapes of one decoder layer (hidden, q, kv, intermediate).
GEMMA_1B = dict(hidden=1152, q=1024, kv=256, inter=6912)
LARGE_SET = dict(hidden=5376, q=4096, kv=2048, inter=21504)

FAMILIES = ("q", "k", "v", "o", "gate", "up", "down")


@dataclass
class Theta:
    """One projection's theta bundle (tensors on the generator's device)."""

    W0: torch.Tensor  # [out, in] bf16
    s: torch.Tensor  # [out] fp32
    U: torch.Tensor  # [out, r] bf16
    V: torch.Tensor  # [in, r] bf16
    meta: dict = field(default_factory=dict)

    @property
    def out(self) -> int:
        return self.W0.shape[0]

    @property
    def inp(self) -> int:
        return self.W0.shape[1]

    @property
    def r(self) -> int:
        return self.U.shape[1]

    def to(self, device) -> "Theta":
        return Theta(self.W0.to(device), self.s.to(device), self.U.to(device),
                     self.V.to(device), dict(self.meta))


def make_generator(seed: int, device: str | torch.device = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32, device=gen.device)


def draw_x(gen: torch.Generator, T: int, d: int) -> torch.Tensor:
    """x [T, d] bf16 ~ N(0, 1)."""
    return _randn(gen, (T, d)).to(torch.bfloat16)


def draw_theta(gen: torch.Generator, inp: int, out: int, r: int,
               kind: str = "random") -> Theta:
    """Draw W0, s, U, V in that order."""
    if kind not in ("random", "degenerate", "passthrough", "delta"):
        raise ValueError(f"unknown kind {kind!r}")
    uv = 0.2 if kind == "delta" else 0.02
    W0 = (_randn(gen, (out, inp)) * (1.0 / math.sqrt(inp))).to(torch.bfloat16)
    s = 1.0 + 0.1 * _randn(gen, (out,))
    U = (_randn(gen, (out, r)) * uv).to(torch.bfloat16)
    V = (_randn(gen, (inp, r)) * uv).to(torch.bfloat16)
    if kind in ("degenerate", "passthrough"):
        s = torch.ones_like(s)
        U = torch.zeros_like(U)
        V = torch.zeros_like(V)
    return Theta(W0.contiguous(), s.contiguous(), U.contiguous(), V.contiguous(),
                 {"kind": kind})


def draw_x_f32(gen: torch.Generator, T: int, d: int) -> torch.Tensor:
    """x [T, d] fp32 ~ N(0, 1) (the fp32 encoding of the inputs)."""
    return _randn(gen, (T, d)).contiguous()


def draw_theta_f32(gen: torch.Generator, inp: int, out: int, r: int, kind: str = "random") -> Theta:
    """An fp32-encoded bundle: the distributions of draw_theta, kept in fp32
    ("Serve and generate with weightless": the architectures also support
    float32).  Draw order W0, s, U, V."""
    if kind not in ("random", "degenerate", "delta"):
        raise ValueError(f"unknown kind {kind!r}")
    uv = 0.2 if kind == "delta" else 0.02
    W0 = _randn(gen, (out, inp)) * (1.0 / math.sqrt(inp))
    s = 1.0 + 0.1 * _randn(gen, (out,))
    U = _randn(gen, (out, r)) * uv
    V = _randn(gen, (inp, r)) * uv
    if kind == "degenerate":
        s = torch.ones_like(s)
        U = torch.zeros_like(U)
        V = torch.zeros_like(V)
    return Theta(W0.contiguous(), s.contiguous(), U.contiguous(), V.contiguous(), {"kind": kind, "dtype": "f32"})


def linear_case_f32(seed: int, T: int, inp: int, out: int, r: int, kind: str = "random", device="cpu"):
    """x and one fp32-encoded bundle, drawn in the order x, W0, s, U, V."""
    g = make_generator(seed, device)
    x = draw_x_f32(g, T, inp)
    th = draw_theta_f32(g, inp, out, r, kind)
    return x, th


def linear_case(seed: int, T: int, inp: int, out: int, r: int,
                kind: str = "random", device="cpu"):
    """x and one theta bundle, drawn in the order x, W0, s, U, V."""
    g = make_generator(seed, device)
    x = draw_x(g, T, inp)
    th = draw_theta(g, inp, out, r, kind)
    return x, th


def layer_case(seed: int, T: int, hidden: int, q: int, kv: int, inter: int,
               r: int, kind: str = "random", device="cpu"):
    """x [T, hidden] and the seven projections of one decoder layer.

    Families in draw order: q, k, v (hidden -> q/kv/kv), o (q -> hidden),
    gate, up (hidden -> inter), down (inter -> hidden).
    """
    g = make_generator(seed, device)
    x = draw_x(g, T, hidden)
    shapes = {
        "q": (hidden, q), "k": (hidden, kv), "v": (hidden, kv),
        "o": (q, hidden), "gate": (hidden, inter), "up": (hidden, inter),
        "down": (inter, hidden),
    }
    thetas = {}
    for fam in FAMILIES:
        inp, out = shapes[fam]
        thetas[fam] = draw_theta(g, inp, out, r, kind)
    return x, thetas


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (CPU copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
