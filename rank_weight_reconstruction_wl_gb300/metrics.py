"""Analytic size of a weightless model ("What weightless inference costs",
Compression): the theta bundle (W0 + s + U + V over every layer and family)
against the original projection weights it replaces.  Deterministic, no GPU.
"""
from __future__ import annotations


def projection_dims(shapes: dict) -> dict:
    """(in, out) of the seven projection families of a decoder layer."""
    h, q, kv, i = shapes["hidden"], shapes["q"], shapes["kv"], shapes["inter"]
    return {"q": (h, q), "k": (h, kv), "v": (h, kv), "o": (q, h),
            "gate": (h, i), "up": (h, i), "down": (i, h)}


def theta_bytes(shapes: dict, L: int, G: int, r: int, w0_bytes: int = 2, s_bytes: int = 4,
                uv_bytes: int = 2) -> int:
    """Bytes of the bundles of an L-layer model with G shared W0 blocks per
    family: G W0 blocks, and per layer s [out], U [out, r], V [in, r]."""
    if not (1 <= G <= L):
        raise ValueError(f"need 1 <= G <= L, got G={G}, L={L}")
    total = 0
    for inp, out in projection_dims(shapes).values():
        total += G * out * inp * w0_bytes
        total += L * (out * s_bytes + r * (out + inp) * uv_bytes)
    return total


def dense_bytes(shapes: dict, L: int, w_bytes: int = 2) -> int:
    """Bytes of the original (dense) projection weights of L layers."""
    return L * sum(out * inp * w_bytes for inp, out in projection_dims(shapes).values())


def compression_ratio(shapes: dict, L: int, G: int, r: int) -> float:
    """theta bytes / original bytes (lower is better; bf16 W0, U, V, fp32 s,
    bf16 original weights)."""
    return theta_bytes(shapes, L, G, r) / dense_bytes(shapes, L)
