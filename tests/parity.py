"""Shared helpers for the GPU parity tests (test code only)."""
import numpy as np
import torch

import oracle
import wl_synth

# Tolerances of the method's parity contract, relative to rms(y_ref) over the
# whole output of a call: bf16 outputs 1e-2, fp32 outputs 1e-4 (see err_ratio
# for how the final cast to bf16 is accounted for).
TOL = {torch.bfloat16: 1e-2, torch.float32: 1e-4}

GEMMA = wl_synth.GEMMA_1B
SHAPES_1B = {  # family: (in, out)
    "q": (1152, 1024), "k": (1152, 256), "v": (1152, 256), "o": (1024, 1152),
    "gate": (1152, 6912), "up": (1152, 6912), "down": (6912, 1152),
}


def to_gpu(th, dev):
    return th.to(dev)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at each value of v (v itself a bf16 value)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(a > 0, np.exp2(e - 7.0), 2.0 ** -133)


def err_ratio(y_gpu: torch.Tensor, y_ref: np.ndarray, ydt) -> float:
    """Error of a call's output against the exact (fp64) result, / rms(y_ref).

    fp32 outputs: max |y - y_ref|.
    bf16 outputs: the kernel's fp32 value is only seen after its final cast,
    so the error is the distance from y_ref to the set of values that round
    to the output, max(0, |y - y_ref| - ulp(y)/2).  A correctly rounded output
    scores 0; so does one that lands on the other side of a rounding midpoint
    because its fp32 value sits within accumulation noise of that midpoint.
    """
    y = y_gpu.detach().float().cpu().double().numpy()
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y))
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    d = np.abs(y - y_ref)
    if ydt == torch.bfloat16:
        d = np.maximum(0.0, d - 0.5 * bf16_ulp(y))
    if rms == 0.0:
        return 0.0 if np.max(d) == 0.0 else float("inf")
    return float(np.max(d) / rms)


def assert_parity(y_gpu, y_ref, ydt, what=""):
    e = err_ratio(y_gpu, y_ref, ydt)
    assert e <= TOL[ydt], f"{what}: max err / rms = {e:.3e} > {TOL[ydt]:.0e}"
    return e


def guarded_empty(shape, dtype, dev, pad=4096):
    """An output tensor with canary bands on both sides (checked afterwards)."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad,), -12288.0, dtype=dtype, device=dev)
    return buf, buf[pad:pad + n].view(*shape), pad


def assert_canaries(buf, pad):
    lo = buf[:pad].float().cpu()
    hi = buf[-pad:].float().cpu()
    assert torch.all(lo == -12288.0) and torch.all(hi == -12288.0), "write outside the output"
