"""Shared helpers for the GPU parity tests (test code only)."""
import numpy as np
import torch

import oracle
import wl_synth

# Tolerances of the method's parity contract, relative to rms(y_ref) over the
# whole output of a call: bf16 outputs 1e-2 (against the exact result after
# the final round-to-nearest-even cast), fp32 outputs 1e-4.
TOL = {torch.bfloat16: 1e-2, torch.float32: 1e-4}

GEMMA = wl_synth.GEMMA_1B
SHAPES_1B = {  # family: (in, out)
    "q": (1152, 1024), "k": (1152, 256), "v": (1152, 256), "o": (1024, 1152),
    "gate": (1152, 6912), "up": (1152, 6912), "down": (6912, 1152),
}


def to_gpu(th, dev):
    return th.to(dev)


def err_ratio(y_gpu: torch.Tensor, y_ref: np.ndarray, ydt) -> float:
    """max|y_gpu - ref| / rms(y_ref); ref is y_ref after the output cast."""
    y = y_gpu.detach().float().cpu().double().numpy()
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y))
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    ref = oracle.round_bf16(y_ref) if ydt == torch.bfloat16 else y_ref
    if rms == 0.0:
        return 0.0 if np.max(np.abs(y - ref)) == 0.0 else float("inf")
    return float(np.max(np.abs(y - ref)) / rms)


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
