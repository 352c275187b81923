"""fp64 CPU oracle for the weightless linear projection -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never imports, links or calls it, and this package never imports the
CUDA library.

The arithmetic lives in ``wl_oracle.c`` (plain C, fp64, OpenMP over output
rows); this module compiles it with gcc on first use (or via :func:`build`)
and wraps it with ctypes over numpy arrays.  bf16 tensors cross as their
uint16 bit patterns, fp32 scales as float32 arrays.

Pinning status (what each function is checked against in ``tests/``):

* ``linear``/``linear_sel``: factored form, brute force, torch float64,
  closed forms, hand-worked golden example -- pinned.
* ``linear_f32`` (fp32-encoded bundles): brute force, torch float64, equal to
  ``linear`` on bf16-representable fp32 inputs -- pinned.
* ``mlp_geglu``: gelu pins + composition from pinned linear pieces -- pinned.
* ``materialize_f32``/``materialize_bf16``: per-element recomputation with
  Python's correctly rounded float ops and numpy float32, passthrough -- pinned.
* ``f64_to_bf16``/``round_bf16``: exact rational rounding, torch's fp32 cast
  on fp32-representable values -- pinned.
* ``rel_frobenius``: zero at passthrough, closed form for an added E -- pinned.
* ``decompose`` (module): W -> theta of a band (mean W0, least-squares s,
  truncated SVD of the residual for U, V) -- pinned by the passthrough point
  (exact), an exactly planted rank-r residual, the Eckart-Young error, the
  normal equations of s and monotonicity in r; planted mistakes fail a pin.
  The mean / least-squares / SVD steps are a reading for G < L (the pages fix
  only the passthrough point).
* ``band_of_layer``: G = L identity, G = 1 constant -- pinned for those G;
  the contiguous-band formula for 1 < G < L is a reading (parity unpinned
  there beyond monotonicity and band sizes).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wl_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liborc.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]


def build(force: bool = False) -> str:
    """Compile wl_oracle.c into oracle/_build/liborc.so with gcc."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _u16p():
    return np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")


def _f32p():
    return np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")


def _f64p():
    return np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def _configure(L):
    i64 = C.c_int64
    vp = C.c_void_p
    L.orc_set_threads.argtypes = [C.c_int]
    L.orc_get_threads.restype = C.c_int
    L.orc_weff.argtypes = [_u16p(), _f32p(), vp, vp, i64, i64, i64, _f64p()]
    L.orc_linear.argtypes = [_u16p(), _u16p(), _f32p(), vp, vp, i64, i64, i64, i64, _f64p()]
    L.orc_linear_sel.argtypes = [_u16p(), _u16p(), _f32p(), vp, vp, i64, i64, i64, i64,
                                 vp, i64, vp, i64, _f64p()]
    L.orc_linear_f64in.argtypes = [_f64p(), _u16p(), _f32p(), vp, vp, i64, i64, i64, i64,
                                   vp, i64, _f64p()]
    L.orc_linear_factored.argtypes = [_u16p(), _u16p(), _f32p(), vp, vp, i64, i64, i64,
                                      i64, _f64p()]
    L.orc_linear_f32w.argtypes = [_f32p(), _f32p(), _f32p(), vp, vp, i64, i64, i64, i64, _f64p()]
    L.orc_gelu_tanh.argtypes = [C.c_double]
    L.orc_gelu_tanh.restype = C.c_double
    L.orc_mlp_geglu.argtypes = ([_u16p()] + [_u16p(), _f32p(), vp, vp] * 3
                                + [i64, i64, i64, i64, vp, i64, vp, i64, _f64p(), vp])
    L.orc_materialize_f32.argtypes = [_u16p(), _f32p(), vp, vp, i64, i64, i64, _f32p()]
    L.orc_materialize_bf16.argtypes = [_u16p(), _f32p(), vp, vp, i64, i64, i64, _u16p()]
    L.orc_f32_to_bf16.argtypes = [_f32p(), i64, _u16p()]
    L.orc_f64_to_bf16.argtypes = [_f64p(), i64, _u16p()]
    L.orc_rel_frobenius.argtypes = [_f64p(), _u16p(), _f32p(), vp, vp, i64, i64, i64]
    L.orc_rel_frobenius.restype = C.c_double
    L.orc_band_of_layer.argtypes = [i64, i64, i64]
    L.orc_band_of_layer.restype = i64
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(C.CDLL(build()))
    return _lib


def _swap_library(path):
    """Test hook: load another build of wl_oracle.c (e.g. a planted mutant)
    in place of the real one; returns the previous handle.  Pass None to
    restore the real library."""
    global _lib
    with _lock:
        prev = _lib
        _lib = _configure(C.CDLL(path)) if path else None
    return prev


# ---------------------------------------------------------------- helpers --
def _bits(a) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 array; return contiguous uint16."""
    try:
        import torch

        if isinstance(a, torch.Tensor):
            assert a.dtype == torch.bfloat16, a.dtype
            return np.ascontiguousarray(
                a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(a)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


def _f32(a) -> np.ndarray:
    try:
        import torch

        if isinstance(a, torch.Tensor):
            return np.ascontiguousarray(a.detach().cpu().float().numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _idx(a):
    if a is None:
        return None, 0
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int64))
    return a, a.size


class _Th:
    """theta as flat arrays (keeps references alive for the call)."""

    def __init__(self, W0, s, U, V):
        self.W0 = _bits(W0)
        self.s = _f32(s)
        self.U = _bits(U)
        self.V = _bits(V)
        self.out, self.inp = self.W0.shape
        self.r = self.U.shape[1] if self.U.ndim == 2 else 0
        assert self.s.shape == (self.out,)
        assert self.U.shape == (self.out, self.r)
        assert self.V.shape == (self.inp, self.r)


def _th(theta):
    if isinstance(theta, _Th):
        return theta
    if isinstance(theta, (tuple, list)):
        return _Th(*theta)
    return _Th(theta.W0, theta.s, theta.U, theta.V)


# ------------------------------------------------------------- public API --
def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


def weff(theta) -> np.ndarray:
    """W_eff = diag(s) W0 + U V^T in fp64, [out, in]."""
    t = _th(theta)
    y = np.empty((t.out, t.inp), np.float64)
    lib().orc_weff(t.W0, t.s, _ptr(t.U), _ptr(t.V), t.out, t.inp, t.r, y)
    return y


def linear(x, theta) -> np.ndarray:
    """y = x W_eff^T in fp64, [T, out] (explicit-W_eff form)."""
    t = _th(theta)
    xb = _bits(x)
    T = xb.shape[0]
    assert xb.shape == (T, t.inp)
    y = np.empty((T, t.out), np.float64)
    lib().orc_linear(xb, t.W0, t.s, _ptr(t.U), _ptr(t.V), T, t.inp, t.out, t.r, y)
    return y


def linear_sel(x, theta, tok=None, col=None) -> np.ndarray:
    """y restricted to tokens ``tok`` and outputs ``col`` (None = all)."""
    t = _th(theta)
    xb = _bits(x)
    T = xb.shape[0]
    ta, nt = _idx(tok)
    ca, no = _idx(col)
    y = np.empty((nt if ta is not None else T, no if ca is not None else t.out), np.float64)
    lib().orc_linear_sel(xb, t.W0, t.s, _ptr(t.U), _ptr(t.V), T, t.inp, t.out, t.r,
                         _ptr(ta), nt, _ptr(ca), no, y)
    return y


def linear_f64in(x64, theta, col=None) -> np.ndarray:
    """y = x64 W_eff^T for an fp64 input (no rounding of x)."""
    t = _th(theta)
    x64 = np.ascontiguousarray(np.asarray(x64, np.float64))
    T = x64.shape[0]
    ca, no = _idx(col)
    y = np.empty((T, no if ca is not None else t.out), np.float64)
    lib().orc_linear_f64in(x64, t.W0, t.s, _ptr(t.U), _ptr(t.V), T, t.inp, t.out, t.r,
                           _ptr(ca), no, y)
    return y


def linear_factored(x, theta) -> np.ndarray:
    """s[None,:] * (x W0^T) + (x V) U^T in fp64 (pinning aid)."""
    t = _th(theta)
    xb = _bits(x)
    T = xb.shape[0]
    y = np.empty((T, t.out), np.float64)
    lib().orc_linear_factored(xb, t.W0, t.s, _ptr(t.U), _ptr(t.V), T, t.inp, t.out, t.r, y)
    return y


def linear_f32(x, theta) -> np.ndarray:
    """y = x W_eff^T in fp64 for an fp32-encoded bundle and fp32 x ("Serve and
    generate with weightless", "Supported encodings and devices"): every fp32
    operand converted to fp64 exactly, then the explicit-W_eff form.
    theta: (W0, s, U, V) fp32 arrays or tensors (U, V may be None when r = 0)."""
    W0, s_, U, V = (theta if isinstance(theta, (tuple, list)) else (theta.W0, theta.s, theta.U, theta.V))
    f = lambda a: np.ascontiguousarray(np.asarray(a.cpu() if hasattr(a, "cpu") else a, dtype=np.float32))
    x = f(x)
    W0, s_ = f(W0), f(s_)
    out, inp = W0.shape
    r = 0 if U is None else int(np.asarray(U.shape)[1])
    Uc = f(U) if r > 0 else None
    Vc = f(V) if r > 0 else None
    T = x.shape[0]
    y = np.zeros((T, out), dtype=np.float64)
    lib().orc_linear_f32w(x, W0, s_, _ptr(Uc), _ptr(Vc), T, inp, out, r, y)
    return y


def gelu_tanh(v: float) -> float:
    return float(lib().orc_gelu_tanh(float(v)))


def mlp_geglu(x, gate, up, down, tok=None, col=None, want_h=False):
    """GeGLU MLP in fp64: y = (gelu_tanh(x Wg^T) * (x Wu^T)) Wd^T."""
    g, u, d = _th(gate), _th(up), _th(down)
    xb = _bits(x)
    T, hidden = xb.shape
    inter = g.out
    assert g.inp == hidden and u.inp == hidden and u.out == inter
    assert d.inp == inter and d.out == hidden
    assert g.r == u.r == d.r
    ta, nt = _idx(tok)
    ca, no = _idx(col)
    nrows = nt if ta is not None else T
    y = np.empty((nrows, no if ca is not None else hidden), np.float64)
    h = np.empty((nrows, inter), np.float64) if want_h else None
    lib().orc_mlp_geglu(xb, g.W0, g.s, _ptr(g.U), _ptr(g.V), u.W0, u.s, _ptr(u.U), _ptr(u.V),
                        d.W0, d.s, _ptr(d.U), _ptr(d.V), T, hidden, inter, g.r,
                        _ptr(ta), nt, _ptr(ca), no, y, _ptr(h))
    return (y, h) if want_h else y


def materialize_f32(theta) -> np.ndarray:
    """Bit-exact fixed-order fp32 W_eff, [out, in] float32."""
    t = _th(theta)
    y = np.empty((t.out, t.inp), np.float32)
    lib().orc_materialize_f32(t.W0, t.s, _ptr(t.U), _ptr(t.V), t.out, t.inp, t.r, y)
    return y


def materialize_bf16(theta) -> np.ndarray:
    """The fp32 value above rounded to bf16 (RNE), as uint16 bits."""
    t = _th(theta)
    y = np.empty((t.out, t.inp), np.uint16)
    lib().orc_materialize_bf16(t.W0, t.s, _ptr(t.U), _ptr(t.V), t.out, t.inp, t.r, y)
    return y


def f32_to_bf16(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, np.float32))
    b = np.empty(a.shape, np.uint16)
    lib().orc_f32_to_bf16(a.reshape(-1), a.size, b.reshape(-1))
    return b


def f64_to_bf16(a) -> np.ndarray:
    """fp64 -> bf16 bits with one correct rounding (RNE)."""
    a = np.ascontiguousarray(np.asarray(a, np.float64))
    b = np.empty(a.shape, np.uint16)
    lib().orc_f64_to_bf16(a.reshape(-1), a.size, b.reshape(-1))
    return b


def round_bf16(a) -> np.ndarray:
    """The fp64 values after the method's final cast to bf16, as float64."""
    return bf16_bits_to_f64(f64_to_bf16(a))


def rel_frobenius(W, theta) -> float:
    """||W - (diag(s) W0 + U V^T)||_F / ||W||_F in fp64."""
    t = _th(theta)
    W = np.ascontiguousarray(np.asarray(W, np.float64))
    assert W.shape == (t.out, t.inp)
    return float(lib().orc_rel_frobenius(W, t.W0, t.s, _ptr(t.U), _ptr(t.V), t.out, t.inp, t.r))


def band_of_layer(layer: int, L: int, G: int) -> int:
    return int(lib().orc_band_of_layer(int(layer), int(L), int(G)))


def bf16_bits_to_f64(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64 (no arithmetic)."""
    b = np.asarray(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
