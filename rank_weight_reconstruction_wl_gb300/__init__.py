"""Weightless linear projections on GB300: thin Python binding of libwl.so.

Every function here marshals torch CUDA tensors into the C ABI declared in
``include/wl.h`` and calls it; all arithmetic runs in the library's CUDA
kernels.  There is no Python or CPU fallback: if ``libwl.so`` is missing or a
call fails, an exception is raised.

The weightless projection ("In-kernel reconstruction", formula section):

    y[t,o] = s[o] * sum_i W0[o,i] x[t,i] + sum_k U[o,k] * sum_i V[i,k] x[t,i]

Theta arguments (``q``, ``gate`` ...) are any object with ``W0, s, U, V``
attributes, or a ``(W0, s, U, V)`` tuple.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

__all__ = [
    "WLError", "lib", "library_path", "wl_linear", "wl_qkv_fused", "wl_mlp_workspace_bytes",
    "wl_mlp_geglu_fused", "wl_mlp_geglu_fused_noalloc", "wl_materialize", "wl_decompose_band", "decompose",
    "wl_band_of_layer", "wl_device_status",
    "wl_last_error", "wl_version", "wl_selftest_wait", "WLStack", "EXPORTED_SYMBOLS", "WL_OK", "WL_ERR_INVALID_ARG",
    "WL_ERR_UNSUPPORTED", "WL_ERR_CUDA", "WL_ERR_TIMEOUT", "WL_ERR_WORKSPACE", "WL_ERR_INTERNAL", "WL_MAX_RANK",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libwl.so")

WL_OK, WL_ERR_INVALID_ARG, WL_ERR_UNSUPPORTED, WL_ERR_CUDA, WL_ERR_TIMEOUT, WL_ERR_WORKSPACE, WL_ERR_INTERNAL = range(7)
WL_OUT_BF16, WL_OUT_F32 = 0, 1
WL_MAX_RANK = 128
STATUS_NAMES = {0: "WL_OK", 1: "WL_ERR_INVALID_ARG", 2: "WL_ERR_UNSUPPORTED", 3: "WL_ERR_CUDA",
                4: "WL_ERR_TIMEOUT", 5: "WL_ERR_WORKSPACE", 6: "WL_ERR_INTERNAL"}

# Every function include/wl.h declares.
EXPORTED_SYMBOLS = ("wl_linear", "wl_qkv_fused", "wl_linear_f32", "wl_qkv_fused_f32", "wl_decompose_workspace_bytes",
                    "wl_decompose_band", "wl_mlp_workspace_bytes", "wl_mlp_geglu_fused",
                    "wl_mlp_geglu_fused_noalloc", "wl_materialize", "wl_stack_create", "wl_stack_decode",
                    "wl_stack_destroy", "wl_band_of_layer", "wl_device_status", "wl_last_error", "wl_version", "wl_selftest_wait")


class WLError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class _Proj(C.Structure):
    _fields_ = [("W0", C.c_void_p), ("s", C.c_void_p), ("U", C.c_void_p), ("V", C.c_void_p),
                ("out", C.c_int64)]


class _ProjF32(C.Structure):
    _fields_ = [("W0", C.c_void_p), ("s", C.c_void_p), ("U", C.c_void_p), ("V", C.c_void_p),
                ("out", C.c_int64)]


class _Layer(C.Structure):
    _fields_ = [(n, _Proj) for n in ("q", "k", "v", "o", "gate", "up", "down")]


class _LayerOut(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("yq", "yk", "yv", "yo", "ym")]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib():
    """Load libwl.so (built in-tree by build.py); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libwl.so not found at {_LIB_PATH}; build it with "
                "`python -m rank_weight_reconstruction_wl_gb300.build` (needs nvcc)")
        L = C.CDLL(_LIB_PATH)
        i64, vp, st = C.c_int64, C.c_void_p, C.c_int
        L.wl_linear.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, C.c_int, vp]
        L.wl_linear.restype = st
        L.wl_qkv_fused.argtypes = [vp, _Proj, _Proj, _Proj, vp, vp, vp, i64, i64, i64, C.c_int, vp]
        L.wl_qkv_fused.restype = st
        L.wl_linear_f32.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, C.c_int, vp]
        L.wl_linear_f32.restype = st
        L.wl_qkv_fused_f32.argtypes = [vp, _ProjF32, _ProjF32, _ProjF32, vp, vp, vp, i64, i64, i64, C.c_int, vp]
        L.wl_qkv_fused_f32.restype = st
        L.wl_decompose_workspace_bytes.argtypes = [i64, i64, i64, i64]
        L.wl_decompose_workspace_bytes.restype = C.c_size_t
        L.wl_decompose_band.argtypes = [C.POINTER(C.c_void_p), i64, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp, vp,
                                        C.c_size_t, vp]
        L.wl_decompose_band.restype = st
        L.wl_mlp_workspace_bytes.argtypes = [i64, i64, i64, i64, C.c_int]
        L.wl_mlp_workspace_bytes.restype = C.c_size_t
        L.wl_mlp_geglu_fused.argtypes = [vp, _Proj, _Proj, _Proj, vp, i64, i64, i64, i64, vp,
                                         C.c_size_t, C.c_int, vp]
        L.wl_mlp_geglu_fused.restype = st
        L.wl_mlp_geglu_fused_noalloc.argtypes = [vp, _Proj, _Proj, _Proj, vp, i64, i64, i64, i64,
                                                 C.c_int, vp]
        L.wl_mlp_geglu_fused_noalloc.restype = st
        L.wl_materialize.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, C.c_int, vp]
        L.wl_materialize.restype = st
        L.wl_stack_create.argtypes = [C.POINTER(C.c_void_p), C.POINTER(_Layer), C.POINTER(_LayerOut),
                                      i64, i64, i64, i64]
        L.wl_stack_create.restype = st
        L.wl_stack_decode.argtypes = [vp, vp, vp]
        L.wl_stack_decode.restype = st
        L.wl_stack_destroy.argtypes = [vp]
        L.wl_stack_destroy.restype = None
        L.wl_band_of_layer.argtypes = [i64, i64, i64]
        L.wl_band_of_layer.restype = i64
        L.wl_device_status.argtypes = [vp]
        L.wl_device_status.restype = st
        L.wl_selftest_wait.argtypes = [vp]
        L.wl_selftest_wait.restype = st
        L.wl_last_error.restype = C.c_char_p
        L.wl_version.restype = C.c_char_p
        _lib = L
        return L


# ------------------------------------------------------------ marshalling --
def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _theta(th):
    if isinstance(th, (tuple, list)):
        return tuple(th)
    return th.W0, th.s, th.U, th.V


def _proj(th, inp: int, r: int, name: str):
    W0, s, U, V = _theta(th)
    out = W0.shape[0]
    _need(W0, f"{name}.W0", torch.bfloat16, (out, inp))
    _need(s, f"{name}.s", torch.float32, (out,))
    if r > 0:
        _need(U, f"{name}.U", torch.bfloat16, (out, r))
        _need(V, f"{name}.V", torch.bfloat16, (inp, r))
    return _Proj(W0.data_ptr(), s.data_ptr(), U.data_ptr() if r > 0 else None,
                 V.data_ptr() if r > 0 else None, out)


def _proj_f32(th, inp: int, r: int, name: str):
    W0, s, U, V = _theta(th)
    out = W0.shape[0]
    _need(W0, f"{name}.W0", torch.float32, (out, inp))
    _need(s, f"{name}.s", torch.float32, (out,))
    if r > 0:
        _need(U, f"{name}.U", torch.float32, (out, r))
        _need(V, f"{name}.V", torch.float32, (inp, r))
    return _ProjF32(W0.data_ptr(), s.data_ptr(), U.data_ptr() if r > 0 else None,
                    V.data_ptr() if r > 0 else None, out)


def _rank(th) -> int:
    U = _theta(th)[2]
    return 0 if U is None else int(U.shape[1])


def _ydt(dtype) -> int:
    if dtype in (torch.bfloat16, "bf16"):
        return WL_OUT_BF16
    if dtype in (torch.float32, "f32", "fp32"):
        return WL_OUT_F32
    raise ValueError(f"output dtype must be bfloat16 or float32, got {dtype}")


def _tdt(ydt: int):
    return torch.float32 if ydt == WL_OUT_F32 else torch.bfloat16


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _check(status: int):
    if status != WL_OK:
        raise WLError(status, lib().wl_last_error().decode())


# -------------------------------------------------------------------- API --
def wl_linear(x, W0, s, U, V, y=None, ydt=torch.bfloat16, stream=None):
    """y = s*(x W0^T) + (x V) U^T  (x [T,in] -> y [T,out] bf16/fp32).

    bf16 x and bundle: wl_linear; fp32 x and bundle (the fp32 encoding):
    wl_linear_f32."""
    T, inp = x.shape
    out = W0.shape[0]
    r = 0 if U is None else int(U.shape[1])
    code = _ydt(ydt)
    if x.dtype == torch.float32:
        p = _proj_f32((W0, s, U, V), inp, r, "theta")
        if y is None:
            y = torch.empty(T, out, dtype=_tdt(code), device=x.device)
        _need(x, "x", torch.float32)
        _need(y, "y", _tdt(code), (T, out))
        with torch.cuda.device(x.device):
            _check(lib().wl_linear_f32(_ptr(x), p.W0, p.s, p.U, p.V, _ptr(y), T, inp, out, r, code,
                                       _stream(stream, x.device)))
        return y
    _need(x, "x", torch.bfloat16)
    p = _proj((W0, s, U, V), inp, r, "theta")
    if y is None:
        y = torch.empty(T, out, dtype=_tdt(code), device=x.device)
    _need(y, "y", _tdt(code), (T, out))
    with torch.cuda.device(x.device):
        _check(lib().wl_linear(_ptr(x), p.W0, p.s, p.U, p.V, _ptr(y), T, inp, out, r, code,
                               _stream(stream, x.device)))
    return y


def wl_qkv_fused(x, q, k, v, outs=None, ydt=torch.bfloat16, stream=None):
    """Q/K/V projections of one x in one launch; returns (yq, yk, yv)."""
    T, inp = x.shape
    r = _rank(q)
    code = _ydt(ydt)
    if x.dtype == torch.float32:
        _need(x, "x", torch.float32)
        ps = [_proj_f32(th, inp, r, n) for th, n in ((q, "q"), (k, "k"), (v, "v"))]
        if outs is None:
            outs = tuple(torch.empty(T, p.out, dtype=_tdt(code), device=x.device) for p in ps)
        for o, p, n in zip(outs, ps, ("yq", "yk", "yv")):
            _need(o, n, _tdt(code), (T, p.out))
        with torch.cuda.device(x.device):
            _check(lib().wl_qkv_fused_f32(_ptr(x), ps[0], ps[1], ps[2], _ptr(outs[0]), _ptr(outs[1]),
                                          _ptr(outs[2]), T, inp, r, code, _stream(stream, x.device)))
        return tuple(outs)
    _need(x, "x", torch.bfloat16)
    ps = [_proj(th, inp, r, n) for th, n in ((q, "q"), (k, "k"), (v, "v"))]
    if outs is None:
        outs = tuple(torch.empty(T, p.out, dtype=_tdt(code), device=x.device) for p in ps)
    for o, p, n in zip(outs, ps, ("yq", "yk", "yv")):
        _need(o, n, _tdt(code), (T, p.out))
    with torch.cuda.device(x.device):
        _check(lib().wl_qkv_fused(_ptr(x), ps[0], ps[1], ps[2], _ptr(outs[0]), _ptr(outs[1]),
                                  _ptr(outs[2]), T, inp, r, code, _stream(stream, x.device)))
    return tuple(outs)


def wl_mlp_workspace_bytes(T, hidden, inter, r, ydt=torch.bfloat16) -> int:
    return int(lib().wl_mlp_workspace_bytes(T, hidden, inter, r, _ydt(ydt)))


_ws_cache: dict = {}


def mlp_workspace(T, hidden, inter, r, ydt=torch.bfloat16, device=None) -> torch.Tensor:
    """A zeroed workspace of the right size (cached per device and size)."""
    n = wl_mlp_workspace_bytes(T, hidden, inter, r, ydt)
    if n == 0:
        raise ValueError("invalid MLP sizes")
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    key = (dev.index, n)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = torch.zeros(n + 256, dtype=torch.uint8, device=dev)
        off = (-ws.data_ptr()) % 256
        ws = ws[off:off + n]
        _ws_cache[key] = ws
    return ws


def wl_mlp_geglu_fused(x, gate, up, down, y=None, workspace=None, ydt=torch.bfloat16,
                       stream=None):
    """y = (gelu_tanh(x Wg^T) * (x Wu^T)) Wd^T with every W a weightless projection."""
    T, hidden = x.shape
    r = _rank(gate)
    inter = _theta(gate)[0].shape[0]
    code = _ydt(ydt)
    _need(x, "x", torch.bfloat16)
    pg = _proj(gate, hidden, r, "gate")
    pu = _proj(up, hidden, r, "up")
    pd = _proj(down, inter, r, "down")
    if y is None:
        y = torch.empty(T, hidden, dtype=_tdt(code), device=x.device)
    _need(y, "y", _tdt(code), (T, hidden))
    if workspace is None:
        workspace = mlp_workspace(T, hidden, inter, r, ydt, x.device)
    with torch.cuda.device(x.device):
        _check(lib().wl_mlp_geglu_fused(_ptr(x), pg, pu, pd, _ptr(y), T, hidden, inter, r,
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        code, _stream(stream, x.device)))
    return y


def wl_mlp_geglu_fused_noalloc(x, gate, up, down, y, ydt=torch.bfloat16, stream=None):
    """Same MLP without a caller workspace (library's built-in 4 MiB scratch),
    for callers that cannot allocate device memory.  `y` must be given."""
    T, hidden = x.shape
    r = _rank(gate)
    inter = _theta(gate)[0].shape[0]
    code = _ydt(ydt)
    _need(x, "x", torch.bfloat16)
    pg = _proj(gate, hidden, r, "gate")
    pu = _proj(up, hidden, r, "up")
    pd = _proj(down, inter, r, "down")
    _need(y, "y", _tdt(code), (T, hidden))
    with torch.cuda.device(x.device):
        _check(lib().wl_mlp_geglu_fused_noalloc(_ptr(x), pg, pu, pd, _ptr(y), T, hidden, inter, r,
                                                code, _stream(stream, x.device)))
    return y


def wl_materialize(W0, s, U, V, dt=torch.bfloat16, out=None, stream=None):
    """W_eff = s*W0 + U V^T, bit-exact fixed fp32 order, as bf16 or fp32."""
    o, inp = W0.shape
    r = 0 if U is None else int(U.shape[1])
    code = _ydt(dt)
    p = _proj((W0, s, U, V), inp, r, "theta")
    if out is None:
        out = torch.empty(o, inp, dtype=_tdt(code), device=W0.device)
    _need(out, "W_eff", _tdt(code), (o, inp))
    with torch.cuda.device(W0.device):
        _check(lib().wl_materialize(p.W0, p.s, p.U, p.V, _ptr(out), o, inp, r, code,
                                    _stream(stream, W0.device)))
    return out


def wl_decompose_band(Ws, r, p=8, iters=4, omega=None, seed=0, stream=None):
    """The theta bundle of one band: Ws (list of n bf16 [out, in] weights of
    one projection family, sharing one W0) -> (W0 [out, in] bf16, s [n, out]
    fp32, U [n, out, r] bf16, V [n, in, r] bf16).  omega [in, r + p] fp32 is
    the Gaussian start of the subspace iteration (drawn from `seed` when not
    given).  The binding allocates the outputs and the workspace; the library
    call allocates nothing."""
    n = len(Ws)
    out, inp = Ws[0].shape
    dev = Ws[0].device
    for i, W in enumerate(Ws):
        _need(W, f"Ws[{i}]", torch.bfloat16, (out, inp))
    k = r + p
    if omega is None:
        g = torch.Generator(device=dev)
        g.manual_seed(int(seed))
        omega = torch.randn(inp, k, generator=g, device=dev, dtype=torch.float32)
    if r > 0:
        _need(omega, "omega", torch.float32, (inp, k))
    W0 = torch.empty(out, inp, dtype=torch.bfloat16, device=dev)
    s = torch.empty(n, out, dtype=torch.float32, device=dev)
    U = torch.empty(n, out, r, dtype=torch.bfloat16, device=dev)
    V = torch.empty(n, inp, r, dtype=torch.bfloat16, device=dev)
    # 0 for sizes the library rejects: the call below then reports why
    nb = int(lib().wl_decompose_workspace_bytes(out, inp, r, p))
    ws = torch.empty(nb + 256, dtype=torch.uint8, device=dev)
    off = (-ws.data_ptr()) % 256
    ptrs = (C.c_void_p * n)(*[W.data_ptr() for W in Ws])
    with torch.cuda.device(dev):
        _check(lib().wl_decompose_band(ptrs, n, out, inp, r, p, iters, _ptr(omega) if r > 0 else None, _ptr(W0),
                                       _ptr(s), _ptr(U) if r > 0 else None, _ptr(V) if r > 0 else None,
                                       C.c_void_p(ws.data_ptr() + off), nb, _stream(stream, dev)))
    return W0, s, U, V


def decompose(Ws, G, r, p=8, iters=4, seed=0, stream=None):
    """Theta bundles of a family's L dense weights with G shared W0 blocks:
    layer l uses block wl_band_of_layer(l, L, G).  Returns a list of L
    (W0, s, U, V) tuples; layers of a band share their W0 tensor."""
    L = len(Ws)
    bands = [[] for _ in range(G)]
    for l in range(L):
        bands[wl_band_of_layer(l, L, G)].append(l)
    res = [None] * L
    for b, members in enumerate(bands):
        W0, s, U, V = wl_decompose_band([Ws[l] for l in members], r, p, iters, seed=seed + b, stream=stream)
        for j, l in enumerate(members):
            res[l] = (W0, s[j], U[j], V[j])
    return res


class WLStack:
    """A stack of weightless decoder layers run by one launch per step
    (wl_stack_create / wl_stack_decode).

    layers: objects with q, k, v, o, gate, up, down theta bundles (all bf16
    W0, U, V and fp32 s on one device).  The stack owns one set of bf16 output
    buffers per layer, ``outs[l] = {"yq", "yk", "yv", "yo", "ym"}``;
    ``decode(x)`` writes all of them and returns ``outs[-1]["ym"]``.
    Raises WLError (WL_ERR_UNSUPPORTED) for sizes the stack kernels do not
    take (T > 32, r > 32, hidden / q.out / gate.out not multiples of 64).
    """

    def __init__(self, layers, T: int, device=None):
        self.dev = torch.device(device) if device is not None else layers[0].q.W0.device
        self.T = int(T)
        th0 = layers[0]
        self.hidden = int(th0.q.W0.shape[1])
        self.r = _rank(th0.q)
        qd, kd, vd = th0.q.W0.shape[0], th0.k.W0.shape[0], th0.v.W0.shape[0]
        inter = th0.gate.W0.shape[0]
        h, r = self.hidden, self.r
        L = len(layers)
        z = dict(dtype=torch.bfloat16, device=self.dev)
        self.outs = [{"yq": torch.empty(T, qd, **z), "yk": torch.empty(T, kd, **z),
                      "yv": torch.empty(T, vd, **z), "yo": torch.empty(T, h, **z),
                      "ym": torch.empty(T, h, **z)} for _ in range(L)]
        self._layers = (_Layer * L)()
        self._louts = (_LayerOut * L)()
        self._keep = layers  # the stack refers to the layers' device memory
        for l, th in enumerate(layers):
            ly = self._layers[l]
            ly.q = _proj(th.q, h, r, f"layer {l} q")
            ly.k = _proj(th.k, h, r, f"layer {l} k")
            ly.v = _proj(th.v, h, r, f"layer {l} v")
            ly.o = _proj(th.o, qd, r, f"layer {l} o")
            ly.gate = _proj(th.gate, h, r, f"layer {l} gate")
            ly.up = _proj(th.up, h, r, f"layer {l} up")
            ly.down = _proj(th.down, inter, r, f"layer {l} down")
            o = self.outs[l]
            self._louts[l] = _LayerOut(o["yq"].data_ptr(), o["yk"].data_ptr(), o["yv"].data_ptr(),
                                       o["yo"].data_ptr(), o["ym"].data_ptr())
        self._h = C.c_void_p()
        with torch.cuda.device(self.dev):
            _check(lib().wl_stack_create(C.byref(self._h), self._layers, self._louts, L, self.T, h, r))

    @property
    def out(self) -> torch.Tensor:
        return self.outs[-1]["ym"]

    def decode(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        _need(x, "x", torch.bfloat16, (self.T, self.hidden))
        with torch.cuda.device(self.dev):
            _check(lib().wl_stack_decode(self._h, _ptr(x), _stream(stream, self.dev)))
        return self.out

    def close(self):
        if self._h:
            lib().wl_stack_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def wl_band_of_layer(layer: int, L: int, G: int) -> int:
    return int(lib().wl_band_of_layer(layer, L, G))


def wl_device_status(stream=None, device=None) -> int:
    """Synchronise and return (and clear) the device status code."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        return int(lib().wl_device_status(_stream(stream, dev)))


def wl_selftest_wait(stream=None, device=None):
    """Launch the diagnostic kernel whose bounded wait gives up (about 2 s);
    the next wl_device_status() reports WL_ERR_TIMEOUT."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        _check(lib().wl_selftest_wait(_stream(stream, dev)))


def wl_last_error() -> str:
    return lib().wl_last_error().decode()


def wl_version() -> str:
    return lib().wl_version().decode()
