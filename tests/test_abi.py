"""CPU checks of the C ABI: the library loads, exports every function the
header declares, and rejects bad arguments before any launch.  No compute
call runs here (there is no GPU on the build machine)."""
import ctypes as C
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wl.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(wl_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_binding_symbols(wl):
    assert _declared() == sorted(wl.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(wl):
    L = wl.lib()
    for name in _declared():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", wl.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (wl_[a-z0-9_]+)$", out, flags=re.M))
    assert set(_declared()) <= exported


def test_header_compiles_as_c(tmp_path):
    c = tmp_path / "use.c"
    c.write_text('#include "wl.h"\nint main(void){return (int)wl_band_of_layer(3, 26, 26) - 3;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                    "-c", str(c), "-o", str(tmp_path / "use.o")], check=True)


def test_version_and_empty_error(wl):
    assert "sm_103a" in wl.wl_version()


def test_band_of_layer_matches_oracle(wl, orc):
    for L in (1, 2, 26, 60):
        for G in range(1, L + 1):
            for l in range(L):
                assert wl.wl_band_of_layer(l, L, G) == orc.band_of_layer(l, L, G)
    assert wl.wl_band_of_layer(0, 26, 0) == -1
    assert wl.wl_band_of_layer(26, 26, 26) == -1
    assert wl.wl_band_of_layer(-1, 26, 2) == -1


def test_mlp_workspace_bytes(wl):
    n = wl.wl_mlp_workspace_bytes(1, 1152, 6912, 32)
    assert n >= 8 * 6912 * 4 and n % 256 == 0
    assert wl.wl_mlp_workspace_bytes(1, 1152, 6913, 32) == 0
    assert wl.wl_mlp_workspace_bytes(0, 1152, 6912, 32) == 0
    assert wl.wl_mlp_workspace_bytes(1, 1152, 6912, 129) == 0


# ---- argument validation (returns before touching the GPU) ---------------
P = 1 << 20  # a fake, aligned device address: never dereferenced here


def _lin(wl, x=P, W0=P, s=P, U=P, V=P, y=P, T=4, n_in=1152, out=1024, r=4, ydt=0):
    L = wl.lib()
    st = L.wl_linear(C.c_void_p(x), C.c_void_p(W0), C.c_void_p(s), C.c_void_p(U), C.c_void_p(V),
                     C.c_void_p(y), T, n_in, out, r, ydt, None)
    return st, L.wl_last_error().decode()


@pytest.mark.parametrize("kw,frag", [
    (dict(T=0), "T must be"),
    (dict(n_in=12), "multiple of 8"),
    (dict(n_in=0), "multiple of 8"),
    (dict(out=0), "out must be"),
    (dict(r=-1), "r must be"),
    (dict(r=129), "r must be"),
    (dict(x=0), "must not be NULL"),
    (dict(y=0), "must not be NULL"),
    (dict(W0=0), "W0 and s"),
    (dict(U=0), "U and V"),
    (dict(x=P + 8), "16-byte aligned"),
    (dict(W0=P + 2), "W0 must be 16-byte"),
    (dict(ydt=7), "dtype"),
])
def test_linear_rejects_bad_arguments(wl, kw, frag):
    st, msg = _lin(wl, **kw)
    assert st == wl.WL_ERR_INVALID_ARG, (st, msg)
    assert frag in msg


def test_rank_zero_allows_null_uv(wl):
    st, msg = _lin(wl, U=0, V=0, r=0)
    # valid arguments: without a GPU the call must fail loudly at the CUDA step,
    # never fall back to anything else
    if not torch.cuda.is_available():
        assert st == wl.WL_ERR_CUDA, (st, msg)


def test_no_gpu_fails_loudly(wl):
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    st, msg = _lin(wl)
    assert st == wl.WL_ERR_CUDA and msg


def test_mlp_rejects_small_or_misaligned_workspace(wl):
    L = wl.lib()
    pr = wl._Proj(P, P, P, P, 6912)
    pd = wl._Proj(P, P, P, P, 1152)
    need = wl.wl_mlp_workspace_bytes(1, 1152, 6912, 4)
    st = L.wl_mlp_geglu_fused(C.c_void_p(P), pr, pr, pd, C.c_void_p(P), 1, 1152, 6912, 4,
                              C.c_void_p(P), need - 1, 0, None)
    assert st == wl.WL_ERR_WORKSPACE
    st = L.wl_mlp_geglu_fused(C.c_void_p(P), pr, pr, pd, C.c_void_p(P), 1, 1152, 6912, 4,
                              C.c_void_p(P + 16), need, 0, None)
    assert st == wl.WL_ERR_WORKSPACE
    bad = wl._Proj(P, P, P, P, 1000)
    st = L.wl_mlp_geglu_fused(C.c_void_p(P), bad, pr, pd, C.c_void_p(P), 1, 1152, 6912, 4,
                              C.c_void_p(P), need, 0, None)
    assert st == wl.WL_ERR_INVALID_ARG


def test_qkv_and_materialize_validation(wl):
    L = wl.lib()
    q = wl._Proj(P, P, P, P, 1024)
    k = wl._Proj(P, P, 0, P, 256)
    st = L.wl_qkv_fused(C.c_void_p(P), q, k, q, C.c_void_p(P), C.c_void_p(P), C.c_void_p(P),
                        1, 1152, 4, 0, None)
    assert st == wl.WL_ERR_INVALID_ARG and "k:" in L.wl_last_error().decode()
    st = L.wl_materialize(C.c_void_p(P), C.c_void_p(P), C.c_void_p(P), C.c_void_p(P),
                          C.c_void_p(P + 4), 64, 64, 4, 0, None)
    assert st == wl.WL_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(wl):
    x = torch.zeros(1, 8, dtype=torch.bfloat16)
    W0 = torch.zeros(8, 8, dtype=torch.bfloat16)
    s = torch.ones(8)
    with pytest.raises(ValueError, match="CUDA"):
        wl.wl_linear(x, W0, s, None, None)
