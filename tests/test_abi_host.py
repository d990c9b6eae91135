"""The C-ABI library on the host: it builds, loads, exports every declared symbol, and
rejects bad arguments before any CUDA call (so these run without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

from efficient_transformer_gb300 import build as la_build
from efficient_transformer_gb300 import la

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    la_build.build()
    return la.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"\b(la_[A-Za-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_headers_declare_entry_points():
    names = declared_functions()
    for required in ("la_fwd", "la_bwd", "la_workspace_size", "la_get_status", "la_status_str"):
        assert required in names


@pytest.mark.parametrize("name", declared_functions())
def test_symbol_exported(lib, name):
    assert getattr(lib, name) is not None


def test_status_strings(lib):
    for code in range(7):
        assert lib.la_status_str(code)
    assert lib.la_status_str(99) == b"unknown status"


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails its checks
MISALIGNED = ctypes.c_void_p(0x10008)


def fwd_call(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, Hq=4, Hkv=2, N=64, D=64, dt=la.LA_BF16,
             causal=1, phi=0, eps=1e-6, cw=None, sw=None, ws=None, ws_bytes=0, stream=None)
    a.update(over)
    return lib.la_fwd(a["q"], a["k"], a["v"], a["out"], a["B"], a["Hq"], a["Hkv"], a["N"], a["D"],
                      a["dt"], a["causal"], a["phi"], a["eps"], a["cw"], a["sw"], a["ws"],
                      a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(q=None), la.LA_ERR_ARG),
    (dict(out=None), la.LA_ERR_ARG),
    (dict(B=0), la.LA_ERR_ARG),
    (dict(N=-1), la.LA_ERR_ARG),
    (dict(Hq=3), la.LA_ERR_ARG),              # not a multiple of Hkv (gqa rule)
    (dict(Hkv=0), la.LA_ERR_ARG),
    (dict(eps=-1.0), la.LA_ERR_ARG),
    (dict(eps=float("inf")), la.LA_ERR_ARG),
    (dict(eps=float("nan")), la.LA_ERR_ARG),
    (dict(dt=7), la.LA_ERR_ARG),
    (dict(phi=5), la.LA_ERR_ARG),
    (dict(cw=FAKE), la.LA_ERR_ARG),           # one weight without the other
    (dict(D=48), la.LA_ERR_UNSUPPORTED),
    (dict(D=256), la.LA_ERR_UNSUPPORTED),
    (dict(k=MISALIGNED), la.LA_ERR_ALIGN),
    (dict(ws=None, ws_bytes=0), la.LA_ERR_WORKSPACE),
    (dict(ws=FAKE, ws_bytes=16), la.LA_ERR_WORKSPACE),
])
def test_fwd_rejects(lib, over, code):
    assert fwd_call(lib, **over) == code


def test_bwd_rejects(lib):
    args = [FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 1, 4, 2, 64, 64, la.LA_BF16, 1, 0, 1e-6,
            None, None, None, 0, None]
    assert lib.la_bwd(*args) == la.LA_ERR_ARG      # grad_out missing
    args[3] = FAKE
    assert lib.la_bwd(*args) == la.LA_ERR_WORKSPACE


def test_workspace_sizes(lib):
    f = lib.la_workspace_size(1, 32, 8, 65536, 128, la.LA_BF16, 1, 0, 0)
    b = lib.la_workspace_size(1, 32, 8, 65536, 128, la.LA_BF16, 1, 0, 1)
    assert 0 < f < b
    # the backward keeps two float32 values per query row on top of its states
    assert b >= 2 * 4 * 32 * 65536
    assert lib.la_workspace_size(1, 3, 2, 64, 64, la.LA_BF16, 1, 0, 0) == 0     # invalid
    # deterministic plan
    assert f == lib.la_workspace_size(1, 32, 8, 65536, 128, la.LA_BF16, 1, 0, 0)
    # the causal tensor-core backward also holds a bf16 row of phi(q)/den per query position
    # (written by its dq kernel for its dk/dv kernel); the bidirectional one does not
    assert lib.la_kernel_path(1, 32, 8, 65536, 128, la.LA_BF16, 1, 0, 1) == la.LA_PATH_TCGEN05
    bidir = lib.la_workspace_size(1, 32, 8, 65536, 128, la.LA_BF16, 0, 0, 1)
    assert b - bidir >= 32 * 65536 * 128 * 2
    # the float32 (CUDA-core) backward keeps no such array
    b32 = lib.la_workspace_size(1, 32, 8, 65536, 128, la.LA_F32, 1, 0, 1)
    assert b32 < 32 * 65536 * 128 * 2


def test_tensor_core_shapes(lib):
    """bf16 without position weights runs the tensor-core kernels, forward and backward, at
    D = 64 and 128 for every n_rep in {1, 2, 4, 8} (D = 128 with n_rep 1 or 2 on tiles of a
    larger group, rows masked), with cos/sin weights too (two passes); other head dimensions
    and n_rep values do not."""
    for D in (64, 128):
        for n_rep in (1, 2, 4, 8):
            for causal in (0, 1):
                for is_bwd in (0, 1):
                    assert lib.la_kernel_path(2, 8 * n_rep, 8, 3000, D, la.LA_BF16, causal, 0, is_bwd) == \
                        la.LA_PATH_TCGEN05, (D, n_rep, causal, is_bwd)
    for is_bwd in (0, 1):
        assert lib.la_kernel_path(1, 3, 1, 512, 64, la.LA_BF16, 1, 0, is_bwd) == la.LA_PATH_SIMT   # n_rep 3
        assert lib.la_kernel_path(1, 16, 1, 512, 64, la.LA_BF16, 1, 0, is_bwd) == la.LA_PATH_SIMT  # n_rep 16
        assert lib.la_kernel_path(1, 4, 4, 512, 32, la.LA_BF16, 1, 0, is_bwd) == la.LA_PATH_SIMT   # D = 32
    # cos/sin weights: tensor cores too (two passes, one per term)
    for is_bwd in (0, 1):
        assert lib.la_kernel_path(2, 16, 16, 8192, 128, la.LA_BF16, 1, 1, is_bwd) == la.LA_PATH_TCGEN05


def test_float32_always_takes_simt(lib):
    assert lib.la_kernel_path(1, 2, 2, 256, 32, la.LA_F32, 1, 0, 0) == la.LA_PATH_SIMT
    assert lib.la_kernel_path(1, 32, 8, 65536, 128, la.LA_F32, 1, 0, 1) == la.LA_PATH_SIMT


def test_python_binding_phi_codes():
    assert la._phi_code("identity") == 2
    with pytest.raises(NotImplementedError):
        la._phi_code("softmax_free")
    with pytest.raises(ValueError):
        la._phi_code("gelu")


def test_bwd_from_fwd_argument_errors(lib):
    """la_bwd_from_fwd checks its arguments like la_bwd, and needs the forward's workspace."""
    i, f = ctypes.c_int, ctypes.c_float
    base = [FAKE] * 7 + [i(1), i(4), i(2), i(64), i(64), i(la.LA_BF16), i(1), i(0), f(1e-6), None, None]
    # no forward workspace
    assert lib.la_bwd_from_fwd(*(base + [None, ctypes.c_size_t(0), FAKE, ctypes.c_size_t(1 << 30), None])) == la.LA_ERR_ARG
    # a forward workspace but no backward workspace
    assert lib.la_bwd_from_fwd(*(base + [FAKE, ctypes.c_size_t(1 << 30), None, ctypes.c_size_t(0), None])) == la.LA_ERR_WORKSPACE
    # Hq not a multiple of Hkv
    bad = list(base)
    bad[8] = i(3)
    assert lib.la_bwd_from_fwd(*(bad + [FAKE, ctypes.c_size_t(1 << 30), FAKE, ctypes.c_size_t(1 << 30), None])) == la.LA_ERR_ARG


def test_strided_argument_errors(lib):
    """la_fwd_strided / la_bwd_strided reject negative strides (LA_ERR_ARG) and, on the
    tensor-core path, strides that are not multiples of 8 elements (LA_ERR_ALIGN), before any
    CUDA call."""
    i, f, sz = ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    S = la.LaStrides
    neg = S(-1, 64 * 64, 64)
    odd = S(4 * 64 * 64, 64 * 64 + 4, 64)
    shape = [i(1), i(4), i(2), i(64), i(64), i(la.LA_BF16), i(1), i(0), f(1e-6), None, None]
    assert lib.la_kernel_path(1, 4, 2, 64, 64, la.LA_BF16, 1, 0, 0) == la.LA_PATH_TCGEN05

    def fwd(sq, sk):
        return lib.la_fwd_strided(*([FAKE] * 4 + shape + [sq, sk, None, FAKE, sz(1 << 30), None]))

    assert fwd(ctypes.byref(neg), None) == la.LA_ERR_ARG
    assert fwd(None, ctypes.byref(odd)) == la.LA_ERR_ALIGN

    def bwd(sg):
        return lib.la_bwd_strided(*([FAKE] * 7 + shape + [None, None, None, sg, None, sz(0), FAKE, sz(1 << 30), None]))

    assert bwd(ctypes.byref(neg)) == la.LA_ERR_ARG
    assert bwd(ctypes.byref(odd)) == la.LA_ERR_ALIGN


def test_value_width_entry_points(lib):
    """la_*_v: a value width Dv of its own.  Dv = D is the plain call (same plan, same
    workspace, same kernel family); Dv != D runs on the CUDA cores; Dv outside {32, 64, 128}
    is unsupported and checked before any CUDA call."""
    for D in (32, 64, 128):
        for is_bwd in (0, 1):
            assert lib.la_workspace_size_v(1, 8, 2, 3000, D, D, la.LA_BF16, 1, 0, is_bwd) == \
                lib.la_workspace_size(1, 8, 2, 3000, D, la.LA_BF16, 1, 0, is_bwd)
            assert lib.la_kernel_path_v(1, 8, 2, 3000, D, D, la.LA_BF16, 1, 0, is_bwd) == \
                lib.la_kernel_path(1, 8, 2, 3000, D, la.LA_BF16, 1, 0, is_bwd)
            for Dv in (32, 64, 128):
                if Dv != D:
                    assert lib.la_kernel_path_v(1, 8, 2, 3000, D, Dv, la.LA_BF16, 1, 0, is_bwd) == la.LA_PATH_SIMT
                    assert lib.la_workspace_size_v(1, 8, 2, 3000, D, Dv, la.LA_BF16, 1, 0, is_bwd) > 0
    # the states hold D (Dv + 1) floats per segment: a wider value grows the workspace
    assert lib.la_workspace_size_v(1, 8, 2, 3000, 64, 128, la.LA_F32, 1, 0, 0) > \
        lib.la_workspace_size_v(1, 8, 2, 3000, 64, 32, la.LA_F32, 1, 0, 0)
    for Dv in (0, -1):
        assert lib.la_workspace_size_v(1, 8, 2, 64, 64, Dv, la.LA_F32, 1, 0, 0) == 0
    assert lib.la_workspace_size_v(1, 8, 2, 64, 64, 48, la.LA_F32, 1, 0, 0) == 0
    fake = ctypes.c_void_p(256)   # never dereferenced: the checks fail first
    args = (1, 2, 2, 64, 64)
    assert lib.la_fwd_v(fake, fake, fake, fake, *args, 48, la.LA_F32, 1, 0, 1e-6, None, None, None, 0,
                        None) == la.LA_ERR_UNSUPPORTED
    assert lib.la_fwd_v(fake, fake, fake, fake, *args, 0, la.LA_F32, 1, 0, 1e-6, None, None, None, 0,
                        None) == la.LA_ERR_ARG
    assert lib.la_bwd_v(fake, fake, fake, fake, fake, fake, fake, *args, 256, la.LA_F32, 1, 0, 1e-6, None, None,
                        None, 0, None, 0, None) == la.LA_ERR_UNSUPPORTED
    # a valid Dv with no workspace is a workspace error, still before any CUDA call
    assert lib.la_fwd_v(fake, fake, fake, fake, *args, 32, la.LA_F32, 1, 0, 1e-6, None, None, None, 0,
                        None) == la.LA_ERR_WORKSPACE
