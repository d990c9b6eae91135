"""Thin Python binding of libla.so (argument marshalling only).

``fwd`` and ``bwd`` follow the signatures of the linear_attn page
(module neuralops.core.triton_kernels.linear_attn): ``fwd(q, k, v, is_causal=False,
phi="elu+1", eps=1e-6, cos_weight=None, sin_weight=None)`` and ``bwd(q, k, v, grad_out,
...) -> (dq, dk, dv)``.  The key/value head count is read from ``k.shape[1]``; when it is
smaller than ``q.shape[1]`` the call is grouped-query attention (module
neuralops.core.triton_kernels.gqa) with the expansion fused into the kernels, and dk, dv
come back with the key/value shape, summed over each group.  Inputs may be strided views
(last dimension contiguous, e.g. slices of a fused qkv projection): their strides go to
``la_fwd_strided`` / ``la_bwd_strided``; outputs are contiguous.

PyTorch supplies device memory and the current stream; every arithmetic step runs in
the library's CUDA kernels.  There is no fallback: if libla.so is missing or a call
fails, an exception says why.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libla.so")

LA_OK, LA_ERR_ARG, LA_ERR_UNSUPPORTED, LA_ERR_ALIGN, LA_ERR_CUDA, LA_ERR_TIMEOUT, LA_ERR_WORKSPACE = range(7)
LA_F32, LA_BF16 = 0, 1
LA_PATH_SIMT, LA_PATH_TCGEN05 = 0, 1
PHI = {"elu+1": 0, "relu": 1, "identity": 2}
_NOT_BUILT = {"softmax_free"}

_lib = None


class LaStrides(ctypes.Structure):
    """la_strides: element strides of a [B, H, N, D] input along B, H, N."""
    _fields_ = [("b", ctypes.c_longlong), ("h", ctypes.c_longlong), ("n", ctypes.c_longlong)]


class LinearAttentionError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(what)


def load(path: str | None = None) -> ctypes.CDLL:
    """Open libla.so (built by ``efficient_transformer_gb300.build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libla.so not found at {p}: build it with "
                           "`python -m efficient_transformer_gb300.build` (no fallback exists)")
    lib = ctypes.CDLL(p)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.la_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
    lib.la_workspace_size.restype = sz
    lib.la_kernel_path.argtypes = [i, i, i, i, i, i, i, i, i]
    lib.la_kernel_path.restype = i
    lib.la_workspace_size_v.argtypes = [i, i, i, i, i, i, i, i, i, i]
    lib.la_workspace_size_v.restype = sz
    lib.la_kernel_path_v.argtypes = [i, i, i, i, i, i, i, i, i, i]
    lib.la_kernel_path_v.restype = i
    lib.la_fwd_v.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, vp, vp, vp, sz, vp]
    lib.la_fwd_v.restype = i
    lib.la_bwd_v.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, vp, vp, vp, sz, vp, sz, vp]
    lib.la_bwd_v.restype = i
    lib.la_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp, vp, vp, sz, vp]
    lib.la_fwd.restype = i
    lib.la_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp, vp, vp, sz, vp]
    lib.la_bwd.restype = i
    lib.la_bwd_from_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp, vp, vp, sz, vp, sz,
                                    vp]
    lib.la_bwd_from_fwd.restype = i
    sp = ctypes.POINTER(LaStrides)
    lib.la_fwd_strided.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp, vp, sp, sp, sp, vp, sz, vp]
    lib.la_fwd_strided.restype = i
    lib.la_bwd_strided.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp, vp, sp, sp, sp, sp,
                                   vp, sz, vp, sz, vp]
    lib.la_bwd_strided.restype = i
    lib.la_get_status.argtypes = [vp]
    lib.la_get_status.restype = i
    lib.la_status_str.argtypes = [i]
    lib.la_status_str.restype = ctypes.c_char_p
    lib.la_last_cuda_error.argtypes = []
    lib.la_last_cuda_error.restype = ctypes.c_char_p
    lib.la_lowrank_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.la_lowrank_fwd.restype = i
    lib.la_lowrank_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.la_lowrank_workspace_size.restype = sz
    lib.la_lowrank_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp, sz, vp]
    lib.la_lowrank_fwd_t.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.la_lowrank_fwd_t.restype = i
    lib.la_lowrank_bwd_t.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp, sz, vp]
    lib.la_lowrank_bwd_t.restype = i
    lib.la_lowrank_bwd.restype = i
    lib.la_trace_start.argtypes = []
    lib.la_trace_start.restype = i
    lib.la_trace_stop.argtypes = []
    lib.la_trace_stop.restype = i
    lib.la_trace_collect.argtypes = []
    lib.la_trace_collect.restype = i
    lib.la_trace_kernel.argtypes = [i, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(i),
                                    ctypes.POINTER(ctypes.c_double)]
    lib.la_trace_kernel.restype = i
    if path is None:
        _lib = lib
    return lib


def _raise(lib, status: int, call: str):
    what = lib.la_status_str(status).decode()
    if status == LA_ERR_CUDA:
        what += ": " + lib.la_last_cuda_error().decode()
    raise LinearAttentionError(status, f"{call}: {what}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LA_F32
    if t.dtype == torch.bfloat16:
        return LA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _phi_code(phi: str) -> int:
    if phi in _NOT_BUILT:
        raise NotImplementedError(f"phi={phi!r} is not built (only 'elu+1', 'relu' and 'identity')")
    if phi not in PHI:
        raise ValueError(f"unknown phi {phi!r}")
    return PHI[phi]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_inputs(q, k, v, cos_weight, sin_weight, extra=()):
    for name, t in (("q", q), ("k", k), ("v", v)) + tuple(extra):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dim() != 4 or (t.shape[3] > 1 and t.stride(3) != 1) or min(t.stride()) < 0:
            raise ValueError(f"{name} must be a [B, H, N, D] tensor whose last dimension is contiguous")
        if t.dtype != q.dtype:
            raise TypeError(f"{name} has dtype {t.dtype}, q has {q.dtype}")
    B, Hq, N, D = q.shape
    if k.shape[0] != B or k.shape[2:] != (N, D) or v.shape[:3] != k.shape[:3]:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    if (cos_weight is None) != (sin_weight is None):
        raise ValueError("give both cos_weight and sin_weight or neither")
    for name, w in (("cos_weight", cos_weight), ("sin_weight", sin_weight)):
        if w is not None and (w.dtype != torch.float32 or not w.is_cuda or w.shape != (N,)
                              or not w.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 CUDA vector of length N={N}")
    return B, Hq, k.shape[1], N, D, v.shape[3]


def _strides(t):
    """la_strides of an input (None when contiguous: the plain entry points take it)."""
    if t.is_contiguous():
        return None
    return ctypes.pointer(LaStrides(t.stride(0), t.stride(1), t.stride(2)))


def _stream_handle(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def workspace_size(B, Hq, Hkv, N, D, dtype: torch.dtype, is_causal: bool, has_weights: bool,
                   is_bwd: bool, Dv: int | None = None) -> int:
    code = LA_F32 if dtype == torch.float32 else LA_BF16
    return int(load().la_workspace_size_v(B, Hq, Hkv, N, D, D if Dv is None else Dv, code, int(is_causal),
                                          int(has_weights), int(is_bwd)))


def kernel_path(B, Hq, Hkv, N, D, dtype: torch.dtype, is_causal: bool, has_weights: bool,
                is_bwd: bool, Dv: int | None = None) -> int:
    code = LA_F32 if dtype == torch.float32 else LA_BF16
    return int(load().la_kernel_path_v(B, Hq, Hkv, N, D, D if Dv is None else Dv, code, int(is_causal),
                                       int(has_weights), int(is_bwd)))


def _workspace(nbytes: int, device, given):
    if nbytes == 0:
        return None
    if given is not None:
        if given.numel() * given.element_size() < nbytes:
            raise ValueError(f"workspace holds {given.numel() * given.element_size()} bytes, "
                             f"{nbytes} needed")
        return given
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, is_causal: bool = False,
        phi: str = "elu+1", eps: float = 1e-6, cos_weight: torch.Tensor | None = None,
        sin_weight: torch.Tensor | None = None, *, out: torch.Tensor | None = None,
        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Linear-attention forward; returns ``out`` [B, Hq, N, Dv] in the dtype of ``q`` (Dv =
    v's last dimension; with Dv != D the inputs must be contiguous)."""
    lib = load()
    B, Hq, Hkv, N, D, Dv = _check_inputs(q, k, v, cos_weight, sin_weight)
    oshape = (B, Hq, N, Dv)
    if out is None:
        out = torch.empty(oshape, dtype=q.dtype, device=q.device)
    elif tuple(out.shape) != oshape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {oshape} tensor of q's dtype")
    dt = _dtype_code(q)
    ws = _workspace(lib.la_workspace_size_v(B, Hq, Hkv, N, D, Dv, dt, int(is_causal),
                                            int(cos_weight is not None), 0), q.device, workspace)
    nws = 0 if ws is None else ws.numel() * ws.element_size()
    strides = [_strides(t) for t in (q, k, v)]
    if Dv != D:
        if any(x is not None for x in strides):
            raise ValueError("with Dv != D, q, k and v must be contiguous")
        st = lib.la_fwd_v(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, N, D, Dv, dt, int(is_causal),
                          _phi_code(phi), float(eps), _ptr(cos_weight), _ptr(sin_weight), _ptr(ws), nws,
                          _stream_handle(stream))
        call = "la_fwd_v"
    elif all(x is None for x in strides):
        st = lib.la_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, N, D, dt, int(is_causal),
                        _phi_code(phi), float(eps), _ptr(cos_weight), _ptr(sin_weight), _ptr(ws), nws,
                        _stream_handle(stream))
        call = "la_fwd"
    else:
        st = lib.la_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, N, D, dt, int(is_causal),
                                _phi_code(phi), float(eps), _ptr(cos_weight), _ptr(sin_weight), *strides,
                                _ptr(ws), nws, _stream_handle(stream))
        call = "la_fwd_strided"
    if st != LA_OK:
        _raise(lib, st, call)
    return out


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, grad_out: torch.Tensor,
        is_causal: bool = False, phi: str = "elu+1", eps: float = 1e-6,
        cos_weight: torch.Tensor | None = None, sin_weight: torch.Tensor | None = None, *,
        dq: torch.Tensor | None = None, dk: torch.Tensor | None = None,
        dv: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None,
        fwd_workspace: torch.Tensor | None = None):
    """Linear-attention backward; returns ``(dq, dk, dv)`` with the shapes of q, k and v.

    ``fwd_workspace``: the workspace of the ``fwd`` call just made on the same inputs (ordered
    before this call); its per-segment states are then reused instead of recomputed
    (``la_bwd_from_fwd``).  The results are the same either way."""
    lib = load()
    B, Hq, Hkv, N, D, Dv = _check_inputs(q, k, v, cos_weight, sin_weight, (("grad_out", grad_out),))
    if tuple(grad_out.shape) != (B, Hq, N, Dv):
        raise ValueError("grad_out must have the shape of out ([B, Hq, N, Dv])")
    dq = torch.empty(q.shape, dtype=q.dtype, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=k.dtype, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=v.dtype, device=v.device) if dv is None else dv
    for name, t, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t.shape != like.shape or t.dtype != like.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor like its input")
    dt = _dtype_code(q)
    ws = _workspace(lib.la_workspace_size_v(B, Hq, Hkv, N, D, Dv, dt, int(is_causal),
                                            int(cos_weight is not None), 1), q.device, workspace)
    nws = 0 if ws is None else ws.numel() * ws.element_size()
    if fwd_workspace is not None and fwd_workspace.device != q.device:
        raise ValueError("fwd_workspace must be on q's device")
    strides = [_strides(t) for t in (q, k, v, grad_out)]
    if Dv != D:
        if any(x is not None for x in strides):
            raise ValueError("with Dv != D, q, k, v and grad_out must be contiguous")
        fws = 0 if fwd_workspace is None else fwd_workspace.numel() * fwd_workspace.element_size()
        st = lib.la_bwd_v(_ptr(q), _ptr(k), _ptr(v), _ptr(grad_out), _ptr(dq), _ptr(dk), _ptr(dv),
                          B, Hq, Hkv, N, D, Dv, dt, int(is_causal), _phi_code(phi), float(eps),
                          _ptr(cos_weight), _ptr(sin_weight), _ptr(fwd_workspace), fws,
                          _ptr(ws), nws, _stream_handle(stream))
        call = "la_bwd_v"
    elif any(x is not None for x in strides):
        fws = 0 if fwd_workspace is None else fwd_workspace.numel() * fwd_workspace.element_size()
        st = lib.la_bwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(grad_out), _ptr(dq), _ptr(dk), _ptr(dv),
                                B, Hq, Hkv, N, D, dt, int(is_causal), _phi_code(phi), float(eps),
                                _ptr(cos_weight), _ptr(sin_weight), *strides, _ptr(fwd_workspace), fws,
                                _ptr(ws), nws, _stream_handle(stream))
        call = "la_bwd_strided"
    elif fwd_workspace is None:
        st = lib.la_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(grad_out), _ptr(dq), _ptr(dk), _ptr(dv),
                        B, Hq, Hkv, N, D, dt, int(is_causal), _phi_code(phi), float(eps),
                        _ptr(cos_weight), _ptr(sin_weight), _ptr(ws), nws, _stream_handle(stream))
        call = "la_bwd"
    else:
        st = lib.la_bwd_from_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(grad_out), _ptr(dq), _ptr(dk), _ptr(dv),
                                 B, Hq, Hkv, N, D, dt, int(is_causal), _phi_code(phi), float(eps),
                                 _ptr(cos_weight), _ptr(sin_weight), _ptr(fwd_workspace),
                                 fwd_workspace.numel() * fwd_workspace.element_size(), _ptr(ws), nws,
                                 _stream_handle(stream))
        call = "la_bwd_from_fwd"
    if st != LA_OK:
        _raise(lib, st, call)
    return dq, dk, dv


def _check_lowrank(x, U, V, bias):
    for name, t in (("x", x), ("U", U), ("V", V)) + ((("bias", bias),) if bias is not None else ()):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if t.dtype != x.dtype:
            raise TypeError(f"{name} has dtype {t.dtype}, x has {x.dtype}")
    if U.dim() != 2 or V.dim() != 2 or x.shape[-1] != V.shape[1] or U.shape[1] != V.shape[0]:
        raise ValueError(f"shapes disagree: x {tuple(x.shape)}, U {tuple(U.shape)}, V {tuple(V.shape)}")
    if bias is not None and bias.shape != (U.shape[0],):
        raise ValueError("bias must have K_out = U.shape[0] elements")
    M = x.numel() // x.shape[-1]
    return M, V.shape[1], V.shape[0], U.shape[0]


def lowrank_fwd(x: torch.Tensor, U: torch.Tensor, V: torch.Tensor, bias: torch.Tensor | None = None, *,
                out: torch.Tensor | None = None, t_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Low-rank projection ``y = (x @ V.T) @ U.T + bias`` (module
    neuralops.core.triton_kernels.low_rank, ``fwd``): x [..., K_in], U [K_out, r], V [r, K_in];
    returns y [..., K_out].  ``t_out`` ([M, r], x's dtype): also receives the bottleneck
    t = x V^T for ``lowrank_bwd(..., t=t_out)`` (``la_lowrank_fwd_t``)."""
    lib = load()
    M, K_in, r, K_out = _check_lowrank(x, U, V, bias)
    if out is None:
        out = torch.empty(x.shape[:-1] + (K_out,), dtype=x.dtype, device=x.device)
    elif out.shape != x.shape[:-1] + (K_out,) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor [..., K_out] of x's dtype")
    if t_out is None:
        st = lib.la_lowrank_fwd(_ptr(x), _ptr(U), _ptr(V), _ptr(bias), _ptr(out), M, K_in, r, K_out,
                                _dtype_code(x), _stream_handle(stream))
        call = "la_lowrank_fwd"
    else:
        if t_out.shape != (M, r) or t_out.dtype != x.dtype or not t_out.is_contiguous() or not t_out.is_cuda:
            raise ValueError(f"t_out must be a contiguous CUDA tensor [{M}, {r}] of x's dtype")
        st = lib.la_lowrank_fwd_t(_ptr(x), _ptr(U), _ptr(V), _ptr(bias), _ptr(out), _ptr(t_out), M, K_in, r,
                                  K_out, _dtype_code(x), _stream_handle(stream))
        call = "la_lowrank_fwd_t"
    if st != LA_OK:
        _raise(lib, st, call)
    return out


def lowrank_bwd(x: torch.Tensor, U: torch.Tensor, V: torch.Tensor, grad_out: torch.Tensor,
                bias: torch.Tensor | None = None, *, workspace: torch.Tensor | None = None,
                t: torch.Tensor | None = None, stream=None):
    """Backward of ``lowrank_fwd`` (module neuralops.core.triton_kernels.low_rank, ``bwd``):
    returns ``(dx, dU, dV, dbias)``, dbias None without a bias.  ``t``: the bottleneck that
    ``lowrank_fwd(..., t_out=t)`` left for these x, V (``la_lowrank_bwd_t``: same results,
    one pass over x fewer)."""
    lib = load()
    M, K_in, r, K_out = _check_lowrank(x, U, V, bias)
    if grad_out.shape != x.shape[:-1] + (K_out,) or grad_out.dtype != x.dtype or not grad_out.is_contiguous():
        raise ValueError("grad_out must be a contiguous tensor [..., K_out] of x's dtype")
    dt = _dtype_code(x)
    dx, dU, dV = torch.empty_like(x), torch.empty_like(U), torch.empty_like(V)
    db = torch.empty_like(bias) if bias is not None else None
    ws = _workspace(lib.la_lowrank_workspace_size(M, K_in, r, K_out, dt, 1), x.device, workspace)
    nws = 0 if ws is None else ws.numel() * ws.element_size()
    if t is None:
        st = lib.la_lowrank_bwd(_ptr(x), _ptr(U), _ptr(V), _ptr(grad_out), _ptr(dx), _ptr(dU), _ptr(dV), _ptr(db),
                                M, K_in, r, K_out, dt, _ptr(ws), nws, _stream_handle(stream))
        call = "la_lowrank_bwd"
    else:
        if t.shape != (M, r) or t.dtype != x.dtype or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"t must be a contiguous CUDA tensor [{M}, {r}] of x's dtype")
        st = lib.la_lowrank_bwd_t(_ptr(x), _ptr(U), _ptr(V), _ptr(t), _ptr(grad_out), _ptr(dx), _ptr(dU), _ptr(dV),
                                  _ptr(db), M, K_in, r, K_out, dt, _ptr(ws), nws, _stream_handle(stream))
        call = "la_lowrank_bwd_t"
    if st != LA_OK:
        _raise(lib, st, call)
    return dx, dU, dV, db


def get_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel latched an error since the last check."""
    lib = load()
    st = lib.la_get_status(_stream_handle(stream))
    if st != LA_OK:
        _raise(lib, st, "la_get_status")


def trace_start() -> None:
    """Start bracketing every library kernel launch with CUDA events (for reports)."""
    load().la_trace_start()


def trace_stop() -> dict:
    """Stop tracing; return {kernel name: (launches, total device ms)} since trace_start()."""
    lib = load()
    lib.la_trace_stop()
    n = lib.la_trace_collect()
    res = {}
    for idx in range(n):
        name, launches, ms = ctypes.c_char_p(), ctypes.c_int(), ctypes.c_double()
        if lib.la_trace_kernel(idx, ctypes.byref(name), ctypes.byref(launches), ctypes.byref(ms)) == LA_OK:
            res[name.value.decode()] = (launches.value, ms.value)
    return res
