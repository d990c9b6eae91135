"""la_fwd_static_ws: the forward for callers that cannot allocate device memory.

Some callers of this library cannot get scratch memory on the GPU: a plugin host that only
hands over its input and output buffers, or a latency-critical loop that must not call
cudaMalloc/cudaFree because they can synchronise the device.  For them the library offers
la_fwd_static_ws, which keeps its scratch in a static device array instead of a caller
workspace.  These tests call it through the C ABI (ctypes, no Python binding in between)
and check, on two calls in a row that leave the shared scratch dirty for each other, that
its output is bit-for-bit la_fwd's (both take the same plan and run the same kernels, so
any difference would mean the shared scratch leaked from one call into the next).

This file is named to be collected last, so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import gpu_helpers as H
from efficient_transformer_gb300 import build as la_build
from efficient_transformer_gb300 import inputs as gen
from efficient_transformer_gb300 import la

pytestmark = pytest.mark.gpu

LA_ERR_STATIC_WS_LIMIT = 7
STATIC_WS_BYTES = 64 * 1024 * 1024


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    la_build.build()
    lib = la.load()
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.la_fwd_static_ws.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp, vp, vp]
    lib.la_fwd_static_ws.restype = i
    return lib


def call_static(lib, w, dev, out):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    dt = la.LA_F32 if w.dtype == "f32" else la.LA_BF16
    return lib.la_fwd_static_ws(p(dev["q"]), p(dev["k"]), p(dev["v"]), p(out), w.B, w.Hq, w.Hkv,
                                w.N, w.D, dt, int(w.causal), la.PHI[w.phi], w.eps,
                                p(dev["cos_weight"]), p(dev["sin_weight"]),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


# Two different problems back to back: the second starts from the first one's leftovers.
CALLS = [
    gen.Workload("static_ws_gqa_causal", 1, 8, 2, 3000, 128, "bf16", True, "elu+1", scale=0.5),
    gen.Workload("static_ws_bidir_cossin", 2, 4, 4, 700, 64, "bf16", False, "relu", weights=True),
]


def test_matches_la_fwd_on_two_calls_in_a_row(lib):
    for w in CALLS:
        assert la.workspace_size(w.B, w.Hq, w.Hkv, w.N, w.D, w.torch_dtype, w.causal, w.weights,
                                 False) <= STATIC_WS_BYTES
        dev = H.to_dev(gen.make_inputs(w, seed=21))
        want = la.fwd(dev["q"], dev["k"], dev["v"], w.causal, w.phi, w.eps, dev["cos_weight"],
                      dev["sin_weight"])
        got = torch.full_like(want, float("nan"))
        assert call_static(lib, w, dev, got) == la.LA_OK
        la.get_status()
        assert torch.isfinite(got.double()).all()
        assert torch.equal(got, want), f"{w.name}: la_fwd_static_ws differs from la_fwd"


def test_rejects_problems_larger_than_the_static_scratch(lib):
    w = gen.Workload("too_big", 1, 640, 640, 256, 128, "bf16", True, "relu", weights=True)
    assert la.workspace_size(w.B, w.Hq, w.Hkv, w.N, w.D, w.torch_dtype, w.causal, True,
                             False) > STATIC_WS_BYTES
    fake = ctypes.c_void_p(0x10000)   # never touched: the size check comes first
    rc = lib.la_fwd_static_ws(fake, fake, fake, fake, w.B, w.Hq, w.Hkv, w.N, w.D, la.LA_BF16, 1, 1,
                              1e-6, fake, fake, None)
    assert rc == LA_ERR_STATIC_WS_LIMIT
    assert b"static workspace" in lib.la_status_str(rc)
