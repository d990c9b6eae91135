"""The bounded-wait path on the GPU: a wait that runs out is reported, and the library
stays usable.

Every wait of the tensor-core kernels gives up after a time limit, raises a flag that the
other warps of the block see, drains its copies in flight, frees its TMEM and returns; the
block latches LA_ERR_TIMEOUT for la_get_status().  The test build of the library
(``build(variant="test")``: 5 ms limit) has one switch that makes warp 4 of block 0 of the
forward kernel withhold its arrival for the first chunk, so the MMA warp's wait for that
chunk runs out.  No kernel traps or faults: the wait simply ends with an error status.
"""
import ctypes

import pytest
import torch

import gpu_helpers as H
from efficient_transformer_gb300 import build as la_build
from efficient_transformer_gb300 import inputs as gen
from efficient_transformer_gb300 import la

pytestmark = pytest.mark.gpu

# causal tensor-core forward, n_rep 2 (C = 64), 64 key/value heads: two segments of three
# chunks per head, fewer chunks than pipeline stages
W = gen.Workload("timeout_case", 1, 128, 64, 384, 64, "bf16", True, "elu+1", scale=0.5)


@pytest.fixture(scope="module")
def tlib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    lib = la.load(la_build.build(variant="test"))
    lib.la_test_withhold_arrival.argtypes = [ctypes.c_int]
    lib.la_test_withhold_arrival.restype = ctypes.c_int
    return lib


def fwd(lib, dev, out, ws):
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.la_fwd(p(dev["q"]), p(dev["k"]), p(dev["v"]), p(out), W.B, W.Hq, W.Hkv, W.N, W.D, la.LA_BF16,
                      int(W.causal), la.PHI[W.phi], W.eps, None, None, p(ws), ws.numel(),
                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def status(lib):
    return lib.la_get_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_wait_that_runs_out_is_reported_and_the_next_call_is_clean(tlib):
    assert la.kernel_path(W.B, W.Hq, W.Hkv, W.N, W.D, torch.bfloat16, True, False, False) == la.LA_PATH_TCGEN05
    inp = gen.make_inputs(W, seed=17)
    dev = H.to_dev(inp)
    ws = torch.empty(tlib.la_workspace_size(W.B, W.Hq, W.Hkv, W.N, W.D, la.LA_BF16, 1, 0, 0),
                     dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(dev["q"])
    assert status(tlib) == la.LA_OK
    assert tlib.la_test_withhold_arrival(1) == 0
    try:
        assert fwd(tlib, dev, out, ws) == la.LA_OK          # enqueued; the kernel runs out later
        assert status(tlib) == la.LA_ERR_TIMEOUT            # reported once ...
    finally:
        assert tlib.la_test_withhold_arrival(0) == 0
    assert status(tlib) == la.LA_OK                         # ... and cleared
    out.fill_(float("nan"))
    assert fwd(tlib, dev, out, ws) == la.LA_OK
    assert status(tlib) == la.LA_OK
    ref = H.run_oracle(W, inp)[0]
    H.compare(W, (out,), (ref,), label="after a timeout", names=("out",))
