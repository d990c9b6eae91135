"""A value width Dv different from the head dimension D (la_fwd_v, la_bwd_v) against the
oracle: out and dv are [.., N, Dv], dq and dk stay [.., N, D].  These shapes run on the
CUDA-core kernels (the tensor-core tiles are laid out for Dv = D)."""
import pytest
import torch

import gpu_helpers as H
from efficient_transformer_gb300 import inputs as gen
from efficient_transformer_gb300 import la

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, N, D, Dv, dtype, causal, phi, weights
    (1, 2, 1, 300, 64, 32, "f32", True, "elu+1", False),
    (2, 4, 2, 77, 32, 128, "f32", False, "relu", True),
    (1, 2, 2, 1000, 128, 64, "bf16", True, "relu", True),
    (1, 8, 2, 161, 64, 128, "bf16", True, "elu+1", False),
    (2, 3, 3, 40, 128, 32, "bf16", False, "elu+1", False),
    (1, 4, 4, 17, 32, 64, "f32", True, "relu", False),
    (1, 1, 1, 1, 64, 128, "f32", True, "elu+1", False),
]


def workload(case):
    B, Hq, Hkv, N, D, Dv, dt, causal, phi, weights = case
    return gen.Workload(f"dv_b{B}_hq{Hq}_hkv{Hkv}_n{N}_d{D}_dv{Dv}_{dt}", B, Hq, Hkv, N, D, dt, causal, phi,
                        eps=100.0 if N == 1 else 1e-6, weights=weights, Dv=Dv)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_value_width(case):
    w = workload(case)
    assert la.kernel_path(w.B, w.Hq, w.Hkv, w.N, w.D, w.torch_dtype, w.causal, w.weights, False,
                          Dv=w.Dv) == la.LA_PATH_SIMT
    inp = gen.make_inputs(w, seed=31)
    ref = H.run_oracle(w, inp)
    dev = H.to_dev(inp)
    got = H.run_gpu(w, dev, from_fwd=False)
    assert tuple(got[0].shape) == (w.B, w.Hq, w.N, w.Dv) and tuple(got[3].shape) == (w.B, w.Hkv, w.N, w.Dv)
    H.compare(w, got, ref, label="bwd")
    # the backward that takes the forward's segment states gives the same bits
    got2 = H.run_gpu(w, dev, from_fwd=True)
    for a, b in zip(got, got2):
        assert torch.equal(a, b)


def test_value_width_equal_to_d_is_la_fwd():
    """la_fwd_v with Dv = D is la_fwd (same plan, same kernels): identical bits."""
    w = gen.Workload("dv_equal", 1, 8, 2, 700, 128, "bf16", True, "elu+1", Dv=128)
    dev = H.to_dev(gen.make_inputs(w, seed=5))
    lib = la.load()
    dt = la.LA_BF16
    n = lib.la_workspace_size(w.B, w.Hq, w.Hkv, w.N, w.D, dt, 1, 0, 0)
    assert n == lib.la_workspace_size_v(w.B, w.Hq, w.Hkv, w.N, w.D, w.D, dt, 1, 0, 0)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    o1, o2 = torch.empty_like(dev["q"]), torch.empty_like(dev["q"])
    s = la._stream_handle(None)
    P = la._ptr
    assert lib.la_fwd(P(dev["q"]), P(dev["k"]), P(dev["v"]), P(o1), w.B, w.Hq, w.Hkv, w.N, w.D, dt, 1, 0, 1e-6,
                      None, None, P(ws), n, s) == 0
    assert lib.la_fwd_v(P(dev["q"]), P(dev["k"]), P(dev["v"]), P(o2), w.B, w.Hq, w.Hkv, w.N, w.D, w.D, dt, 1, 0,
                        1e-6, None, None, P(ws), n, s) == 0
    la.get_status()
    assert torch.equal(o1, o2)
