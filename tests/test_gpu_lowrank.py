"""GPU parity of the low-rank projection y = (x V^T) U^T + bias (tensor cores, through the C
ABI) against the float64 oracle, max|gpu - oracle| / max|oracle| <= 2e-2 for bf16."""
import pytest
import torch

import gpu_helpers as H
from efficient_transformer_gb300 import build as la_build
from efficient_transformer_gb300 import inputs as gen
from efficient_transformer_gb300 import la
from oracle import low_rank as lr_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    la_build.build()
    la.load()


CASES = [
    # M, K_in, r, K_out, bias     (ragged M, K_in, r and K_out; every padded rank 64..256)
    (1000, 512, 64, 384, True),
    (777, 200, 48, 136, True),
    (300, 1024, 128, 1024, False),
    (2048, 256, 200, 520, True),
    (513, 768, 256, 640, True),
    (128, 64, 8, 64, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_lowrank_forward(case):
    M, K_in, r, K_out, bias = case
    w = gen.LowRankWorkload(f"lr_m{M}_kin{K_in}_r{r}_kout{K_out}", M, K_in, r, K_out, bias=bias)
    inp = gen.make_lowrank_inputs(w, seed=31)
    dev = H.to_dev(inp)
    y = la.lowrank_fwd(dev["x"], dev["U"], dev["V"], dev["bias"])
    la.get_status()
    ref = lr_oracle.fwd(inp["x"], inp["U"], inp["V"], inp["bias"])
    err = H.rel_err(y, ref)
    H.record_named(w.name, "lowrank fwd", {"y": err})
    assert err <= H.TOL["bf16"], err


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_lowrank_backward(case):
    M, K_in, r, K_out, bias = case
    w = gen.LowRankWorkload(f"lr_m{M}_kin{K_in}_r{r}_kout{K_out}", M, K_in, r, K_out, bias=bias)
    inp = gen.make_lowrank_inputs(w, seed=37)
    dev = H.to_dev(inp)
    got = la.lowrank_bwd(dev["x"], dev["U"], dev["V"], dev["grad_out"], dev["bias"])
    again = la.lowrank_bwd(dev["x"], dev["U"], dev["V"], dev["grad_out"], dev["bias"])
    la.get_status()
    ref = lr_oracle.bwd(inp["x"], inp["U"], inp["V"], inp["grad_out"], inp["bias"])
    errs = {}
    for name, a, b, c in zip(("dx", "dU", "dV", "dbias"), got, ref, again):
        if b is None:
            assert a is None
            continue
        errs[name] = H.rel_err(a, b)
        assert torch.equal(a, c), f"{name} differs between two runs"
    H.record_named(w.name, "lowrank bwd", errs)
    assert all(e <= H.TOL["bf16"] for e in errs.values()), errs


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_lowrank_saved_t(case):
    """la_lowrank_fwd_t writes the same y as la_lowrank_fwd plus t = bf16(x V^T), and
    la_lowrank_bwd_t given that t returns exactly la_lowrank_bwd's gradients."""
    M, K_in, r, K_out, bias = case
    w = gen.LowRankWorkload(f"lr_m{M}_kin{K_in}_r{r}_kout{K_out}", M, K_in, r, K_out, bias=bias)
    dev = H.to_dev(gen.make_lowrank_inputs(w, seed=41))
    y = la.lowrank_fwd(dev["x"], dev["U"], dev["V"], dev["bias"])
    t = torch.empty((M, r), dtype=torch.bfloat16, device="cuda")
    y_t = la.lowrank_fwd(dev["x"], dev["U"], dev["V"], dev["bias"], t_out=t)
    got = la.lowrank_bwd(dev["x"], dev["U"], dev["V"], dev["grad_out"], dev["bias"], t=t)
    ref = la.lowrank_bwd(dev["x"], dev["U"], dev["V"], dev["grad_out"], dev["bias"])
    la.get_status()
    assert torch.equal(y, y_t)
    # t is the bottleneck rounded once: within bf16 rounding of the exact x V^T
    exact = dev["x"].double() @ dev["V"].double().T
    assert float((t.double() - exact).abs().max() / exact.abs().max()) <= 2 ** -8
    for name, a, b in zip(("dx", "dU", "dV", "dbias"), got, ref):
        assert (a is None) == (b is None)
        if a is not None:
            assert torch.equal(a, b), f"{name} with the forward's t differs"


def test_lowrank_leading_dims_and_deterministic():
    w = gen.LowRankWorkload("lr_lead", 2 * 300, 256, 64, 256)
    inp = gen.make_lowrank_inputs(w, seed=5)
    dev = H.to_dev(inp)
    x3 = dev["x"].view(2, 300, 256)
    a = la.lowrank_fwd(x3, dev["U"], dev["V"], dev["bias"])
    b = la.lowrank_fwd(x3, dev["U"], dev["V"], dev["bias"])
    la.get_status()
    assert a.shape == (2, 300, 256) and torch.equal(a, b)
    ref = lr_oracle.fwd(inp["x"].view(2, 300, 256), inp["U"], inp["V"], inp["bias"])
    assert H.rel_err(a, ref) <= H.TOL["bf16"]


def test_lowrank_rejects():
    x = torch.zeros(4, 64, device="cuda", dtype=torch.bfloat16)
    U = torch.zeros(64, 300, device="cuda", dtype=torch.bfloat16)
    V = torch.zeros(300, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(la.LinearAttentionError):
        la.lowrank_fwd(x, U, V)            # r > 256
    with pytest.raises(ValueError):
        la.lowrank_fwd(x, U[:, :8], V)     # shapes disagree
