"""Every workspace byte a kernel reads was written by the library first: with workspaces
filled with 0xFF (NaN as float32, a NaN pattern as bf16) instead of zeros, every call gives
bit for bit the results it gives with zero-filled workspaces.  A read of memory no kernel
wrote would carry the fill into the outputs (freshly allocated memory often holds zeros, so
such a read can otherwise pass unnoticed)."""
import pytest
import torch

import gpu_helpers as H
from efficient_transformer_gb300 import inputs as gen
from efficient_transformer_gb300 import la

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, N, D, dtype, causal, phi, weights
    (1, 8, 2, 1500, 128, "bf16", True, "elu+1", False),    # tensor cores, GQA
    (1, 4, 4, 1500, 128, "bf16", True, "relu", True),      # cos/sin passes, masked rows
    (1, 8, 8, 900, 64, "bf16", False, "elu+1", True),      # cos/sin passes, bidirectional
    (1, 6, 3, 700, 128, "bf16", True, "elu+1", False),     # masked rows (n_rep 2)
    (1, 4, 2, 300, 64, "f32", True, "elu+1", True),        # CUDA cores
]


def run(w, dev, fill):
    cw, sw = dev["cos_weight"], dev["sin_weight"]
    nf = la.workspace_size(w.B, w.Hq, w.Hkv, w.N, w.D, dev["q"].dtype, w.causal, w.weights, False)
    nb = la.workspace_size(w.B, w.Hq, w.Hkv, w.N, w.D, dev["q"].dtype, w.causal, w.weights, True)
    wf = torch.full((max(1, nf),), fill, dtype=torch.uint8, device="cuda")
    wb = torch.full((max(1, nb),), fill, dtype=torch.uint8, device="cuda")
    out = la.fwd(dev["q"], dev["k"], dev["v"], w.causal, w.phi, w.eps, cw, sw, workspace=wf)
    ctx = la.bwd(dev["q"], dev["k"], dev["v"], dev["grad_out"], w.causal, w.phi, w.eps, cw, sw, workspace=wb,
                 fwd_workspace=wf)
    wb.fill_(fill)
    own = la.bwd(dev["q"], dev["k"], dev["v"], dev["grad_out"], w.causal, w.phi, w.eps, cw, sw, workspace=wb)
    la.get_status()
    return (out,) + ctx + own


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_results_do_not_depend_on_workspace_contents(case):
    B, Hq, Hkv, N, D, dt, causal, phi, weights = case
    w = gen.Workload("poison", B, Hq, Hkv, N, D, dt, causal, phi, scale=0.5, weights=weights)
    dev = H.to_dev(gen.make_inputs(w, seed=3))
    clean = run(w, dev, 0)
    poisoned = run(w, dev, 0xFF)
    for n, a, b in zip(("out", "dq", "dk", "dv", "dq(bwd)", "dk(bwd)", "dv(bwd)"), poisoned, clean):
        assert torch.isfinite(a.float()).all(), f"{n}: non-finite values with a 0xFF-filled workspace"
        assert torch.equal(a, b), f"{n}: differs between 0xFF- and zero-filled workspaces"


def test_lowrank_results_do_not_depend_on_workspace_contents():
    wl = gen.LowRankWorkload("poison_lr", 700, 512, 128, 384)
    d = H.to_dev(gen.make_lowrank_inputs(wl, seed=3))
    nb = la.load().la_lowrank_workspace_size(wl.M, wl.K_in, wl.r, wl.K_out, la.LA_BF16, 1)
    res = []
    for fill in (0, 0xFF):
        ws = torch.full((nb,), fill, dtype=torch.uint8, device="cuda")
        res.append(la.lowrank_bwd(d["x"], d["U"], d["V"], d["grad_out"], d["bias"], workspace=ws))
    la.get_status()
    for n, a, b in zip(("dx", "dU", "dV", "dbias"), *res):
        assert torch.equal(a, b), f"{n}: differs between 0xFF- and zero-filled workspaces"
