"""Strided inputs (la_fwd_strided / la_bwd_strided): q, k, v, grad_out as views into fused
buffers, as a fused qkv projection leaves them ([B, N, H, D] storage seen as [B, H, N, D]).
The results must equal those of the same values passed contiguous, bit for bit (the kernels
read the same numbers), and match the oracle."""
import pytest
import torch

from efficient_transformer_gb300 import inputs as gen
from efficient_transformer_gb300 import la

import gpu_helpers as H

pytestmark = pytest.mark.gpu


def fused_views(tensors, pad_heads=0):
    """Views [B, H_i, N, D] into one [B, N, sum H_i + pad_heads, D] buffer, holding the
    values of `tensors`."""
    B, _, N, D = tensors[0].shape
    total = sum(t.shape[1] for t in tensors) + pad_heads
    buf = torch.full((B, N, total, D), float("nan"), dtype=tensors[0].dtype, device="cuda")
    views, h0 = [], 0
    for t in tensors:
        view = buf[:, :, h0:h0 + t.shape[1]].permute(0, 2, 1, 3)
        view.copy_(t)
        views.append(view)
        h0 += t.shape[1]
    return views


CASES = [
    # B, Hq, Hkv, N, D, dtype, causal, phi, weights
    (1, 8, 2, 700, 128, "bf16", True, "elu+1", False),    # tensor cores, GQA
    (2, 4, 4, 513, 64, "bf16", False, "relu", False),     # tensor cores, bidirectional
    (1, 4, 4, 600, 128, "bf16", True, "relu", True),      # tensor cores, cos/sin passes, masked rows
    (1, 4, 2, 300, 64, "f32", True, "elu+1", False),      # CUDA cores
    (1, 6, 3, 200, 32, "bf16", True, "elu+1", True),      # CUDA cores (D = 32)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_strided_inputs(case):
    B, Hq, Hkv, N, D, dt, causal, phi, weights = case
    w = gen.Workload("strided", B, Hq, Hkv, N, D, dt, causal, phi, scale=0.5, weights=weights)
    inp = gen.make_inputs(w, seed=23)
    dev = H.to_dev(inp)
    cw, sw = dev["cos_weight"], dev["sin_weight"]
    # q, k, v from one fused buffer (one spare head of padding), grad_out from another
    qs, ks, vs = fused_views([dev["q"], dev["k"], dev["v"]], pad_heads=1)
    (gs,) = fused_views([dev["grad_out"]], pad_heads=2)
    assert not qs.is_contiguous() and not gs.is_contiguous()
    # the same values, contiguous
    ref_gpu = H.run_gpu(w, dev, from_fwd=True)
    ws = torch.empty(max(1, la.workspace_size(B, Hq, Hkv, N, D, qs.dtype, causal, weights, False)),
                     dtype=torch.uint8, device="cuda")
    out = la.fwd(qs, ks, vs, causal, phi, w.eps, cw, sw, workspace=ws)
    got_ctx = la.bwd(qs, ks, vs, gs, causal, phi, w.eps, cw, sw, fwd_workspace=ws)
    got = la.bwd(qs, ks, vs, gs, causal, phi, w.eps, cw, sw)
    la.get_status()
    for name, a, b in zip(("out", "dq", "dk", "dv"), (out,) + got_ctx, ref_gpu):
        assert torch.equal(a, b), f"{name}: strided inputs differ from contiguous ones"
    for name, a, b in zip(("dq", "dk", "dv"), got, ref_gpu[1:]):
        assert torch.equal(a, b), f"{name} (la_bwd_strided without the forward's workspace) differs"
    H.compare(w, (out,) + got_ctx, H.run_oracle(w, inp), label="strided inputs")


def test_strides_off_the_tma_grid_are_rejected_on_the_tensor_core_path():
    """bf16 on the tensor-core path needs strides in multiples of 8 elements."""
    w = gen.Workload("strided_bad", 1, 2, 2, 64, 64, "bf16", True, "elu+1")
    dev = H.to_dev(gen.make_inputs(w, seed=1))
    buf = torch.zeros(2 * 4100, dtype=torch.bfloat16, device="cuda")
    # heads 4100 elements apart (not a multiple of 8)
    q = torch.as_strided(buf, (1, 2, 64, 64), (2 * 4100, 4100, 64, 1))
    with pytest.raises(la.LinearAttentionError) as err:
        la.fwd(q, dev["k"], dev["v"], True)
    assert err.value.status == la.LA_ERR_ALIGN
