"""The seeded input recipe (CPU): the value width only changes the shapes of v and grad_out,
and an unset value width draws exactly what Dv = D draws, so the stored workloads keep their
inputs."""
import torch

from efficient_transformer_gb300 import inputs as gen


def test_value_width_unset_equals_d():
    w = gen.Workload("w", 2, 4, 2, 37, 64, "bf16", True, "elu+1", weights=True, scale=0.5)
    a = gen.make_inputs(w, seed=3)
    b = gen.make_inputs(w.with_(Dv=64), seed=3)
    for name in ("q", "k", "v", "grad_out", "cos_weight", "sin_weight"):
        assert torch.equal(a[name], b[name]), name


def test_value_width_shapes():
    w = gen.Workload("w", 2, 6, 3, 19, 32, "f32", False, "relu", Dv=128)
    t = gen.make_inputs(w, seed=1)
    assert tuple(t["q"].shape) == (2, 6, 19, 32) and tuple(t["k"].shape) == (2, 3, 19, 32)
    assert tuple(t["v"].shape) == (2, 3, 19, 128) and tuple(t["grad_out"].shape) == (2, 6, 19, 128)
    assert w.value_dim == 128 and gen.Workload("x", 1, 1, 1, 1, 64, "f32", True, "relu").value_dim == 64


def test_draw_order_q_k_v_grad_out():
    """q, k, v and grad_out are consecutive standard-normal draws of one seeded generator."""
    w = gen.Workload("w", 1, 2, 1, 5, 32, "f32", True, "elu+1", Dv=64)
    t = gen.make_inputs(w, seed=9)
    g = torch.Generator(device="cpu")
    g.manual_seed(9)
    want = [torch.randn(s, generator=g, dtype=torch.float32)
            for s in ((1, 2, 5, 32), (1, 1, 5, 32), (1, 1, 5, 64), (1, 2, 5, 64))]
    for name, x in zip(("q", "k", "v", "grad_out"), want):
        assert torch.equal(t[name], x), name
