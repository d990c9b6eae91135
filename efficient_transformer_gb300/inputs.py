"""Seeded synthetic inputs for linear attention (shared by the tests, the smoke check and
the benchmark).

This module holds no arithmetic of the method: it only draws random tensors and the
cosFormer position weights, which are inputs of the operation.  The recipe:

* one CPU ``torch.Generator`` seeded with ``seed`` (0 by default);
* float32 standard normal draws in the order q, k, v, grad_out, each of its own shape
  ([B, Hq, N, D] for q, [B, Hkv, N, D] for k, [B, Hkv, N, Dv] for v and [B, Hq, N, Dv] for
  grad_out, the value width Dv being D unless the workload sets it);
* q, k and v multiplied by ``scale`` (grad_out is not scaled);
* for workloads marked ``positive`` (the identity feature map, whose features the pages
  call non-negative), q and k replaced by their absolute values;
* a cast to the workload's dtype (round to nearest even for bf16);
* cosFormer weights cos(pi*i/(2N)) and sin(pi*i/(2N)) for i = 0..N-1, evaluated in
  float64 and stored as float32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    D: int
    dtype: str          # "f32" or "bf16"
    causal: bool
    phi: str            # "elu+1" or "relu"
    eps: float = 1e-6
    weights: bool = False   # cosFormer cos/sin position weights
    scale: float = 1.0
    positive: bool = False  # |q|, |k| (non-negative features for phi = identity)
    Dv: int | None = None   # value width (v, out, grad_out, dv); None: D

    @property
    def value_dim(self) -> int:
        return self.D if self.Dv is None else self.Dv

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def tokens(self) -> int:
        return self.B * self.N

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The workloads the operation is measured and checked on.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("causal_b1_h2_n256_d32_f32", 1, 2, 2, 256, 32, "f32", True, "elu+1"),
        Workload("bidir_b2_h8_n2048_d64_bf16_elu1", 2, 8, 8, 2048, 64, "bf16", False, "elu+1"),
        Workload("bidir_b2_h8_n2048_d64_bf16_relu", 2, 8, 8, 2048, 64, "bf16", False, "relu"),
        Workload("causal_b4_h16_n4096_d64_bf16", 4, 16, 16, 4096, 64, "bf16", True, "elu+1"),
        Workload("cosformer_causal_b2_h16_n8192_d128_bf16", 2, 16, 16, 8192, 128, "bf16", True,
                 "relu", weights=True),
        Workload("gqa_causal_b1_hq32_hkv8_n65536_d128_bf16", 1, 32, 8, 65536, 128, "bf16", True,
                 "elu+1", scale=0.5),
    ]
}

# The workload the benchmark times (the long-context grouped-query case).
BENCH_WORKLOAD = "gqa_causal_b1_hq32_hkv8_n65536_d128_bf16"


def position_weights(N: int):
    """cosFormer weights (cos(pi*i/(2N)), sin(pi*i/(2N))) as float32 CPU tensors."""
    i = torch.arange(N, dtype=torch.float64)
    ang = i * (math.pi / (2.0 * N))
    return torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)


def make_inputs(w: Workload, seed: int = 0, device: str | torch.device = "cpu"):
    """Return dict(q, k, v, grad_out, cos_weight, sin_weight) for workload ``w``.

    Draws happen on the CPU so that every consumer sees the same values; the tensors
    are then moved to ``device``.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    qs = (w.B, w.Hq, w.N, w.D)
    ks = (w.B, w.Hkv, w.N, w.D)
    q = torch.randn(qs, generator=gen, dtype=torch.float32)
    k = torch.randn(ks, generator=gen, dtype=torch.float32)
    v = torch.randn(ks[:3] + (w.value_dim,), generator=gen, dtype=torch.float32)
    g = torch.randn(qs[:3] + (w.value_dim,), generator=gen, dtype=torch.float32)
    if w.scale != 1.0:
        q.mul_(w.scale)
        k.mul_(w.scale)
        v.mul_(w.scale)
    if w.positive:
        q.abs_()
        k.abs_()
    dt = w.torch_dtype
    out = {"q": q.to(dt), "k": k.to(dt), "v": v.to(dt), "grad_out": g.to(dt),
           "cos_weight": None, "sin_weight": None}
    if w.weights:
        out["cos_weight"], out["sin_weight"] = position_weights(w.N)
    if str(device) != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out


@dataclass(frozen=True)
class LowRankWorkload:
    """y = (x V^T) U^T + bias over M rows."""
    name: str
    M: int
    K_in: int
    r: int
    K_out: int
    dtype: str = "bf16"
    bias: bool = True

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


# The low-rank projection measured beside the attention: 64 K rows (a batch of long
# sequences) projected through a rank-256 bottleneck between 4096-wide activations.
LOWRANK_WORKLOADS = {
    w.name: w
    for w in [
        LowRankWorkload("lowrank_m65536_kin4096_r256_kout4096_bf16", 65536, 4096, 256, 4096),
    ]
}


def make_lowrank_inputs(w: LowRankWorkload, seed: int = 0):
    """x ~ N(0, 1); V ~ N(0, 1/K_in) and U ~ N(0, 1/r), so that t and y stay of order one;
    bias and grad_out ~ N(0, 1); drawn in the order x, V, U, bias, grad_out on a CPU
    generator seeded with `seed`, then cast to the workload's dtype."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    x = torch.randn((w.M, w.K_in), generator=gen)
    V = torch.randn((w.r, w.K_in), generator=gen) / math.sqrt(w.K_in)
    U = torch.randn((w.K_out, w.r), generator=gen) / math.sqrt(w.r)
    b = torch.randn((w.K_out,), generator=gen)
    g = torch.randn((w.M, w.K_out), generator=gen)
    dt = w.torch_dtype
    return {"x": x.to(dt), "U": U.to(dt), "V": V.to(dt), "bias": b.to(dt) if w.bias else None,
            "grad_out": g.to(dt)}


def kv_group_slice(inputs: dict, w: Workload, b: int, g: int):
    """Inputs restricted to batch ``b`` and key/value head ``g`` with its n_rep query
    heads.  Groups are independent, so the oracle on this slice gives exactly the
    matching rows of the full result."""
    n_rep = w.Hq // w.Hkv
    hs = slice(g * n_rep, (g + 1) * n_rep)
    return {
        "q": inputs["q"][b:b + 1, hs],
        "k": inputs["k"][b:b + 1, g:g + 1],
        "v": inputs["v"][b:b + 1, g:g + 1],
        "grad_out": inputs["grad_out"][b:b + 1, hs],
        "cos_weight": inputs["cos_weight"],
        "sin_weight": inputs["sin_weight"],
    }
