"""Shared helpers of the GPU parity tests: run the CUDA path through the binding, run the
oracle on the same inputs, and compare per output tensor."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from efficient_transformer_gb300 import inputs as gen
from efficient_transformer_gb300 import la

# max|gpu - oracle| / max|oracle| per output tensor
TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_dev(inp: dict) -> dict:
    return {n: (t.cuda() if t is not None else None) for n, t in inp.items()}


def run_gpu(w: gen.Workload, dev: dict, from_fwd: bool = False):
    """la_fwd, then la_bwd (from_fwd=False: the backward recomputes the forward's states) or
    la_bwd_from_fwd on the forward's workspace (from_fwd=True: the benchmark's step)."""
    has_w = dev["cos_weight"] is not None
    ws_f = None
    if from_fwd:
        n = la.workspace_size(w.B, w.Hq, w.Hkv, w.N, w.D, w.torch_dtype, w.causal, has_w, False, Dv=w.value_dim)
        ws_f = torch.empty(max(n, 1), dtype=torch.uint8, device=dev["q"].device)
    out = la.fwd(dev["q"], dev["k"], dev["v"], w.causal, w.phi, w.eps, dev["cos_weight"],
                 dev["sin_weight"], workspace=ws_f)
    dq, dk, dv = la.bwd(dev["q"], dev["k"], dev["v"], dev["grad_out"], w.causal, w.phi, w.eps,
                        dev["cos_weight"], dev["sin_weight"], fwd_workspace=ws_f)
    la.get_status()
    return out, dq, dk, dv


def run_oracle(w: gen.Workload, inp: dict):
    args = (inp["q"], inp["k"], inp["v"])
    kw = dict(is_causal=w.causal, phi=w.phi, eps=w.eps, cos_weight=inp["cos_weight"],
              sin_weight=inp["sin_weight"])
    out = oracle.fwd(*args, **kw)
    dq, dk, dv = oracle.bwd(*args, inp["grad_out"], **kw)
    return out, dq, dk, dv


def rel_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.detach().to("cpu", torch.float64).numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU result"
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def record(w: gen.Workload, errs: dict, label: str = "") -> None:
    """Append the achieved errors to the JSON-lines file named by LA_PARITY_RECORD (if set),
    so that the margin below the bar can be read after a run."""
    path = os.environ.get("LA_PARITY_RECORD")
    if not path:
        return
    fwd_path = la.kernel_path(w.B, w.Hq, w.Hkv, w.N, w.D, w.torch_dtype, w.causal, w.weights, False, Dv=w.value_dim)
    bwd_path = la.kernel_path(w.B, w.Hq, w.Hkv, w.N, w.D, w.torch_dtype, w.causal, w.weights, True, Dv=w.value_dim)
    names = {la.LA_PATH_SIMT: "simt", la.LA_PATH_TCGEN05: "tcgen05"}
    row = {"workload": w.name, "label": label, "dtype": w.dtype, "tol": TOL[w.dtype],
           "fwd_path": names[fwd_path], "bwd_path": names[bwd_path],
           "shape": [w.B, w.Hq, w.Hkv, w.N, w.D, w.value_dim], "causal": w.causal, "phi": w.phi, "eps": w.eps,
           "weights": w.weights, "errors": errs}
    d = os.path.dirname(os.path.abspath(path))
    os.makedirs(d, exist_ok=True)
    with open(path, "a") as f:
        f.write(json.dumps(row) + "\n")


def record_named(name: str, label: str, errs: dict) -> None:
    """record() for workloads of other operations (the low-rank projection)."""
    path = os.environ.get("LA_PARITY_RECORD")
    if not path:
        return
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "a") as f:
        f.write(json.dumps({"workload": name, "label": label, "dtype": "bf16", "tol": TOL["bf16"],
                            "errors": errs}) + "\n")


def compare(w: gen.Workload, got, ref, label: str = "", names=("out", "dq", "dk", "dv")):
    tol = TOL[w.dtype]
    errs = {n: rel_err(a, b) for n, a, b in zip(names, got, ref)}
    record(w, errs, label)
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"{label} {w.name}: errors {errs} exceed {tol}"
    return errs


def group_rows(w: gen.Workload, results, b: int, g: int):
    """The rows of (out, dq, dk, dv) that belong to batch b and key/value head g."""
    n_rep = w.Hq // w.Hkv
    out, dq, dk, dv = results
    hs = slice(g * n_rep, (g + 1) * n_rep)
    return out[b:b + 1, hs], dq[b:b + 1, hs], dk[b:b + 1, g:g + 1], dv[b:b + 1, g:g + 1]
