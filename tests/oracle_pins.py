"""Independent pins for the float64 oracle.

Each check compares the oracle with something that is not the oracle:

* ``brute_forward``: the quadratic form of the definition,
  out_i = sum_{j in J(i)} W_ij (phi(q_i).phi(k_j)) v_j / (sum_{j in J(i)} W_ij (phi(q_i).phi(k_j)) + eps)
  with W_ij = sum_p w_i^p w_j^p (1 without position weights), written with matrix
  products, against the oracle's recurrent prefix sums;
* ``autograd_backward``: torch autograd (float64) of that quadratic form, which is what
  the linear_attn page's ``bwd`` returns (the gradient of ``fwd``), against the oracle's
  hand-derived gradients;
* central finite differences of the oracle's own forward;
* closed forms and symmetries (row 0, N = 1, key permutations, all-ones values, dead
  relu rows, causal last row equals bidirectional last row, the cos/sin identity);
* the grouped-query rule of the gqa page: expand k, v with h -> h // n_rep, run every
  query head on its own, then sum dk, dv with view(B, Hkv, n_rep, N, D).sum(2);
* a value width Dv different from the head dimension D: the quadratic form and its
  autograd at Dv != D, and the independence of the value columns (splitting v and g into
  column blocks gives out and dv block by block, and dq, dk as the sum over the blocks,
  every block sharing one den).

The helpers here never call the CUDA library.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle


def phi_np(x, phi):
    if phi == "elu+1":
        return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    if phi == "identity":
        return x
    return np.maximum(x, 0.0)


def phi_torch(x, phi):
    if phi == "elu+1":
        return torch.nn.functional.elu(x) + 1.0
    if phi == "identity":
        return x
    return torch.relu(x)


def expand_kv(k, n_rep):
    """k [B, Hkv, N, D] -> [B, Hkv * n_rep, N, D] with query head h reading kv head h // n_rep."""
    return np.repeat(k, n_rep, axis=1)


def brute_forward(q, k, v, causal, phi, eps, cw=None, sw=None):
    """Quadratic-form definition, numpy float64.  q [B,Hq,N,D], k, v [B,Hkv,N,D]."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    n_rep = q.shape[1] // k.shape[1]
    ke, ve = expand_kv(k, n_rep), expand_kv(v, n_rep)
    N = q.shape[2]
    if cw is None:
        W = np.ones((N, N))
    else:
        cw, sw = np.asarray(cw, np.float64), np.asarray(sw, np.float64)
        W = np.outer(cw, cw) + np.outer(sw, sw)
    if causal:
        W = np.tril(W)
    A = np.einsum("bhid,bhjd->bhij", phi_np(q, phi), phi_np(ke, phi)) * W
    return (A @ ve) / (A.sum(-1, keepdims=True) + eps)


def brute_forward_torch(q, k, v, causal, phi, eps, cw=None, sw=None):
    """The same quadratic form in torch float64 (differentiable)."""
    n_rep = q.shape[1] // k.shape[1]
    ke = k.repeat_interleave(n_rep, dim=1)
    ve = v.repeat_interleave(n_rep, dim=1)
    N = q.shape[2]
    if cw is None:
        W = torch.ones(N, N, dtype=torch.float64)
    else:
        W = torch.outer(cw, cw) + torch.outer(sw, sw)
    if causal:
        W = torch.tril(W)
    A = torch.einsum("bhid,bhjd->bhij", phi_torch(q, phi), phi_torch(ke, phi)) * W
    return (A @ ve) / (A.sum(-1, keepdim=True) + eps)


def autograd_backward(q, k, v, g, causal, phi, eps, cw=None, sw=None):
    t = [torch.tensor(np.asarray(x, np.float64), requires_grad=True) for x in (q, k, v)]
    cwt = None if cw is None else torch.tensor(np.asarray(cw, np.float64))
    swt = None if sw is None else torch.tensor(np.asarray(sw, np.float64))
    out = brute_forward_torch(*t, causal, phi, eps, cwt, swt)
    grads = torch.autograd.grad(out, t, torch.tensor(np.asarray(g, np.float64)))
    return tuple(x.numpy() for x in grads)


def rand_case(B, Hq, Hkv, N, D, seed, weights=False, scale=1.0, avoid_kink=False, positive=False, Dv=None):
    """Random case; positive=True draws |N(0,1)| for q and k (identity feature map, whose
    features the pages call non-negative); Dv is the value width (D when None)."""
    rng = np.random.default_rng(seed)
    Dv = D if Dv is None else Dv
    q = rng.standard_normal((B, Hq, N, D)) * scale
    k = rng.standard_normal((B, Hkv, N, D)) * scale
    if positive:
        q, k = np.abs(q), np.abs(k)
    v = rng.standard_normal((B, Hkv, N, Dv))
    g = rng.standard_normal((B, Hq, N, Dv))
    if avoid_kink:  # keep relu inputs away from 0 for finite differences
        for x in (q, k):
            x[np.abs(x) < 1e-2] += 0.05
    cw = sw = None
    if weights:
        i = np.arange(N, dtype=np.float64)
        cw, sw = np.cos(np.pi * i / (2 * N)), np.sin(np.pi * i / (2 * N))
    return q, k, v, g, cw, sw


def rel_err(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


MODES = [
    # (causal, phi, weights, Hq, Hkv)
    (True, "elu+1", False, 2, 2),
    (False, "elu+1", False, 2, 2),
    (True, "relu", False, 2, 2),
    (False, "relu", False, 2, 2),
    (True, "relu", True, 2, 2),
    (False, "elu+1", True, 2, 2),
    (True, "elu+1", False, 4, 2),
    (False, "relu", True, 6, 2),
    (True, "identity", False, 2, 2),
    (False, "identity", True, 4, 2),
]


def check_forward_brute(lib=None, tol=1e-12):
    fails = []
    for idx, (causal, phi, weights, Hq, Hkv) in enumerate(MODES):
        q, k, v, g, cw, sw = rand_case(2, Hq, Hkv, 9, 5, seed=100 + idx, weights=weights,
                                       positive=phi == "identity")
        ref = brute_forward(q, k, v, causal, phi, 1e-6, cw, sw)
        got = oracle.fwd(q, k, v, causal, phi, 1e-6, cw, sw, lib=lib)
        e = rel_err(got, ref)
        if not e <= tol:
            fails.append(f"fwd brute mode={idx} err={e:.3e}")
    return fails


def check_backward_autograd(lib=None, tol=1e-10):
    fails = []
    for idx, (causal, phi, weights, Hq, Hkv) in enumerate(MODES):
        q, k, v, g, cw, sw = rand_case(2, Hq, Hkv, 7, 4, seed=200 + idx, weights=weights,
                                       positive=phi == "identity")
        ref = autograd_backward(q, k, v, g, causal, phi, 1e-6, cw, sw)
        got = oracle.bwd(q, k, v, g, causal, phi, 1e-6, cw, sw, lib=lib)
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            e = rel_err(a, b)
            if not e <= tol:
                fails.append(f"bwd autograd mode={idx} {name} err={e:.3e}")
    return fails


def check_gqa_rule(lib=None, tol=1e-13):
    """Grouped heads equal expanded heads followed by the group sum of dk, dv."""
    fails = []
    B, Hq, Hkv, N, D = 2, 6, 2, 8, 3
    n_rep = Hq // Hkv
    for causal in (True, False):
        q, k, v, g, cw, sw = rand_case(B, Hq, Hkv, N, D, seed=300 + causal, weights=True)
        out = oracle.fwd(q, k, v, causal, "elu+1", 1e-6, cw, sw, lib=lib)
        dq, dk, dv = oracle.bwd(q, k, v, g, causal, "elu+1", 1e-6, cw, sw, lib=lib)
        ke, ve = expand_kv(k, n_rep), expand_kv(v, n_rep)
        out_x = oracle.fwd(q, ke, ve, causal, "elu+1", 1e-6, cw, sw, lib=lib)
        dq_x, dk_x, dv_x = oracle.bwd(q, ke, ve, g, causal, "elu+1", 1e-6, cw, sw, lib=lib)
        dk_r = dk_x.reshape(B, Hkv, n_rep, N, D).sum(2)
        dv_r = dv_x.reshape(B, Hkv, n_rep, N, D).sum(2)
        for name, a, b in (("out", out, out_x), ("dq", dq, dq_x), ("dk", dk, dk_r), ("dv", dv, dv_r)):
            e = rel_err(a, b)
            if not e <= tol:
                fails.append(f"gqa causal={causal} {name} err={e:.3e}")
        # the head map itself: query head h must match a single-head run on kv head h // n_rep
        for h in range(Hq):
            one = oracle.fwd(q[:, h:h + 1], k[:, h // n_rep:h // n_rep + 1],
                             v[:, h // n_rep:h // n_rep + 1], causal, "elu+1", 1e-6, cw, sw, lib=lib)
            e = rel_err(out[:, h:h + 1], one)
            if not e <= tol:
                fails.append(f"gqa head map h={h} err={e:.3e}")
    return fails


def check_closed_forms(lib=None):
    fails = []
    eps = 1e-6
    for phi in ("elu+1", "relu", "identity"):
        q, k, v, g, _, _ = rand_case(1, 1, 1, 5, 4, seed=400, scale=1.0)
        q[..., 0, :] = np.abs(q[..., 0, :]) + 0.1  # keep row 0 alive under relu
        k[..., 0, :] = np.abs(k[..., 0, :]) + 0.1
        out = oracle.fwd(q, k, v, True, phi, eps, lib=lib)
        s = float(np.dot(phi_np(q[0, 0, 0], phi), phi_np(k[0, 0, 0], phi)))
        want = v[0, 0, 0] * s / (s + eps)
        if rel_err(out[0, 0, 0], want) > 1e-14:
            fails.append(f"row0 closed form phi={phi}")
        for causal in (True, False):  # N = 1
            o1 = oracle.fwd(q[:, :, :1], k[:, :, :1], v[:, :, :1], causal, phi, eps, lib=lib)
            if rel_err(o1[0, 0, 0], want) > 1e-14:
                fails.append(f"N=1 closed form phi={phi} causal={causal}")
    # identity uses the features as given, signs included: row 0 with mixed signs and
    # s = q_0 . k_0 = 1.75 > 0, eps = 1: out_0 = v_0 s / (s + 1)
    q0 = np.array([[[[1.0, -0.5, 2.0, -1.0]]]])
    k0 = np.array([[[[0.5, 1.0, 1.0, 0.25]]]])
    v0 = np.array([[[[3.0, -1.0, 0.5, 2.0]]]])
    o = oracle.fwd(q0, k0, v0, True, "identity", 1.0, lib=lib)
    if rel_err(o[0, 0, 0], v0[0, 0, 0] * 1.75 / 2.75) > 1e-14:
        fails.append("identity row0 closed form with mixed signs")
    return fails


def check_symmetries(lib=None):
    fails = []
    rng = np.random.default_rng(7)
    for phi in ("elu+1", "relu"):
        q, k, v, g, cw, sw = rand_case(1, 2, 2, 11, 4, seed=500)
        base = oracle.fwd(q, k, v, False, phi, 1e-6, lib=lib)
        perm = rng.permutation(11)
        if rel_err(oracle.fwd(q, k[:, :, perm], v[:, :, perm], False, phi, 1e-6, lib=lib), base) > 1e-13:
            fails.append(f"bidir key permutation phi={phi}")
        if rel_err(oracle.fwd(q[:, :, perm], k, v, False, phi, 1e-6, lib=lib), base[:, :, perm]) > 1e-13:
            fails.append(f"bidir query permutation phi={phi}")
        causal = oracle.fwd(q, k, v, True, phi, 1e-6, lib=lib)
        if rel_err(causal[:, :, -1], base[:, :, -1]) > 1e-13:
            fails.append(f"causal last row vs bidir phi={phi}")
        ones = np.ones_like(v)
        o = oracle.fwd(q, k, ones, True, phi, 0.25, lib=lib)
        A = np.tril(phi_np(q[0, 0], phi) @ phi_np(k[0, 0], phi).T).sum(-1)
        if rel_err(o[0, 0, :, 0], A / (A + 0.25)) > 1e-13 or np.ptp(o[0, 0], axis=-1).max() > 1e-15:
            fails.append(f"ones values phi={phi}")
    # dead relu row: out_i = 0, dq_i = 0
    q, k, v, g, _, _ = rand_case(1, 1, 1, 6, 3, seed=501)
    q[0, 0, 3] = -np.abs(q[0, 0, 3]) - 0.1
    o = oracle.fwd(q, k, v, True, "relu", 1e-6, lib=lib)
    dq, _, _ = oracle.bwd(q, k, v, g, True, "relu", 1e-6, lib=lib)
    if np.any(o[0, 0, 3] != 0) or np.any(dq[0, 0, 3] != 0):
        fails.append("dead relu row")
    # cos/sin identity: c_i c_j + s_i s_j = cos(pi (i - j) / (2N)) gives the same result
    q, k, v, g, cw, sw = rand_case(1, 1, 1, 10, 3, seed=502, weights=True)
    N = 10
    Wc = np.cos(np.pi * (np.arange(N)[:, None] - np.arange(N)[None, :]) / (2 * N))
    A = np.tril(phi_np(q[0, 0], "relu") @ phi_np(k[0, 0], "relu").T * Wc)
    want = (A @ v[0, 0]) / (A.sum(-1, keepdims=True) + 1e-6)
    if rel_err(oracle.fwd(q, k, v, True, "relu", 1e-6, cw, sw, lib=lib)[0, 0], want) > 1e-12:
        fails.append("cosine difference identity")
    return fails


def check_gradient_identities(lib=None):
    """Exact identities of the hand-derived gradients (homogeneity in v; the
    denominator's eps term)."""
    fails = []
    for causal in (True, False):
        q, k, v, g, _, _ = rand_case(1, 1, 1, 8, 3, seed=600 + causal)
        out = oracle.fwd(q, k, v, causal, "elu+1", 0.3, lib=lib)
        dq, dk, dv = oracle.bwd(q, k, v, g, causal, "elu+1", 0.3, lib=lib)
        # out is degree-1 homogeneous in v: sum_j v_j . dv_j = sum_i g_i . out_i
        lhs, rhs = float(np.sum(v * dv)), float(np.sum(g * out))
        if abs(lhs - rhs) > 1e-12 * max(1.0, abs(rhs)):
            fails.append(f"v homogeneity causal={causal}")
    return fails


def phi_grad_np(x, phi):
    if phi == "elu+1":
        return np.where(x > 0, 1.0, np.exp(np.minimum(x, 0.0)))
    if phi == "identity":
        return np.ones_like(x)
    return (x > 0).astype(np.float64)


def check_scaling_identities(lib=None, tol=1e-11):
    """Exact identities of the gradient with respect to the features a_i = w_i phi(q_i) and
    b_j = w_j phi(k_j) (da = dq / phi'(q), db = dk / phi'(k) elementwise; phi' > 0 for elu+1
    and identity).  num_i and den_i - eps are bilinear in (a, b), so
      per row:  sum_d a_id da_id = eps (g_i . out_i) / den_i   (scale a_i alone),
      overall:  sum_j b_j . db_j = sum_i a_i . da_i            (scale every a, or every b),
    with den_i from the quadratic form, not from the oracle."""
    fails = []
    cases = [(True, "elu+1", False, 2, 2), (False, "elu+1", True, 4, 2), (True, "identity", True, 6, 3),
             (False, "identity", False, 2, 1)]
    for idx, (causal, phi, weights, Hq, Hkv) in enumerate(cases):
        eps = 0.7
        q, k, v, g, cw, sw = rand_case(2, Hq, Hkv, 7, 4, seed=900 + idx, weights=weights,
                                       positive=phi == "identity", Dv=5)
        out = oracle.fwd(q, k, v, causal, phi, eps, cw, sw, lib=lib)
        dq, dk, _ = oracle.bwd(q, k, v, g, causal, phi, eps, cw, sw, lib=lib)
        N = q.shape[2]
        W = np.ones((N, N)) if cw is None else np.outer(cw, cw) + np.outer(sw, sw)
        if causal:
            W = np.tril(W)
        n_rep = Hq // Hkv
        A = np.einsum("bhid,bhjd->bhij", phi_np(q, phi), phi_np(expand_kv(k, n_rep), phi)) * W
        den = A.sum(-1) + eps
        # a . da with a = w phi(q) and da = dq / (w phi'(q)): the weights cancel
        a_da = np.sum(phi_np(q, phi) * dq / phi_grad_np(q, phi), axis=-1)
        b_db = np.sum(phi_np(k, phi) * dk / phi_grad_np(k, phi))
        want = eps * np.sum(g * out, axis=-1) / den
        e = rel_err(a_da, want)
        if not e <= tol:
            fails.append(f"per-row a.da identity case={idx} err={e:.3e}")
        if abs(b_db - a_da.sum()) > tol * max(1.0, abs(a_da.sum()), np.abs(a_da).sum()):
            fails.append(f"b.db = a.da identity case={idx}: {b_db} vs {a_da.sum()}")
    return fails


def check_value_width(lib=None, tol_fwd=1e-12, tol_bwd=1e-10, tol_split=1e-13):
    """Dv != D: quadratic form and its autograd, and the value columns' independence."""
    fails = []
    cases = [(True, "elu+1", False, 2, 2, 5, 3), (False, "relu", True, 4, 2, 4, 7), (True, "relu", True, 6, 2, 3, 8),
             (False, "identity", False, 2, 1, 6, 2), (True, "elu+1", True, 2, 1, 2, 9)]
    for idx, (causal, phi, weights, Hq, Hkv, D, Dv) in enumerate(cases):
        q, k, v, g, cw, sw = rand_case(2, Hq, Hkv, 9, D, seed=800 + idx, weights=weights,
                                       positive=phi == "identity", Dv=Dv)
        out = oracle.fwd(q, k, v, causal, phi, 1e-6, cw, sw, lib=lib)
        e = rel_err(out, brute_forward(q, k, v, causal, phi, 1e-6, cw, sw))
        if not e <= tol_fwd:
            fails.append(f"value width fwd brute case={idx} err={e:.3e}")
        got = oracle.bwd(q, k, v, g, causal, phi, 1e-6, cw, sw, lib=lib)
        for name, a, b in zip(("dq", "dk", "dv"), got, autograd_backward(q, k, v, g, causal, phi, 1e-6, cw, sw)):
            e = rel_err(a, b)
            if not e <= tol_bwd:
                fails.append(f"value width bwd autograd case={idx} {name} err={e:.3e}")
        # column blocks [0, c) and [c, Dv): out and dv side by side, dq and dk summed
        c = Dv // 2
        parts = [(v[..., :c], g[..., :c]), (v[..., c:], g[..., c:])]
        outs = [oracle.fwd(q, k, vb, causal, phi, 1e-6, cw, sw, lib=lib) for vb, _ in parts]
        grads = [oracle.bwd(q, k, vb, gb, causal, phi, 1e-6, cw, sw, lib=lib) for vb, gb in parts]
        for name, a, b in (("out", out, np.concatenate(outs, -1)),
                           ("dq", got[0], grads[0][0] + grads[1][0]),
                           ("dk", got[1], grads[0][1] + grads[1][1]),
                           ("dv", got[2], np.concatenate([grads[0][2], grads[1][2]], -1))):
            e = rel_err(a, b)
            if not e <= tol_split:
                fails.append(f"value width column split case={idx} {name} err={e:.3e}")
    return fails


def check_finite_differences(lib=None, h=1e-6, tol=1e-6):
    fails = []
    cases = [(True, "elu+1", False, 2, 1, 3), (False, "relu", False, 1, 1, 3), (True, "relu", True, 2, 2, 3),
             (False, "elu+1", True, 2, 1, 3), (True, "identity", False, 2, 1, 3), (True, "elu+1", True, 2, 1, 5)]
    for idx, (causal, phi, weights, Hq, Hkv, Dv) in enumerate(cases):
        q, k, v, g, cw, sw = rand_case(1, Hq, Hkv, 5, 3, seed=700 + idx, weights=weights,
                                       avoid_kink=True, positive=phi == "identity", Dv=Dv)
        dq, dk, dv = oracle.bwd(q, k, v, g, causal, phi, 1e-6, cw, sw, lib=lib)
        for name, x, dx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            fd = np.zeros_like(x)
            it = np.nditer(x, flags=["multi_index"])
            for _ in it:
                m = it.multi_index
                xp, xm = x.copy(), x.copy()
                xp[m] += h
                xm[m] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = {"q": q, "k": k, "v": v}
                args_p[name], args_m[name] = xp, xm
                lp = np.sum(g * oracle.fwd(args_p["q"], args_p["k"], args_p["v"], causal, phi, 1e-6, cw, sw, lib=lib))
                lm = np.sum(g * oracle.fwd(args_m["q"], args_m["k"], args_m["v"], causal, phi, 1e-6, cw, sw, lib=lib))
                fd[m] = (lp - lm) / (2 * h)
            e = rel_err(dx, fd)
            if not e <= tol:
                fails.append(f"finite differences case={idx} d{name} err={e:.3e}")
    return fails


ALL_CHECKS = [check_forward_brute, check_backward_autograd, check_gqa_rule, check_closed_forms,
              check_symmetries, check_gradient_identities, check_scaling_identities, check_value_width,
              check_finite_differences]


def run_all(lib=None):
    fails = []
    for c in ALL_CHECKS:
        fails += c(lib)
    return fails
