"""The float64 low-rank oracle against pins that do not come from itself (CPU only):
explicit index sums on tiny inputs, special weights with closed forms, the merged-weight
contraction order, central finite differences and exact gradient identities.  A few planted
slips in a copy of the oracle must each fail a pin."""
import itertools

import numpy as np
import pytest

from oracle import low_rank as lr


def case(M, K_in, r, K_out, seed, bias=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K_in))
    V = rng.standard_normal((r, K_in))
    U = rng.standard_normal((K_out, r))
    b = rng.standard_normal(K_out) if bias else None
    g = rng.standard_normal((M, K_out))
    return x, U, V, b, g


def loops_forward(x, U, V, b):
    """y[m][o] = sum_j U[o][j] sum_i x[m][i] V[j][i] + b[o], as explicit index sums."""
    M, K_in = x.shape
    K_out, r = U.shape
    y = np.zeros((M, K_out))
    for m, o in itertools.product(range(M), range(K_out)):
        s = 0.0
        for j in range(r):
            t = 0.0
            for i in range(K_in):
                t += x[m, i] * V[j, i]
            s += U[o, j] * t
        y[m, o] = s + (b[o] if b is not None else 0.0)
    return y


def rel(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b))) / max(np.max(np.abs(b)), 1e-300))


def pins(impl):
    """Every pin of the low-rank oracle `impl` (a module with fwd/bwd); returns failures."""
    fails = []
    x, U, V, b, g = case(3, 5, 2, 4, seed=1)
    if rel(impl.fwd(x, U, V, b), loops_forward(x, U, V, b)) > 1e-13:
        fails.append("index sums")
    if rel(impl.fwd(x, U, V, None), loops_forward(x, U, V, None)) > 1e-13:
        fails.append("index sums without bias")
    # identity weights: U = V = I_r gives y = x + b
    x2, _, _, b2, _ = case(4, 3, 3, 3, seed=2)
    eye = np.eye(3)
    if rel(impl.fwd(x2, eye, eye, b2), x2 + b2) > 1e-15:
        fails.append("identity weights")
    # rank one: y = (x . v) u^T + b
    x3, U3, V3, b3, _ = case(5, 4, 1, 3, seed=3)
    want = np.outer(x3 @ V3[0], U3[:, 0]) + b3
    if rel(impl.fwd(x3, U3, V3, b3), want) > 1e-14:
        fails.append("rank one")
    # contraction order: (x V^T) U^T = x (U V)^T
    x4, U4, V4, b4, g4 = case(6, 7, 3, 5, seed=4)
    if rel(impl.fwd(x4, U4, V4, b4), x4 @ (U4 @ V4).T + b4) > 1e-13:
        fails.append("merged weights")
    # gradients: central finite differences of L = sum g * fwd
    dx, dU, dV, db = impl.bwd(x4, U4, V4, g4, b4)
    h = 1e-6
    for name, arr, grad in (("x", x4, dx), ("U", U4, dU), ("V", V4, dV), ("b", b4, db)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            ap, am = arr.copy(), arr.copy()
            ap[idx] += h
            am[idx] -= h
            args_p = {"x": x4, "U": U4, "V": V4, "b": b4}
            args_m = dict(args_p)
            args_p[name], args_m[name] = ap, am
            lp = np.sum(g4 * impl.fwd(args_p["x"], args_p["U"], args_p["V"], args_p["b"]))
            lm = np.sum(g4 * impl.fwd(args_m["x"], args_m["U"], args_m["V"], args_m["b"]))
            fd[idx] = (lp - lm) / (2 * h)
        if rel(grad, fd) > 1e-7:
            fails.append(f"finite differences d{name}")
    # y - b is degree-1 homogeneous in x, in U and in V: sum a * da = sum g * (y - b) for each
    yb = impl.fwd(x4, U4, V4, None)
    s = float(np.sum(g4 * yb))
    for name, a, da in (("x", x4, dx), ("U", U4, dU), ("V", V4, dV)):
        if abs(float(np.sum(a * da)) - s) > 1e-12 * max(1.0, abs(s)):
            fails.append(f"homogeneity in {name}")
    if db is None or rel(db, g4.sum(0)) > 1e-15:
        fails.append("bias gradient")
    if impl.bwd(x4, U4, V4, g4, None)[3] is not None:
        fails.append("no bias gradient without a bias")
    return fails


def test_pins_hold():
    assert pins(lr) == []


class _Mutant:
    """A copy of the oracle with one plausible slip planted."""

    def __init__(self, name):
        self.name = name

    def fwd(self, x, U, V, bias=None):
        x, U, V, bias = (lr._f64(a) for a in (x, U, V, bias))
        y = (x @ V.T) @ U.T
        if self.name == "drop_bias":
            return y
        if self.name == "bias_twice" and bias is not None:
            return y + 2.0 * bias[None, :]
        return y + (bias[None, :] if bias is not None else 0.0)

    def bwd(self, x, U, V, g, bias=None):
        x, U, V, g, bias = (lr._f64(a) for a in (x, U, V, g, bias))
        t = x @ V.T
        dt = g @ U
        dx, dU, dV = dt @ V, g.T @ t, dt.T @ x
        db = g.sum(0) if bias is not None else None
        if self.name == "dV_from_t":       # t where dt belongs
            dV = t.T @ x
        if self.name == "dU_from_dt":      # dt where t belongs
            dU = g.T @ dt
        if self.name == "db_mean":         # mean over rows instead of the sum
            db = g.mean(0) if bias is not None else None
        return dx, dU, dV, db


@pytest.mark.parametrize("name", ["drop_bias", "bias_twice", "dV_from_t", "dU_from_dt", "db_mean"])
def test_mutant_is_caught(name):
    assert pins(_Mutant(name)), f"mutant {name} passed every pin"
