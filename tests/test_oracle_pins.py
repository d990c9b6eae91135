"""The float64 oracle against pins that do not come from itself (CPU only)."""
import glob
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import oracle_pins as pins

GOLDEN = sorted(glob.glob(os.path.join(os.path.dirname(__file__), "golden", "*.json")))


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    fails = check()
    assert not fails, fails


def _frac_array(x):
    return np.vectorize(lambda s: float(Fraction(s)))(np.array(x, dtype=object)).astype(np.float64)


@pytest.mark.parametrize("path", GOLDEN, ids=os.path.basename)
def test_golden_hand_derived(path):
    case = json.load(open(path))
    assert case["cite"] and case["derivation"]
    q, k, v, g = (_frac_array(case[n]) for n in ("q", "k", "v", "grad_out"))
    cw = _frac_array(case["cos_weight"]) if "cos_weight" in case else None
    sw = _frac_array(case["sin_weight"]) if "sin_weight" in case else None
    eps = float(Fraction(case["eps"]))
    out = oracle.fwd(q, k, v, case["is_causal"], case["phi"], eps, cw, sw)
    dq, dk, dv = oracle.bwd(q, k, v, g, case["is_causal"], case["phi"], eps, cw, sw)
    for name, got in (("out", out), ("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(got, _frac_array(case[name]), rtol=1e-14, atol=1e-15, err_msg=name)


def test_thread_count_does_not_change_result(monkeypatch):
    q, k, v, g, cw, sw = pins.rand_case(2, 4, 2, 16, 4, seed=1, weights=True)
    a = oracle.bwd(q, k, v, g, True, "elu+1", 1e-6, cw, sw)
    b = oracle.bwd(q, k, v, g, True, "elu+1", 1e-6, cw, sw)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_argument_checks():
    q, k, v, g, cw, sw = pins.rand_case(1, 3, 2, 4, 2, seed=2)
    with pytest.raises(ValueError):
        oracle.fwd(q, k, v)          # 3 query heads over 2 kv heads
    q, k, v, g, cw, sw = pins.rand_case(1, 2, 2, 4, 2, seed=2, weights=True)
    with pytest.raises(ValueError):
        oracle.fwd(q, k, v, True, "relu", 1e-6, cw, None)
