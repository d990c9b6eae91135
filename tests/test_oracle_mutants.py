"""Each plausible slip planted in a copy of the oracle (on the CPU) must fail a pin.

This shows the pins can tell a correct oracle from a wrong one: a dropped term, a wrong
sign, a transposed operand, a wrong head map, a wrong weight or a wrong derivative.
"""
import os

import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "la_oracle.c")

MUTANTS = {
    "drop_eps": ("*den = dn + eps;", "*den = dn;"),
    "gd_sign": ("gd[i] = -g_dot_num / (den * den);", "gd[i] = g_dot_num / (den * den);"),
    # (the transposed reads stay inside the P D Dv state: (p Dv + e) D + d)
    "readout_transposed_state": ("num[e] += ad * S[(p * D + d) * Dv + e];", "num[e] += ad * S[(p * Dv + e) * D + d];"),
    "dq_transposed_state": ("da += S[(p * D + d) * Dv + e] * gn[(size_t)i * Dv + e];",
                            "da += S[(p * Dv + e) * D + d] * gn[(size_t)i * Dv + e];"),
    "dv_transposed_state": ("dvh[(size_t)j * Dv + e] += R[(p * D + d) * Dv + e] * bd;",
                            "dvh[(size_t)j * Dv + e] += R[(p * Dv + e) * D + d] * bd;"),
    "gqa_head_map": ("int b = bh / Hq, h = bh % Hq, g = h / n_rep;\n        size_t kv = (size_t)b * Hkv + g;\n        head_forward",
                     "int b = bh / Hq, h = bh % Hq, g = h % Hkv;\n        size_t kv = (size_t)b * Hkv + g;\n        head_forward"),
    "sin_weight_ignored": ("return p == 0 ? cw[i] : sw[i];", "return p == 0 ? cw[i] : cw[i];"),
    "elu_derivative": ("if (phi == ORACLE_PHI_ELU1) return x > 0.0 ? 1.0 : exp(x);",
                       "if (phi == ORACLE_PHI_ELU1) return 1.0;"),
    "drop_r_term": ("double db = r[p * D + d];", "double db = 0.0;"),
    "identity_derivative": ("if (phi == ORACLE_PHI_IDENTITY) return 1.0;", "if (phi == ORACLE_PHI_IDENTITY) return 0.0;"),
    "identity_as_relu": ("if (phi == ORACLE_PHI_IDENTITY) return x;", "if (phi == ORACLE_PHI_IDENTITY) return x > 0.0 ? x : 0.0;"),
    "causal_exclusive_R": ("if (causal)\n            for (int p = 0; p < P; ++p) {  /* row i = j attends to j */",
                           "if (0)\n            for (int p = 0; p < P; ++p) {  /* row i = j attends to j */"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    fails = []
    for check in pins.ALL_CHECKS:
        if check is pins.check_finite_differences:
            continue  # slow; the other pins already cover every mutant
        fails += check(lib)
        if fails:
            break
    assert fails, f"mutant {name} passed every pin"
