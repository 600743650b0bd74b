"""The oracle's pins reject plausible mistakes.

Each case plants one mistake in a copy of oracle.c (a dropped term, a wrong
sign, a transposed operand, a swapped gate/up block, a reversed tie-break, a
missing renormalisation, a wrong bit shift), builds it in a temporary
directory, loads it in place of the real oracle and runs every pin in
test_oracle_pins. At least one pin must fail for every mutation. CPU only.
"""
import inspect
import warnings
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "silu_sign": ("double v = a / (1.0 + exp(-a)) * b;", "double v = a / (1.0 + exp(a)) * b;"),
    "gate_up_swapped": ("const uint16_t* w1 = W13 + i * H;", "const uint16_t* w1 = W13 + (I + i) * H;"),
    "transposed_weight": ("bf16_to_f64(xr[k]) * bf16_to_f64(wr[k]);\n                acc += p;",
                          "bf16_to_f64(xr[k]) * bf16_to_f64(W[k * N + n]);\n                acc += p;"),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k) {\n                double p = bf16_to_f64",
                          "for (int64_t k = 0; k + 1 < K; ++k) {\n                double p = bf16_to_f64"),
    "absref_without_abs": ("accabs += fabs(p);\n            }\n            y[m * N + n] = acc;\n            if (absref) absref[m * N + n] = accabs;\n        }\n    }\n}\n\n/* Same product with double",
                           "accabs += p;\n            }\n            y[m * N + n] = acc;\n            if (absref) absref[m * N + n] = accabs;\n        }\n    }\n}\n\n/* Same product with double"),
    "tie_break_reversed": ("return (a->i < b->i) ? -1 : (a->i > b->i) ? 1 : 0;",
                           "return (a->i < b->i) ? 1 : (a->i > b->i) ? -1 : 0;"),
    "gates_not_renormalised": ("for (int64_t j = 0; j < k; ++j) denom += exp(buf[j].v - lmax);",
                               "for (int64_t j = 0; j < E; ++j) denom += exp(buf[j].v - lmax);"),
    "splitk_drops_remainder": ("int64_t k0 = s * K / S, k1 = (s + 1) * K / S;",
                               "int64_t k0 = s * (K / S), k1 = (s + 1) * (K / S);"),
    "bf16_shift": ("uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)b) << 15;"),
    "round_truncates": ("double q = nearbyint(ldexp(m, 8));", "double q = floor(ldexp(m, 8));"),
    "up_dropped": ("double v = a / (1.0 + exp(-a)) * b;", "double v = a / (1.0 + exp(-a));"),
}


def _pins():
    return [(n, f) for n, f in inspect.getmembers(pins, inspect.isfunction)
            if n.startswith("test_") and "S" not in inspect.signature(f).parameters]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutation(name, tmp_path):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, "mutation anchor not found: " + name
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(before, after))
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                    str(mutated), "-lm"], check=True)
    old = oracle.swap_library(str(so))
    failed = []
    try:
        for n, f in _pins():
            try:
                with warnings.catch_warnings():
                    warnings.simplefilter("ignore")
                    f()
            except Exception:
                failed.append(n)
        for S in (3, 7):   # the split-K pin is parametrised
            try:
                pins.test_linear_splitk_equals_unsplit(S)
            except Exception:
                failed.append("test_linear_splitk_equals_unsplit[%d]" % S)
    finally:
        oracle.restore_library(old)
    assert failed, "no pin caught mutation " + name
