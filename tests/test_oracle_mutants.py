"""Plants plausible mistakes in copies of the oracle's C source and checks that the pins catch each one.

The oracle is pinned by checks that do not reuse its formulas (brute force, closed forms, library
routines, finite differences; tests/test_oracle_pins.py).  Here every mutant -- a dropped term, a sign
or index error, a transposed operand, an off-by-one limit -- is built with the same compiler flags,
swapped in for the real library, and must make at least one pin fail.  CPU only.
"""
import os
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

# (name, text in oracle.c, replacement): each text occurs exactly once
MUTANTS = [
    ("forward scores read K transposed", "for (long c = 0; c < d; ++c) acc += qrow[c] * kj[c];",
     "for (long c = 0; c < d; ++c) acc += qrow[c] * k[c * nk + j];"),
    ("forward exponent sign", "        s[j] = exp(s[j] - m);\n        l += s[j];",
     "        s[j] = exp(m - s[j]);\n        l += s[j];"),
    ("forward probabilities not normalised", "const double p = s[j] / l;", "const double p = s[j];"),
    ("forward LSE without the log", "if (lse) *lse = m + log(l);\n}", "if (lse) *lse = m + l;\n}"),
    ("forward scale applied twice", "        s[j] = scale * acc;\n    }\n    /* pass 1",
     "        s[j] = scale * scale * acc;\n    }\n    /* pass 1"),
    ("forward row limit one short", "limits[i], d, scale, s);", "limits[i] - (limits[i] > 1), d, scale, s);"),
    ("partial state drops the weights", "for (long c = 0; c < d; ++c) o[c] += e * v[j * d + c];",
     "for (long c = 0; c < d; ++c) o[c] += v[j * d + c];"),
    ("merge weight sign", "const double wa = (ma == -INFINITY) ? 0.0 : exp(ma - M);",
     "const double wa = (ma == -INFINITY) ? 0.0 : exp(M - ma);"),
    ("decode chunk drops its last key", "long a = c * L, b = a + L;", "long a = c * L, b = a + L - 1;"),
    ("backward dS sign of D", "const double ds = p[j] * (dp - Di);", "const double ds = p[j] * (dp + Di);"),
    ("backward dK uses dO instead of Q", "dk[j * d + c] += scale * ds * q[i * d + c];",
     "dk[j * d + c] += scale * ds * dout[i * d + c];"),
    ("backward dV uses O instead of dO", "for (long c = 0; c < d; ++c) dv[j * d + c] += p[j] * go[c];",
     "for (long c = 0; c < d; ++c) dv[j * d + c] += p[j] * orow[c];"),
    ("backward dQ misses the scale", "dq[i * d + c] += scale * ds * k[j * d + c];",
     "dq[i * d + c] += ds * k[j * d + c];"),
]

# the pins run against each mutant (parametrised pins with one representative case)
PINS = [
    (pins.test_brute_force_mpmath, dict(nq=3, nk=5, d=4, scale=0.5)),
    (pins.test_brute_force_mpmath, dict(nq=16, nk=11, d=16, scale=0.25)),
    (pins.test_large_scores_need_max_subtraction, {}),
    (pins.test_probabilities_exposed_by_identity_values, {}),
    (pins.test_single_key, {}),
    (pins.test_uniform_scores_average_values, dict(zero="keys")),
    (pins.test_constant_values, {}),
    (pins.test_permutation_invariances, {}),
    (pins.test_library_sdpa_rectangular, {}),
    (pins.test_merge_order_invariance, {}),
    (pins.test_empty_state_is_identity, {}),
    (pins.test_decode_split_equals_full, dict(nk=100, splits=7)),
    (pins.test_tiled_forms_agree, dict(nq=200, nk=333, Br=64, Bc=48)),
    (pins.test_causal_brute_force, dict(nq=5, nk=12)),
    (pins.test_causal_library_and_closed_forms, {}),
    (pins.test_backward_finite_differences, dict(causal=True, hkv=1)),
    (pins.test_backward_autograd_library, {}),
    (pins.test_backward_page_dv_setup, {}),
]


def _caught(fn, kw) -> bool:
    try:
        fn(**kw)
    except AssertionError:
        return True
    except (ValueError, ArithmeticError, RuntimeError):  # e.g. non-finite results rejected by a library
        return True
    return False


def test_unmutated_source_passes_every_pin():
    with tempfile.TemporaryDirectory() as tmp:
        so = oracle.compile_c(oracle.source_path(), os.path.join(tmp, "liboracle_copy.so"))
        with oracle.swapped_library(so):
            failing = [fn.__name__ for fn, kw in PINS if _caught(fn, kw)]
    assert not failing, failing


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    src = open(oracle.source_path()).read()
    assert src.count(old) == 1, f"mutation point not unique or missing: {old!r}"
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "oracle_mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        so = oracle.compile_c(path, os.path.join(tmp, "liboracle_mutant.so"))
        with oracle.swapped_library(so):
            caught = [fn.__name__ for fn, kw in PINS if _caught(fn, kw)]
    assert caught, f"no pin catches the mutant '{name}'"
