"""Plant plausible mistakes in a COPY of the oracle's C source and check that
the pins catch every one of them (all on the CPU; nothing is planted in the
product library).
"""
import ctypes
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "kda_oracle.c")
GOLDEN = os.path.join(HERE, "golden", "kda_worked_examples_2x2.json")

# (name, text in the source, replacement)
MUTANTS = [
    ("decay_rows_not_columns", "S[(size_t)i * dk + c] *= alpha[c];",
     "S[(size_t)i * dk + c] *= alpha[i % dk];"),
    ("decay_sign", "alpha[c] = exp(g[c]);", "alpha[c] = exp(-g[c]);"),
    ("delta_sign", "double u = beta * (v[i] - r);\n        for (int c = 0; c < dk; ++c) s[c] += u * kh[c];\n    }\n    /* output",
     "double u = beta * (v[i] + r);\n        for (int c = 0; c < dk; ++c) s[c] += u * kh[c];\n    }\n    /* output"),
    ("update_sign", "for (int c = 0; c < dk; ++c) s[c] += u * kh[c];\n    }\n    /* output",
     "for (int c = 0; c < dk; ++c) s[c] -= u * kh[c];\n    }\n    /* output"),
    ("beta_sign", "return 1.0 / (1.0 + exp(-b));", "return 1.0 / (1.0 + exp(b));"),
    ("output_reads_key", "acc += s[c] * qh[c];", "acc += s[c] * kh[c];"),
    ("output_unscaled", "o[i] = scale * acc;", "o[i] = acc;"),
    ("key_not_normalised", "l2norm(dk, k, eps, kh);", "memcpy(kh, k, sizeof(double) * (size_t)dk);"),
    ("dropped_beta", "double u = beta * (v[i] - r);\n        for (int c = 0; c < dk; ++c) s[c] += u * kh[c];\n    }\n    /* output",
     "double u = (v[i] - r);\n        for (int c = 0; c < dk; ++c) s[c] += u * kh[c];\n    }\n    /* output"),
    ("transposed_state_index", "double *s = S + (size_t)i * dk;\n        double r = 0.0;\n        for (int c = 0; c < dk; ++c) r += s[c] * kh[c];\n        double u = beta * (v[i] - r);",
     "double *s = S + (size_t)i * dk;\n        double r = 0.0;\n        for (int c = 0; c < dk; ++c) r += S[(size_t)(c % dv) * dk + (i % dk)] * kh[c];\n        double u = beta * (v[i] - r);"),
]


def _build(src_text, out_dir, name):
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", c, "-o", so, "-lm"],
                   check=True)
    lib = ctypes.CDLL(so)
    D = ctypes.POINTER(ctypes.c_double)
    lib.kda_oracle_recurrence.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int64, D, D, D, D, D,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
        ctypes.c_double, D, D]
    return lib


def _rec(lib, q, k, v, g, b, S0, eps, scale):
    n, dk = k.shape
    dv = v.shape[1]
    arrs = [np.ascontiguousarray(x, np.float64) for x in (q, k, v, g, b)]
    S = np.ascontiguousarray(S0, np.float64).copy()
    o = np.zeros((n, dv))
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))  # noqa: E731
    lib.kda_oracle_recurrence(dk, dv, n, *[P(a) for a in arrs], dk, dv, 1,
                              eps, scale, P(S), P(o))
    return o, S


def pins_pass(lib) -> bool:
    """The golden worked examples and the matrix-form pin, via one library."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        toks = case["tokens"]
        arr = lambda key: np.array([t[key] for t in toks], float)  # noqa: E731
        o, S = _rec(lib, arr("q"), arr("k"), arr("v"), arr("g"), arr("b"),
                    np.array(case["S0"], float), case["eps"], 1 / math.sqrt(2))
        if not (np.allclose(o * math.sqrt(2), case["expected_o_times_sqrt2"], atol=1e-12)
                and np.allclose(S, case["expected_S"], atol=1e-12)):
            return False
    rng = np.random.default_rng(1)
    n, dk, dv, eps = 20, 12, 8, 1e-6
    q, k = rng.standard_normal((n, dk)), rng.standard_normal((n, dk))
    v = rng.standard_normal((n, dv))
    g = -np.log1p(np.exp(-(rng.standard_normal((n, dk)) + 2)))
    b = rng.standard_normal(n)
    S0 = rng.standard_normal((dv, dk))
    o, Sf = _rec(lib, q, k, v, g, b, S0, eps, dk ** -0.5)
    S = S0.copy()
    for t in range(n):
        kh = k[t] / np.sqrt(k[t] @ k[t] + eps)
        qh = q[t] / np.sqrt(q[t] @ q[t] + eps)
        beta = 1 / (1 + np.exp(-b[t]))
        S = S @ np.diag(np.exp(g[t])) @ (np.eye(dk) - beta * np.outer(kh, kh)) \
            + beta * np.outer(v[t], kh)
        if not np.allclose(o[t], dk ** -0.5 * S @ qh, rtol=1e-10, atol=1e-12):
            return False
    return bool(np.allclose(Sf, S, rtol=1e-10, atol=1e-12))


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    return str(tmp_path_factory.mktemp("oracle_mutants"))


def test_unmutated_copy_passes(workdir):
    with open(SRC) as f:
        assert pins_pass(_build(f.read(), workdir, "original"))


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(workdir, name, old, new):
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    assert not pins_pass(_build(text.replace(old, new), workdir, name))


def test_oracle_module_uses_same_source():
    assert os.path.samefile(oracle._SRC, SRC)
