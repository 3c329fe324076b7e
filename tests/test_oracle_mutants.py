"""The oracle's pins catch plausible mistakes.  Each case plants one mistake in
a copy of the C oracle (a dropped term or carry, a wrong sign, a transposed
index, an off-by-one exponent, a wrong rounding step), builds the copy in a
temporary directory, and checks that comparing it with the pure-Python
definitions (exact integers and fractions) fails; the unmutated copy passes
the same comparisons.  CPU only."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle

MUTANTS = {
    "int: carry without the product's sign": (
        "hi += (p < 0 ? -1 : 0) + (nlo < lo ? 1 : 0);", "hi += (nlo < lo ? 1 : 0);"),
    "int: B read transposed": (
        "i128 p = (i128)A[(size_t)i * K + k] * (i128)B[(size_t)k * N + j];",
        "i128 p = (i128)A[(size_t)i * K + k] * (i128)B[(size_t)j * K + k];"),
    "int: last term dropped": (
        "for (int k = 0; k < K; k++) {\n        i128 p", "for (int k = 0; k < K - 1; k++) {\n        i128 p"),
    "limbs: product sign from A alone": ("if (sa ^ sb) negate(out, la + lb);", "if (sa) negate(out, la + lb);"),
    "limbs: no sign extension in the sum": (
        "uint64_t ext = (p[np - 1] >> 63) ? ~(uint64_t)0 : 0;", "uint64_t ext = 0;"),
    "enclosure: subnormal exponent off by one": ("    *e = -1074;", "    *e = -1075;"),
    "enclosure: product sign from A alone": ("grid_add((sa ^ sb) ? &neg : &pos,", "grid_add((sa) ? &neg : &pos,"),
    "enclosure: lower end steps past an exact value": (
        "  *lo = c;\n  *hi = cmp_exact_double(V, c) == 0 ? c : nextafter(c, INFINITY);",
        "  *lo = cmp_exact_double(V, c) == 0 ? nextafter(c, -INFINITY) : c;\n"
        "  *hi = cmp_exact_double(V, c) == 0 ? c : nextafter(c, INFINITY);"),
    "interval: radius product Ar Br dropped": (
        "      exact_entry(Ar, Br, i, j, N, K, &t);\n      exact_add(&R, &t, 1);\n", ""),
    "interval: |Am| taken as Am": ("aAm[t] = fabs(Am[t]);", "aAm[t] = Am[t];"),
    "interval: radius added on the low side": ("exact_add(&L, &R, -1);", "exact_add(&L, &R, 1);"),
}


def build_copy(tmp_path, name, find=None, repl=None):
    src = open(oracle._SRC).read()
    if find is not None:
        assert src.count(find) == 1, name
        src = src.replace(find, repl)
    c = tmp_path / f"{abs(hash(name))}.c"
    so = tmp_path / f"{abs(hash(name))}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", str(so), str(c), "-lm"],
                   check=True)
    return oracle._configure(ctypes.CDLL(str(so)))


def comparisons():
    """Each comparison of the C oracle with the Python definitions: name -> passed."""
    rng = np.random.default_rng(5)
    out = {}
    # int64: large magnitudes of both signs (products carry into the high word), K > 1
    A = rng.integers(-(2**62), 2**62, size=(3, 5), dtype=np.int64)
    B = rng.integers(-(2**62), 2**62, size=(5, 4), dtype=np.int64)
    want = oracle.matmul_py(oracle.to_pyint_matrix(A), oracle.to_pyint_matrix(B))
    got = oracle.matmul_i64(A, B, lc=3)
    out["int64"] = [[oracle.limbs_to_int(got[i, j]) for j in range(4)] for i in range(3)] == want
    # two-limb operands of both signs
    L = rng.integers(-(2**63), 2**63 - 1, size=(2, 3, 2), dtype=np.int64, endpoint=True)
    R = rng.integers(-(2**63), 2**63 - 1, size=(3, 2, 2), dtype=np.int64, endpoint=True)
    want = oracle.matmul_py(oracle.to_pyint_matrix(L), oracle.to_pyint_matrix(R))
    got = oracle.matmul_limbs(L, R, 5)
    out["limbs"] = [[oracle.limbs_to_int(got[i, j]) for j in range(2)] for i in range(2)] == want
    # binary64: normal values of both signs, subnormals, and an exactly representable product
    X = np.array([[1.5, -2.25, 5e-324, 3.0], [-0.1, 0.7, 2.0**-1060, -1.0]])
    Y = np.array([[2.0, 0.3], [1.0, -1.1], [3.0, 7.0], [-0.5, 0.25]])
    lo, hi = oracle.enclose_f64(X, Y)
    plo, phi = oracle.enclose_py(X, Y)
    out["enclose"] = np.array_equal(lo, np.array(plo)) and np.array_equal(hi, np.array(phi))
    # a subnormal product beside a normal one: 2^-1022 + 2^-1074 is a double, so the pair closes on it
    # (subnormal products alone scale with the candidates they are compared with)
    X = np.array([[2.0**-1022, 5e-324], [-(2.0**-1022), 3 * 5e-324]])
    Y = np.array([[1.0, 0.5], [1.0, -1.0]])
    lo, hi = oracle.enclose_f64(X, Y)
    plo, phi = oracle.enclose_py(X, Y)
    out["enclose_subnormal"] = np.array_equal(lo, np.array(plo)) and np.array_equal(hi, np.array(phi))
    # intervals of both signs
    Am = np.array([[1.0, -2.0, 0.5], [-3.0, 0.25, 1.5]])
    Ar = np.array([[0.125, 0.5, 0.0], [0.25, 0.0625, 0.5]])
    Bm = np.array([[2.0, -1.0], [-0.5, 3.0], [1.25, -2.0]])
    Br = np.array([[0.5, 0.25], [0.125, 0.0], [0.75, 0.5]])
    ilo, ihi = oracle.interval(Am, Ar, Bm, Br)
    plo, phi = oracle.interval_py(Am, Ar, Bm, Br)
    out["interval"] = np.array_equal(ilo, np.array(plo)) and np.array_equal(ihi, np.array(phi))
    return out


@pytest.fixture
def swap_lib(monkeypatch):
    def use(lib):
        monkeypatch.setattr(oracle, "_lib", lib)
    return use


def test_control_copy_passes(tmp_path, swap_lib):
    swap_lib(build_copy(tmp_path, "control"))
    assert all(comparisons().values())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, swap_lib, name):
    find, repl = MUTANTS[name]
    swap_lib(build_copy(tmp_path, name, find, repl))
    try:
        results = comparisons()
    except (OverflowError, RuntimeError, ValueError):
        return  # the mutant broke a check outright
    assert not all(results.values()), f"{name} passed every comparison: {results}"
