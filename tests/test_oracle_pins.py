"""CPU tests: the fp64 oracle against properties the pages and the mathematics fix, and a
mutation test showing that each plausible slip in the oracle breaks at least one pin."""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(oracle_lib, pin):
    ok, msg = pin(oracle_lib)
    assert ok, msg


# Each mutant: (name, exact text in mlstm_oracle.c, replacement).  Every one is a slip a
# reader could make when writing the cell from the page: a dropped term, a wrong sign, a
# wrong index, a transposed operand, a wrong constant.
MUTANTS = [
    ("stabiliser drops m_{t-1}", "fmax(logf + m, ig[t])", "fmax(logf, ig[t])"),
    ("forget factor drops m_{t-1}", "fgate = exp(logf + m - m_new);", "fgate = exp(logf - m_new);"),
    ("input factor uses old m", "igate = exp(ig[t] - m_new);", "igate = exp(ig[t] - m);"),
    ("log-sigmoid sign", "if (x >= 0.0) return -log1p(exp(-x));", "if (x >= 0.0) return -log1p(exp(x));"),
    ("forget gate exp instead of sigmoid", "return J->exp_forget ? exp(x) : sigmoid(x);", "return exp(x);"),
    ("log forget ignores the variant", "return J->exp_forget ? x : log_sigmoid(x);", "return log_sigmoid(x);"),
    ("log forget always raw", "return J->exp_forget ? x : log_sigmoid(x);", "return x;"),
    ("exp forget gate as sigmoid", "return J->exp_forget ? exp(x) : sigmoid(x);", "return sigmoid(x);"),
    ("key scale 1/d", "1.0 / sqrt((double)DQK); /* k_t", "1.0 / ((double)DQK); /* k_t"),
    ("transposed outer product", "igate * vt[a] * khat[c]", "igate * vt[c % DV] * khat[a % DQK]"),
    ("normaliser with unscaled key", "n[c] = fgate * n[c] + igate * khat[c];", "n[c] = fgate * n[c] + igate * kt[c];"),
    ("normaliser forgets without f", "n[c] = fgate * n[c] + igate * khat[c];", "n[c] = n[c] + igate * khat[c];"),
    ("no absolute value in denominator", "fmax(fabs(nq), floor_)", "fmax(nq, floor_)"),
    ("floor exp(+m)", "(J->kind == 0) ? exp(-m) : 1.0", "(J->kind == 0) ? exp(m) : 1.0"),
    ("retrieval with k instead of q", "acc += row[c] * qt[c];", "acc += row[c] * kt[c];"),
    ("dual-form decay off by one", "for (int tau = j + 1; tau <= t; ++tau)", "for (int tau = j; tau <= t; ++tau)"),
    ("dual-form missing i_j", "double Stj = exp(ig[j]); /* i_j */", "double Stj = 1.0;"),
    ("abs normaliser drops |k|", "igate * fabs(khat[c]);", "igate * khat[c];"),
    ("abs denominator drops |q|", "da += nabs[c] * fabs(qt[c]);", "da += nabs[c] * qt[c];"),
    ("snapshot after the update", "if (J->snap_every > 0 && t % J->snap_every == 0) {",
     "if (J->snap_every > 0 && t % J->snap_every == 0 && t > 0) {"),
]


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(mutant_dir, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    path_c = os.path.join(mutant_dir, f"m{abs(hash(name))}.c")
    path_so = path_c[:-2] + ".so"
    with open(path_c, "w") as f:
        f.write(src.replace(old, new))
    try:
        oracle.build(path_c, path_so)
    except RuntimeError as e:
        pytest.fail(f"mutant did not compile: {e}")
    lib = oracle.load(path_so)
    results = oracle_pins.run_all(lib)
    failed = [r for r in results if not r[1]]
    assert failed, f"mutant '{name}' passed every pin: {results}"


def test_oracle_rejects_bad_arguments(oracle_lib):
    import numpy as np
    q = np.zeros((1, 1, 6, 4))
    with pytest.raises(ValueError):
        oracle.recurrent(q, q, q, np.zeros((1, 1, 6)), np.zeros((1, 1, 6)), snap_every=4)
    with pytest.raises(ValueError):
        oracle.recurrent(q, q, q, np.zeros((1, 1, 5)), np.zeros((1, 1, 6)))


def test_oracle_builds_with_gcc():
    assert shutil.which("gcc"), "gcc is needed to build the oracle"
    out = subprocess.run(["gcc", "--version"], capture_output=True, text=True)
    assert out.returncode == 0
