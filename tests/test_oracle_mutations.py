"""Plant plausible mistakes in a copy of the oracle and check that the pins fail.

Each mutant is a one-line edit of ``oracle/epilogue.py`` (a dropped term, a
wrong sign or index, a swapped map, the wrong variance divisor, the wrong
rounding order...).  The copy is written to a temporary directory and the pin
tests (``test_oracle_pins.py``) are run against it in a subprocess; every
mutant must make at least one pin fail.  The real oracle is never modified.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "epilogue.py")

# (name, original text, planted text)
MUTANTS = [
    ("sample_variance", "var = np.mean(d * d, axis=1)", "var = np.sum(d * d, axis=1) / max(1, d.shape[1] - 1)"),
    ("eps_dropped", "rstd = 1.0 / np.sqrt(var + eps)", "rstd = 1.0 / np.sqrt(var)"),
    ("eps_not_float32", "eps = float(np.float32(epsilon))", "eps = float(epsilon)"),
    ("mean_not_subtracted", "d = s - mu[:, None]", "d = s - 0.0 * mu[:, None]"),
    ("sln_bias_dropped", "            s = s + bb\n        if simplified:", "            s = s\n        if simplified:"),
    ("skip_row_map", "s = x2[r].astype(np.float64) + sk2[r % skip_rows].astype(np.float64)",
     "s = x2[r].astype(np.float64) + sk2[(r * 7) % skip_rows].astype(np.float64)"),
    ("beta_sign", "y = y + b", "y = y - b"),
    ("gamma_dropped", "        y = n * g\n", "        y = n * 1.0\n"),
    ("residual_exact_then_round", "s = x2[r].astype(np.float32) + sk2[r % skip_rows].astype(np.float32)",
     "s = x2[r].astype(np.float64) + sk2[r % skip_rows].astype(np.float64)"),
    ("residual_order", "            s = s + bb\n        out[pos] = s.astype(T)",
     "            s = x2[r].astype(np.float32) + (sk2[r % skip_rows].astype(np.float32) + bb)\n        out[pos] = s.astype(T)"),
    ("inner_map_cyclic", "        return r // inner_repeat", "        return r % bias_rows"),
    ("outer_map_consecutive", "    return r % bias_rows\n", "    return r // inner_repeat\n"),
    ("softmax_no_max_shift", "e = np.exp(z - m[:, None])", "e = np.exp(z)"),
    ("softmax_bias_dropped", "z = d2[r].astype(np.float64) + b2[br].astype(np.float64)", "z = d2[r].astype(np.float64)"),
    ("softmax_global_sum", "out[pos] = e / np.sum(e, axis=1)[:, None]", "out[pos] = e / np.sum(e)"),
    ("bias_add_bias_reversed", "b = np.broadcast_to(b.reshape((1,) * (x.ndim - 1) + (C,)), x.shape)",
     "b = np.broadcast_to(b[::-1].reshape((1,) * (x.ndim - 1) + (C,)), x.shape)"),
    ("bias_add_skip_dropped", "s2, e2 = _two_sum(s1, s)", "s2, e2 = _two_sum(s1, 0.0 * s)"),
    ("bias_add_uncompensated", "        y = s2 + (e1 + e2)\n", "        y = s2\n"),
    ("bias_add_two_sum_error", "    e = (a - (s - bb)) + (b - bb)\n", "    e = b - bb\n"),
    ("gelu_sign", "sig[pos] = 1.0 / (1.0 + np.exp(-t[pos]))", "sig[pos] = 1.0 / (1.0 + np.exp(t[pos]))"),
    ("gelu_alpha_not_float32", "a = float(np.float32(alpha))", "a = float(alpha)"),
    ("gelu_stable_branch", "sig[~pos] = et / (1.0 + et)", "sig[~pos] = et"),
]


def _run_mutant(tmp_root, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    assert mutated != src
    d = os.path.join(tmp_root, name)
    pkg = os.path.join(d, "oracle")
    os.makedirs(pkg)
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), pkg)
    with open(os.path.join(pkg, "epilogue.py"), "w") as f:
        f.write(mutated)
    env = dict(os.environ, EP_ORACLE_MUTANT_DIR=d, PYTHONDONTWRITEBYTECODE="1")
    p = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, p.returncode, p.stdout[-400:]


def test_every_planted_mistake_is_caught(tmp_path):
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        results = list(ex.map(lambda m: _run_mutant(str(tmp_path), *m), MUTANTS))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, f"mutants not caught by the pins: {survivors}"
    # a failure must be a test failure (rc 1), not a collection/import error
    for n, rc, out in results:
        assert rc == 1, (n, rc, out)


def test_unmutated_copy_passes(tmp_path):
    # control: the same harness with the untouched oracle passes
    d = os.path.join(str(tmp_path), "control")
    os.makedirs(os.path.join(d, "oracle"))
    for f in ("__init__.py", "epilogue.py"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(d, "oracle"))
    env = dict(os.environ, EP_ORACLE_MUTANT_DIR=d, PYTHONDONTWRITEBYTECODE="1")
    p = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stdout[-2000:]
