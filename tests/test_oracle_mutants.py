"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/gdr_oracle.c (on the CPU,
in a temporary directory), builds it, and runs the pin suite against that
build. The suite has to fail for every mutant.
"""
import os
import subprocess
import sys

import pytest

from oracle.build import SRC, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "no decay": ("S[i * dv + j] *= alpha;", "S[i * dv + j] *= 1.0;"),
    "decay squared": ("const double alpha = exp(log_alpha[per_channel ? i : 0]);",
                      "const double alpha = exp(2.0 * log_alpha[per_channel ? i : 0]);"),
    "per-channel rate of another channel": ("log_alpha[per_channel ? i : 0]",
                                            "log_alpha[per_channel ? (i + 1) % dk : 0]"),
    "per-channel rates ignored": ("log_alpha[per_channel ? i : 0]", "log_alpha[0]"),
    "per-channel stride of one": ("th * (job->per_channel ? dk : 1)", "th"),
    "sign of the correction": ("beta * k[i] * (v[j] - vhat[j])", "beta * k[i] * (v[j] + vhat[j])"),
    "write strength dropped": ("beta * k[i] * (v[j] - vhat[j])", "k[i] * (v[j] - vhat[j])"),
    "read with the key instead of the query": ("o[j] += S[i * dv + j] * q[i];",
                                               "o[j] += S[i * dv + j] * k[i];"),
    "prediction read with the query": ("vhat[j] += S[i * dv + j] * k[i];",
                                       "vhat[j] += S[i * dv + j] * q[i];"),
    "initial state ignored": ("if (job->S0)", "if (0)"),
    "additive write without beta": ("S[i * dv + j] += beta * k[i] * v[j];",
                                    "S[i * dv + j] += k[i] * v[j];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = build(str(mutant_src), str(tmp_path / "libmutant.so"))
    env = dict(os.environ, GDR_ORACLE_LIB=lib)
    proc = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle_pins.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode != 0, f"pins did not catch mutant {name!r}:\n{proc.stdout[-2000:]}"
