"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant is a plausible slip (a sign, a dropped term, a transposed operand,
a wrong index) applied textually to a temporary copy of ``oracle/gdr_oracle.c``,
compiled with gcc and run through the pin checks on the CPU.  The real oracle
is never modified.
"""
import functools
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests import oracle_checks as oc

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdr_oracle.c")

MUTANTS = {
    "error_sign": ("e[j] -= S[d * V + j] * kd;", "e[j] += S[d * V + j] * kd;"),
    "beta_dropped": ("for (int64_t j = 0; j < V; ++j) e[j] *= b;", ""),
    "output_reads_k": ("ot[j] += S[d * V + j] * qd;", "ot[j] += S[d * V + j] * kt[d];"),
    "gate_sign": ("const double a = exp(g[t * HV + hv]);", "const double a = exp(-g[t * HV + hv]);"),
    "gva_head_map": ("const int64_t n = unit / HV, hv = unit % HV, hq = hv / G;",
                     "const int64_t n = unit / HV, hv = unit % HV, hq = hv % H;"),
    "chunk_state_off_by_one": ("if (h_chunks && p % chunk_size == 0)",
                               "if (h_chunks && (p + 1) % chunk_size == 0 && p + 1 < t1 - t0)"),
    "l2norm_no_sqrt": ("double inv = 1.0 / sqrt(ss + ORACLE_L2_EPS);", "double inv = 1.0 / (ss + ORACLE_L2_EPS);"),
    "kda_gate_transposed": ("for (int64_t j = 0; j < V; ++j) S[d * V + j] *= a;",
                            "for (int64_t j = 0; j < V; ++j) S[d * V + j] *= exp(gt[j % K]);"),
    "write_uses_unnormalized_k": ("S[d * V + j] += kd * e[j];",
                                  "S[d * V + j] += k[(t * H + hq) * K + d] * e[j];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib_path = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(lib_path), str(mutated), "-lm"],
                   check=True)
    fwd = functools.partial(oracle.gdr_fwd_ref, lib=oracle.load_oracle_lib(str(lib_path)))
    caught = []
    for check in oc.ALL_CHECKS:
        try:
            check(fwd, np.random.default_rng(1234))
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
