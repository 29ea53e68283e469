"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Forward mutants go through the forward pins; backward mutants (slips in the
reverse recurrence) go through the backward pins.

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
from tests import oracle_bwd_checks as ob
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


BWD_MUTANTS = {
    "dk_misses_error_path": ("dkn[p * K + d] -= acc;", "dkn[p * K + d] -= 0.0 * acc;"),
    "dstate_not_decayed": ("for (int64_t i = 0; i < KV; ++i) dS[i] *= a;", ""),
    "dq_reads_pre_write_state": ("double acc = kt[d] * udo;", "double acc = 0.0;"),
    "dbeta_uses_v": ("db += du[j] * e[j];", "db += du[j] * v[(t * HV + hv) * V + j];"),
    "norm_bwd_no_projection": ("dx[i] = r * (dy[i] - x[i] * r * ydy);", "dx[i] = r * dy[i];"),
    "dg_before_error_term": ("acc += Sd[d * V + j] * dS[d * V + j];",
                             "acc += Sd[d * V + j] * (dS[d * V + j] + kt[d] * du[j]);"),
    "group_grad_overwritten": ("dqn[p * K + d] += acc;", "dqn[p * K + d] = acc;"),
    "dv_missing_beta": ("du[j] *= b;\n            dvt[j] = du[j];", "dvt[j] = du[j];\n            du[j] *= b;"),
    "dh0_before_last_decay": ("if (dh0) memcpy(dh0 + unit * KV, dS", "if (dh0) memcpy(dh0 + unit * KV, Sprev"),
}


def _mutant_lib(src, old, new, name, tmp_path):
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib_path = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(lib_path), str(mutated), "-lm"],
                   check=True)
    return oracle.load_oracle_lib(str(lib_path))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    lib = _mutant_lib(open(SRC).read(), old, new, name, tmp_path)
    fwd = functools.partial(oracle.gdr_fwd_ref, lib=lib)
    caught = []
    for check in oc.ALL_CHECKS:
        try:
            check(fwd, np.random.default_rng(1234))
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake {name}"


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_bwd_mutant_is_caught(name, tmp_path):
    """The forward stays intact (finite differences use the real forward)."""
    old, new = BWD_MUTANTS[name]
    lib = _mutant_lib(open(SRC).read(), old, new, name, tmp_path)
    bwd = functools.partial(oracle.gdr_bwd_ref, lib=lib)
    caught = []
    for check in ob.ALL_BWD_CHECKS:
        try:
            check(bwd, oracle.gdr_fwd_ref, np.random.default_rng(4321))
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
