"""Writes oracle_tiny.json (a tiny GDN forward) and oracle_bwd_tiny.json (a tiny
KDA varlen backward), both computed by the oracle alone.

Run ``python -m tests.golden.make_golden`` from the repository root.  The inputs
come from the seeded workload generator; the expected values come only from
``oracle/``.  The file guards against silent changes to the oracle and gives the
GPU tests a fixed small case.
"""
import json
import os

import torch


def inputs():
    from workloads import random_case
    _, x = random_case(B=1, T=70, H=1, HV=2, K=8, V=4, dtype=torch.float32, seed=11)
    return x


def compute():
    import oracle
    x = inputs()
    r = oracle.gdr_fwd_ref(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], use_qk_l2norm=True)
    return {"o": r["o"].tolist(), "ht": r["ht"].tolist()}


def bwd_inputs():
    from workloads import random_case
    _, x = random_case(B=1, T=70, H=1, HV=2, K=8, V=4, dtype=torch.float32, lengths=(30, 40),
                       gate_per_k=True, seed=12, grads=True)
    return x


def compute_bwd():
    import oracle
    x = bwd_inputs()
    r = oracle.gdr_bwd_ref(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], dht=x["dht"], h0=x["h0"],
                           cu_seqlens=x["cu_seqlens"], use_qk_l2norm=True)
    return {key: r[key].tolist() for key in ("dq", "dk", "dv", "dg", "dbeta", "dh0")}


if __name__ == "__main__":
    here = os.path.dirname(os.path.abspath(__file__))
    out = {"_about": "oracle output for workloads.random_case(B=1,T=70,H=1,HV=2,K=8,V=4,fp32,seed=11), "
                     "use_qk_l2norm=True; written by tests/golden/make_golden.py", **compute()}
    with open(os.path.join(here, "oracle_tiny.json"), "w") as f:
        json.dump(out, f)
    out = {"_about": "oracle reverse recurrence for workloads.random_case(B=1,T=70,H=1,HV=2,K=8,V=4,fp32,"
                     "lengths=(30,40),gate_per_k=True,seed=12,grads=True), use_qk_l2norm=True; written by "
                     "tests/golden/make_golden.py", **compute_bwd()}
    with open(os.path.join(here, "oracle_bwd_tiny.json"), "w") as f:
        json.dump(out, f)
