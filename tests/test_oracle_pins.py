"""The oracle against facts outside itself (CPU only).

Pages cited: the KCP handbook = "flash-linear-attention KCP 精度失效根因排查手册".
"""
import json
import os

import numpy as np
import pytest

import oracle
from tests import oracle_bwd_checks as ob
from tests import oracle_checks as oc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle.gdr_fwd_ref, np.random.default_rng(1234))


@pytest.mark.parametrize("check", ob.ALL_BWD_CHECKS, ids=lambda f: f.__name__)
def test_oracle_bwd_pin(check):
    check(oracle.gdr_bwd_ref, oracle.gdr_fwd_ref, np.random.default_rng(4321))


def test_chunk_form_per_key_gate():
    oc.check_chunk_form(oracle.gdr_fwd_ref, np.random.default_rng(7), per_k=True, C=8)


def test_chunk_index_matches_handbook_example():
    facts = json.load(open(os.path.join(GOLDEN, "pages_facts.json")))["kcp_chunk_boundaries"]
    cu = np.concatenate([[0], np.cumsum(facts["lengths"])])
    C = facts["chunk_size"]
    idx, off = oracle.chunk_index_ref(cu, C)
    starts = [int(cu[n] + j * C) for n, j in idx]
    second = [s for (n, _), s in zip(idx, starts) if n == 1]
    want = facts["second_sequence_global_chunk_starts_prefix"]
    assert second[:len(want)] == want
    assert off.tolist() == [0, 7, 17]
    # the first sequence's last chunk is cut short: 400 - 6*64 = 16 tokens
    assert int(cu[1]) - starts[6] == 16


def test_chunk_index_edge_cases():
    # lengths 0, 1, 65, 0, 64 -> 0, 1, 2, 0, 1 chunks
    idx, off = oracle.chunk_index_ref([0, 0, 1, 66, 66, 130], 64)
    assert off.tolist() == [0, 0, 1, 3, 3, 4]
    assert idx.tolist() == [[1, 0], [2, 0], [2, 1], [4, 0]]
    idx, off = oracle.chunk_index_ref([0], 32)
    assert idx.shape == (0, 2) and off.tolist() == [0]


def test_sampled_units_equal_whole_run():
    import torch
    rng = np.random.default_rng(3)
    x = oc.rand_case(rng, 1, 20, 2, 4, 3, 2, lengths=[7, 13])
    whole = oracle.gdr_fwd_ref(**x, use_qk_l2norm=True)
    tx = {k: (None if v is None else torch.from_numpy(v)) for k, v in x.items()}
    part = oracle.gdr_fwd_ref_units(tx["q"], tx["k"], tx["v"], tx["g"], tx["beta"], [(1, 3), (0, 2)],
                                    h0=tx["h0"], cu_seqlens=tx["cu_seqlens"], use_qk_l2norm=True)
    cu = x["cu_seqlens"]
    for (n, hv), (o, ht) in part.items():
        np.testing.assert_allclose(o, whole["o"][0, cu[n]:cu[n + 1], hv], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(ht, whole["ht"][n, hv], rtol=1e-13, atol=1e-14)


def test_golden_regression():
    """The oracle still produces the values its committed generator stored."""
    from tests.golden.make_golden import compute
    stored = json.load(open(os.path.join(GOLDEN, "oracle_tiny.json")))
    now = compute()
    for key in ("o", "ht"):
        np.testing.assert_allclose(np.array(now[key]), np.array(stored[key]), rtol=1e-12, atol=1e-13)


def test_golden_bwd_regression():
    """The reverse recurrence still produces the values its committed generator stored."""
    from tests.golden.make_golden import compute_bwd
    stored = json.load(open(os.path.join(GOLDEN, "oracle_bwd_tiny.json")))
    now = compute_bwd()
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        np.testing.assert_allclose(np.array(now[key]), np.array(stored[key]), rtol=1e-12, atol=1e-13)
