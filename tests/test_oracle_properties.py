"""Property checks of the oracle over random tiny shapes (CPU only).

Two facts, each checked on shapes drawn at random rather than on a fixed list:

* the forward equals the recurrence written as explicit K x K matrix products,
  one token at a time (``brute_force``), for every combination of gate kind,
  in-kernel L2 norm, initial state, grouped value heads, chunk size and
  variable-length layout (zero-length sequences included), on o, ht, the
  per-token write vectors and the chunk-start states;
* the reverse recurrence gives the directional derivative of
  L = sum(o * do) + sum(ht * dht) along a random direction in every input,
  measured by central differences of ``brute_force`` (so it does not lean on
  the oracle's own forward), with and without beta given as logits.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
from tests.oracle_checks import brute_force, close, rand_case  # noqa: E402


@st.composite
def cases(draw):
    H = draw(st.integers(1, 2))
    HV = H * draw(st.integers(1, 2))
    K, V = draw(st.integers(1, 6)), draw(st.integers(1, 6))
    per_k, l2, h0 = draw(st.booleans()), draw(st.booleans()), draw(st.booleans())
    if draw(st.booleans()):  # variable-length layout
        lengths = draw(st.lists(st.integers(0, 6), min_size=1, max_size=4))
        B, T = 1, max(1, sum(lengths))
        if sum(lengths) == 0:
            lengths[-1] = 1
    else:
        lengths, B, T = None, draw(st.integers(1, 2)), draw(st.integers(1, 10))
    C = draw(st.integers(1, 5))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return dict(B=B, T=T, H=H, HV=HV, K=K, V=V, per_k=per_k, l2=l2, h0=h0, lengths=lengths, C=C, seed=seed)


def _inputs(c):
    rng = np.random.default_rng(c["seed"])
    return rand_case(rng, c["B"], c["T"], c["H"], c["HV"], c["K"], c["V"], per_k=c["per_k"],
                     lengths=c["lengths"], h0=c["h0"])


@settings(max_examples=60, deadline=None)
@given(cases())
def test_forward_equals_explicit_matrix_recurrence(c):
    x = _inputs(c)
    ref = brute_force(**x, use_qk_l2norm=c["l2"], chunk_size=c["C"])
    got = oracle.gdr_fwd_ref(**x, use_qk_l2norm=c["l2"], chunk_size=c["C"], want_v_new=True)
    for key in ("o", "ht", "v_new", "h_chunks"):
        close(got[key], ref[key], what=f"{key} {c}")


def _loss(x, do, dht, l2, beta_logits):
    y = dict(x)
    if beta_logits:
        y["beta"] = 1.0 / (1.0 + np.exp(-x["beta"]))
    out = brute_force(**y, use_qk_l2norm=l2)
    return float(np.sum(out["o"] * do) + np.sum(out["ht"] * dht))


@settings(max_examples=30, deadline=None)
@given(cases(), st.booleans())
def test_backward_is_the_directional_derivative(c, beta_logits):
    x = _inputs(c)
    rng = np.random.default_rng(c["seed"] + 1)
    if beta_logits:  # beta as logits: any real value
        x["beta"] = rng.standard_normal(x["beta"].shape)
    N = len(c["lengths"]) if c["lengths"] else c["B"]
    do = rng.standard_normal(x["v"].shape)
    dht = rng.standard_normal((N, c["HV"], c["K"], c["V"]))
    if x["h0"] is None:
        x["h0"] = np.zeros((N, c["HV"], c["K"], c["V"]))
    names = ("q", "k", "v", "g", "beta", "h0")
    d = {n: rng.standard_normal(x[n].shape) for n in names}
    grads = oracle.gdr_bwd_ref(x["q"], x["k"], x["v"], x["g"], x["beta"], do, dht=dht, h0=x["h0"],
                               cu_seqlens=x["cu_seqlens"], use_qk_l2norm=c["l2"], beta_logits=beta_logits)
    key = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "h0": "dh0"}
    want = sum(float(np.sum(grads[key[n]] * d[n])) for n in names)
    eps = 1e-6
    xp = {**x, **{n: x[n] + eps * d[n] for n in names}}
    xm = {**x, **{n: x[n] - eps * d[n] for n in names}}
    fd = (_loss(xp, do, dht, c["l2"], beta_logits) - _loss(xm, do, dht, c["l2"], beta_logits)) / (2 * eps)
    scale = max(1.0, abs(want), sum(float(np.abs(grads[key[n]] * d[n]).sum()) for n in names))
    assert abs(fd - want) <= 1e-6 * scale, f"finite difference {fd!r} vs reverse recurrence {want!r} ({c})"
