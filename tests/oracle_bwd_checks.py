"""Checks that pin the oracle's reverse recurrence to facts outside itself.

Each ``check_*`` takes the oracle backward and forward callables (signatures of
``oracle.gdr_bwd_ref`` and ``oracle.gdr_fwd_ref``) and raises AssertionError on
a mismatch, so planted mistakes in a copy of the oracle can be run through them
(``test_oracle_mutants.py``).  The facts used:

* central finite differences of the (separately pinned) forward: the gradient
  of L = sum(o * do) + sum(ht * dht) with respect to every input element;
* a closed form: with beta = 0 and g = 0 the state never moves (S_t = h0), so
  dq_t = h0 do_t, dv = dk = 0, dh0 = dht + sum_t q_t do_t^T,
  dbeta_t = (dS_t^T k_t) . (v_t - h0^T k_t) and dg_t = <h0, dS_t>, with
  dS_t = dht + sum_{s >= t} q_s do_s^T;
* splitting: varlen gradients equal those of the sequences run alone; a
  channel-uniform KDA gate has gradient summing over channels to the GDN one.
"""
from __future__ import annotations

import numpy as np

from tests.oracle_checks import close, rand_case

FD_TOL = 1e-6


def _loss(fwd, case, do, dht, l2, **kw):
    out = fwd(case["q"], case["k"], case["v"], case["g"], case["beta"], h0=case["h0"],
              cu_seqlens=case["cu_seqlens"], use_qk_l2norm=l2, **kw)
    return float(np.sum(out["o"] * do) + np.sum(out["ht"] * dht))


def finite_difference(fwd, case, do, dht, l2, name, step=1e-6, **kw):
    x = case[name]
    grad = np.zeros_like(x)
    flat = x.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        flat[i] = old + step
        lp = _loss(fwd, case, do, dht, l2, **kw)
        flat[i] = old - step
        lm = _loss(fwd, case, do, dht, l2, **kw)
        flat[i] = old
        grad.reshape(-1)[i] = (lp - lm) / (2 * step)
    return grad


def _fd_case(bwd, fwd, rng, per_k, lengths, l2, G):
    H = 1
    if lengths:
        case = rand_case(rng, 1, sum(lengths), H, H * G, 3, 4, per_k=per_k, lengths=lengths)
        N = len(lengths)
    else:
        case = rand_case(rng, 2, 7, H, H * G, 3, 4, per_k=per_k)
        N = 2
    if not l2:  # keep the state bounded without the norm
        for key in ("q", "k"):
            case[key] = case[key] / np.linalg.norm(case[key], axis=-1, keepdims=True)
    B, T = case["q"].shape[:2]
    do = rng.standard_normal((B, T, H * G, 4))
    dht = rng.standard_normal((N, H * G, 3, 4))
    got = bwd(case["q"], case["k"], case["v"], case["g"], case["beta"], do, dht=dht, h0=case["h0"],
              cu_seqlens=case["cu_seqlens"], use_qk_l2norm=l2)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"), ("h0", "dh0")):
        ref = finite_difference(fwd, case, do, dht, l2, name)
        close(got[key], ref, FD_TOL, f"{key} vs finite differences (per_k={per_k}, l2={l2})")


def check_bwd_fd_gdn(bwd, fwd, rng):
    _fd_case(bwd, fwd, rng, per_k=False, lengths=None, l2=True, G=2)


def check_bwd_fd_kda_varlen(bwd, fwd, rng):
    _fd_case(bwd, fwd, rng, per_k=True, lengths=[5, 3], l2=True, G=2)


def check_bwd_fd_no_norm(bwd, fwd, rng):
    _fd_case(bwd, fwd, rng, per_k=False, lengths=[4, 6], l2=False, G=1)


def check_bwd_closed_form_frozen_state(bwd, fwd, rng):
    B, T, H, K, V = 1, 6, 1, 4, 3
    case = rand_case(rng, B, T, H, H, K, V)
    case["q"] = case["q"] / np.linalg.norm(case["q"], axis=-1, keepdims=True)
    case["k"] = case["k"] / np.linalg.norm(case["k"], axis=-1, keepdims=True)
    case["beta"][:] = 0.0
    case["g"][:] = 0.0
    do = rng.standard_normal((B, T, H, V))
    dht = rng.standard_normal((B, H, K, V))
    got = bwd(case["q"], case["k"], case["v"], case["g"], case["beta"], do, dht=dht, h0=case["h0"])
    h0 = case["h0"][0, 0]
    q, k, v = case["q"][0, :, 0], case["k"][0, :, 0], case["v"][0, :, 0]
    dS = dht[0, 0].copy()
    dq, dbeta, dg = np.zeros((T, K)), np.zeros(T), np.zeros(T)
    for t in range(T - 1, -1, -1):
        dS = dS + np.outer(q[t], do[0, t, 0])
        dq[t] = h0 @ do[0, t, 0]
        dbeta[t] = (dS.T @ k[t]) @ (v[t] - h0.T @ k[t])
        dg[t] = np.sum(h0 * dS)
    close(got["dq"][0, :, 0], dq, 1e-12, "dq (frozen state)")
    close(got["dbeta"][0, :, 0], dbeta, 1e-12, "dbeta (frozen state)")
    close(got["dg"][0, :, 0], dg, 1e-12, "dg (frozen state)")
    close(got["dh0"][0, 0], dS, 1e-12, "dh0 (frozen state)")
    assert np.abs(got["dv"]).max() == 0.0 and np.abs(got["dk"]).max() == 0.0, "dv, dk must vanish at beta = 0"


def check_bwd_varlen_equals_separate(bwd, fwd, rng):
    lengths = [5, 9, 1]
    case = rand_case(rng, 1, sum(lengths), 2, 4, 5, 3, per_k=True, lengths=lengths)
    T = sum(lengths)
    do = rng.standard_normal((1, T, 4, 3))
    dht = rng.standard_normal((3, 4, 5, 3))
    got = bwd(case["q"], case["k"], case["v"], case["g"], case["beta"], do, dht=dht, h0=case["h0"],
              cu_seqlens=case["cu_seqlens"], use_qk_l2norm=True)
    cu = case["cu_seqlens"]
    for n in range(3):
        s = slice(cu[n], cu[n + 1])
        one = bwd(case["q"][:, s], case["k"][:, s], case["v"][:, s], case["g"][:, s], case["beta"][:, s], do[:, s],
                  dht=dht[n:n + 1], h0=case["h0"][n:n + 1], use_qk_l2norm=True)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            close(got[key][:, s], one[key], 1e-13, f"{key} of sequence {n}")
        close(got["dh0"][n:n + 1], one["dh0"], 1e-13, f"dh0 of sequence {n}")


def check_bwd_kda_uniform_equals_gdn(bwd, fwd, rng):
    case = rand_case(rng, 1, 10, 1, 2, 4, 3)
    do = rng.standard_normal((1, 10, 2, 3))
    dht = rng.standard_normal((1, 2, 4, 3))
    gdn = bwd(case["q"], case["k"], case["v"], case["g"], case["beta"], do, dht=dht, h0=case["h0"],
              use_qk_l2norm=True)
    g4 = np.repeat(case["g"][..., None], 4, axis=-1)
    kda = bwd(case["q"], case["k"], case["v"], g4, case["beta"], do, dht=dht, h0=case["h0"], use_qk_l2norm=True)
    for key in ("dq", "dk", "dv", "dbeta", "dh0"):
        close(kda[key], gdn[key], 1e-12, f"{key} (uniform KDA gate vs GDN)")
    close(kda["dg"].sum(-1), gdn["dg"], 1e-12, "dg summed over channels")


def check_bwd_fd_beta_logits(bwd, fwd, rng):
    """beta given as logits: dbeta is the gradient with respect to the logits."""
    case = rand_case(rng, 1, 9, 1, 2, 3, 4)
    case["beta"] = rng.standard_normal(case["beta"].shape) * 2.0
    do = rng.standard_normal((1, 9, 2, 4))
    dht = rng.standard_normal((1, 2, 3, 4))
    got = bwd(case["q"], case["k"], case["v"], case["g"], case["beta"], do, dht=dht, h0=case["h0"],
              use_qk_l2norm=True, beta_logits=True)
    for name, key in (("beta", "dbeta"), ("k", "dk")):
        ref = finite_difference(fwd, case, do, dht, True, name, beta_logits=True)
        close(got[key], ref, FD_TOL, f"{key} vs finite differences (beta logits)")


ALL_BWD_CHECKS = [check_bwd_fd_beta_logits, check_bwd_fd_gdn, check_bwd_fd_kda_varlen, check_bwd_fd_no_norm,
                  check_bwd_closed_form_frozen_state, check_bwd_varlen_equals_separate,
                  check_bwd_kda_uniform_equals_gdn]
