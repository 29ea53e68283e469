"""Checks that pin the oracle to facts outside itself.

Each ``check_*`` takes an oracle forward callable (same signature as
``oracle.gdr_fwd_ref``) and raises AssertionError on a mismatch, so the same
checks can be run against deliberately broken copies of the oracle (see
``test_oracle_mutants.py``).  The facts used:

* brute force: the recurrence as a product of explicit K x K matrices,
  S_t = (I - beta k k^T) D_t S_{t-1} + beta k v^T, o_t = S_t^T q_t, for T <= 8;
* closed forms: beta = 0, g = 0 gives o_t = h0^T q_t and ht = h0; g -> -inf
  resets the state so o_t = beta_t (k_t . q_t) v_t; beta = 1 with unit k makes
  the write exact, S_t^T k_t = v_t;
* the WY representation of the coverage guide (section 二): with g = 0,
  S^r = P^r S^0 + H^r and P^r = I - sum_i k^i w^i^T;
* splitting: varlen equals the sequences run alone; a call resumed from the
  final state of a prefix equals one call; a channel-uniform KDA gate equals
  the scalar GDN gate;
* the chunk form (UT transform): v_new = u - w h, h' = e^{G_C} h +
  (K * e^{G_C - G})^T v_new, o from the inter + intra terms.

Pages cited: the coverage guide = "FLA 算子内核正确性测试与覆盖矩阵" (fla/ops correctness-coverage guide).
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-11


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def close(a, b, tol=RTOL, what=""):
    r = rel(a, b)
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    assert r <= tol, f"{what}: relative L2 error {r:.3e} > {tol:.1e}"


def rand_case(rng, B, T, H, HV, K, V, per_k=False, lengths=None, h0=True):
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, HV, V))
    gshape = (B, T, HV, K) if per_k else (B, T, HV)
    g = np.log(1.0 / (1.0 + np.exp(-rng.standard_normal(gshape))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, HV))))
    N = len(lengths) if lengths else B
    hz = 0.1 * rng.standard_normal((N, HV, K, V)) if h0 else None
    cu = None if not lengths else np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=hz, cu_seqlens=cu)


def brute_force(q, k, v, g, beta, h0=None, cu_seqlens=None, use_qk_l2norm=False, chunk_size=None):
    """Explicit matrix products of the recurrence, one token at a time."""
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    G = HV // H
    per_k = g.ndim == 4
    if cu_seqlens is None:
        seqs = [(b, 0, T) for b in range(B)]
    else:
        seqs = [(0, int(cu_seqlens[n]), int(cu_seqlens[n + 1])) for n in range(len(cu_seqlens) - 1)]
    o = np.zeros((B, T, HV, V))
    ht = np.zeros((len(seqs), HV, K, V))
    vnew = np.zeros((B, T, HV, V))
    hch = []
    I = np.eye(K)
    for n, (b, s0, s1) in enumerate(seqs):
        for hv in range(HV):
            hq = hv // G
            S = np.zeros((K, V)) if h0 is None else h0[n, hv].copy()
            for t in range(s0, s1):
                if chunk_size and (t - s0) % chunk_size == 0:
                    hch.append((n, (t - s0) // chunk_size, hv, S.copy()))
                qt, kt = q[b, t, hq].copy(), k[b, t, hq].copy()
                if use_qk_l2norm:
                    qt = qt / np.sqrt(qt @ qt + 1e-6)
                    kt = kt / np.sqrt(kt @ kt + 1e-6)
                D = np.diag(np.exp(g[b, t, hv])) if per_k else np.exp(g[b, t, hv]) * I
                bt = beta[b, t, hv]
                Sd = D @ S
                vnew[b, t, hv] = bt * (v[b, t, hv] - Sd.T @ kt)
                S = (I - bt * np.outer(kt, kt)) @ D @ S + bt * np.outer(kt, v[b, t, hv])
                o[b, t, hv] = S.T @ qt
            ht[n, hv] = S
    out = {"o": o, "ht": ht, "v_new": vnew}
    if chunk_size:
        hch.sort(key=lambda x: (x[0], x[1], x[2]))
        NT = len({(a, c) for a, c, _, _ in hch})
        arr = np.zeros((NT, HV, K, V))
        idx = {}
        for n, c, hv, S in hch:
            key = (n, c)
            if key not in idx:
                idx[key] = len(idx)
            arr[idx[key], hv] = S
        out["h_chunks"] = arr
    return out


def check_brute_force(fwd, rng):
    cases = [
        dict(B=1, T=8, H=1, HV=1, K=3, V=2, per_k=False, l2=False),
        dict(B=2, T=5, H=1, HV=2, K=4, V=3, per_k=False, l2=True),
        dict(B=1, T=7, H=2, HV=4, K=3, V=5, per_k=True, l2=True),
        dict(B=2, T=6, H=1, HV=1, K=2, V=2, per_k=True, l2=False),
    ]
    for c in cases:
        x = rand_case(rng, c["B"], c["T"], c["H"], c["HV"], c["K"], c["V"], per_k=c["per_k"])
        ref = brute_force(**x, use_qk_l2norm=c["l2"], chunk_size=3)
        got = fwd(**x, use_qk_l2norm=c["l2"], chunk_size=3, want_v_new=True)
        for key in ("o", "ht", "v_new", "h_chunks"):
            close(got[key], ref[key], what=f"brute force {key} {c}")
    # varlen with a zero-length sequence and GVA
    x = rand_case(rng, 1, 9, 1, 2, 3, 2, lengths=[4, 0, 5])
    ref = brute_force(**x, chunk_size=2)
    got = fwd(**x, chunk_size=2, want_v_new=True)
    for key in ("o", "ht", "v_new", "h_chunks"):
        close(got[key], ref[key], what=f"brute force varlen {key}")


def check_closed_form_identity(fwd, rng):
    """beta = 0 and g = 0: the state never changes, o_t = h0^T q_t."""
    x = rand_case(rng, 2, 11, 2, 4, 5, 3)
    x["beta"][:] = 0.0
    x["g"][:] = 0.0
    got = fwd(**x)
    G = 2
    for b in range(2):
        for hv in range(4):
            exp_o = x["q"][b, :, hv // G] @ x["h0"][b, hv]
            close(got["o"][b, :, hv], exp_o, what="beta=0,g=0 o")
    close(got["ht"], x["h0"], what="beta=0,g=0 ht")


def check_closed_form_reset(fwd, rng):
    """g = -1000 (exp underflows to exactly 0): S_t = beta_t k_t v_t^T."""
    x = rand_case(rng, 1, 9, 1, 2, 4, 3)
    x["g"][:] = -1000.0
    got = fwd(**x)
    for hv in range(2):
        kq = np.sum(x["k"][0, :, 0] * x["q"][0, :, 0], axis=-1)
        exp_o = (x["beta"][0, :, hv] * kq)[:, None] * x["v"][0, :, hv]
        close(got["o"][0, :, hv], exp_o, what="reset o")
        exp_ht = x["beta"][0, -1, hv] * np.outer(x["k"][0, -1, 0], x["v"][0, -1, hv])
        close(got["ht"][0, hv], exp_ht, what="reset ht")


def check_exact_write(fwd, rng):
    """beta = 1 and unit-norm k: the delta rule writes v exactly, S_t^T k_t = v_t."""
    x = rand_case(rng, 2, 10, 1, 1, 4, 3)
    x["beta"][:] = 1.0
    x["k"] = x["k"] / np.linalg.norm(x["k"], axis=-1, keepdims=True)
    x["q"] = x["k"].copy()
    got = fwd(**x)
    close(got["o"], x["v"], tol=1e-12, what="exact write")


def check_wy_identity(fwd, rng):
    """Coverage guide, section 二: S^r = P^r S^0 + H^r, P^r = I - sum_i k^i w^i^T (g = 0)."""
    from oracle import chunk_form_ref
    K = V = 4
    r = 6
    x = rand_case(rng, 1, r, 1, 1, K, V)
    x["g"][:] = 0.0
    k = x["k"][0, :, 0]
    beta = x["beta"][0, :, 0]
    # P^r by running the recurrence from S^0 = I with v = 0
    xp = {**x, "v": np.zeros_like(x["v"]), "h0": np.eye(K)[None, None].copy()}
    P = fwd(**xp)["ht"][0, 0]
    P_prod = np.eye(K)
    for i in range(r):
        P_prod = (np.eye(K) - beta[i] * np.outer(k[i], k[i])) @ P_prod
    close(P, P_prod, what="P^r vs ordered Householder product")
    cf = chunk_form_ref(k, np.zeros((r, V)), np.zeros(r), beta)
    P_wy = np.eye(K) - k.T @ cf["w"]
    close(P, P_wy, what="P^r vs WY form I - sum k w^T")
    # H^r from zero state, and the decomposition S^r = P^r S^0 + H^r
    Hr = fwd(**{**x, "h0": None})["ht"][0, 0]
    Sr = fwd(**x)["ht"][0, 0]
    close(Sr, P @ x["h0"][0, 0] + Hr, what="S^r = P^r S^0 + H^r")


def check_varlen_equals_separate(fwd, rng):
    lengths = [5, 1, 0, 9, 4]
    x = rand_case(rng, 1, sum(lengths), 2, 4, 3, 5, per_k=True, lengths=lengths)
    whole = fwd(**x, use_qk_l2norm=True)
    cu = x["cu_seqlens"]
    for n in range(len(lengths)):
        s0, s1 = int(cu[n]), int(cu[n + 1])
        if s1 == s0:
            close(whole["ht"][n], x["h0"][n], what="empty sequence keeps h0")
            continue
        part = fwd(q=x["q"][:, s0:s1], k=x["k"][:, s0:s1], v=x["v"][:, s0:s1], g=x["g"][:, s0:s1],
                   beta=x["beta"][:, s0:s1], h0=x["h0"][n:n + 1], use_qk_l2norm=True)
        close(whole["o"][:, s0:s1], part["o"], what=f"varlen o seq {n}")
        close(whole["ht"][n], part["ht"][0], what=f"varlen ht seq {n}")


def check_split_resume(fwd, rng):
    x = rand_case(rng, 2, 13, 1, 2, 3, 4)
    whole = fwd(**x)
    t1 = 6
    a = fwd(**{key: (val[:, :t1] if key in ("q", "k", "v", "g", "beta") else val) for key, val in x.items()})
    b = fwd(**{**{key: (val[:, t1:] if key in ("q", "k", "v", "g", "beta") else val) for key, val in x.items()},
               "h0": a["ht"]})
    close(np.concatenate([a["o"], b["o"]], axis=1), whole["o"], what="resume o")
    close(b["ht"], whole["ht"], what="resume ht")


def check_kda_uniform_equals_gdn(fwd, rng):
    x = rand_case(rng, 1, 8, 1, 2, 4, 3)
    gk = np.repeat(x["g"][..., None], 4, axis=-1)
    a = fwd(**x)
    b = fwd(**{**x, "g": gk})
    close(b["o"], a["o"], what="uniform KDA o")
    close(b["ht"], a["ht"], what="uniform KDA ht")


def check_l2norm(fwd, rng):
    """In-kernel L2 norm equals normalizing first; it is invariant to a positive scale."""
    x = rand_case(rng, 1, 7, 1, 1, 5, 3)
    a = fwd(**x, use_qk_l2norm=True)
    qn = x["q"] / np.sqrt((x["q"] ** 2).sum(-1, keepdims=True) + 1e-6)
    kn = x["k"] / np.sqrt((x["k"] ** 2).sum(-1, keepdims=True) + 1e-6)
    b = fwd(**{**x, "q": qn, "k": kn})
    close(a["o"], b["o"], tol=1e-6, what="l2norm vs pre-normalized")
    c = fwd(**{**x, "q": 7.0 * x["q"], "k": 7.0 * x["k"]}, use_qk_l2norm=True)
    close(c["o"], a["o"], tol=1e-6, what="l2norm scale invariance")


def check_chunk_form(fwd, rng, per_k=False, C=8):
    """UT-transform chunk form against the per-token recurrence, chunk by chunk."""
    from oracle import chunk_form_ref
    T, K, V = 3 * C - 3, 5, 4
    x = rand_case(rng, 1, T, 1, 1, K, V, per_k=per_k)
    ref = fwd(**x, use_qk_l2norm=True, chunk_size=C, want_v_new=True)
    q = x["q"][0, :, 0]
    qn = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6)
    for c in range((T + C - 1) // C):
        s0, s1 = c * C, min(T, (c + 1) * C)
        gch = x["g"][0, s0:s1, 0]
        cf = chunk_form_ref(x["k"][0, s0:s1, 0], x["v"][0, s0:s1, 0], gch, x["beta"][0, s0:s1, 0],
                            use_qk_l2norm=True, gate_per_k=per_k)
        h = ref["h_chunks"][c, 0]
        U = cf["u"] - cf["w"] @ h
        close(U, ref["v_new"][0, s0:s1, 0], tol=1e-10, what=f"v_new = u - w h, chunk {c}")
        Gm, kk = cf["Gamma"], cf["k"]
        h_next = np.exp(Gm[-1])[:, None] * h + (kk * np.exp(Gm[-1] - Gm)).T @ U
        nxt = ref["h_chunks"][c + 1, 0] if s1 < T else ref["ht"][0, 0]
        close(h_next, nxt, tol=1e-10, what=f"state update, chunk {c}")
        Lc = s1 - s0
        Pm = np.zeros((Lc, Lc))
        for r in range(Lc):
            for i in range(r + 1):
                Pm[r, i] = np.sum(qn[s0 + r] * kk[i] * np.exp(Gm[r] - Gm[i]))
        o = (qn[s0:s1] * np.exp(Gm)) @ h + Pm @ U
        close(o, ref["o"][0, s0:s1, 0], tol=1e-10, what=f"chunk output, chunk {c}")


ALL_CHECKS = [check_brute_force, check_closed_form_identity, check_closed_form_reset, check_exact_write,
              check_wy_identity, check_varlen_equals_separate, check_split_resume,
              check_kda_uniform_equals_gdn, check_l2norm, check_chunk_form]
