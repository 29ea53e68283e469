"""Plain, slow, fp64 CPU oracle for the chunked gated delta rule forward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  It shares no code with the
CUDA library (``chunked_gated_delta_08_gb300``) and never imports it.

Contents
--------
* ``gdr_fwd_ref``      -- the per-token recurrence (C, fp64, OpenMP over
                          (sequence, value head)); see ``gdr_oracle.c``.
* ``gdr_fwd_ref_units``-- the same on a sampled subset of (sequence, head) units,
                          for workloads too large to run whole.
* ``gdr_bwd_ref``      -- the reverse recurrence: gradients of o and ht with
                          respect to q, k, v, g, beta and h0 (C, fp64).
* ``chunk_index_ref``  -- the varlen chunk map (sequence, chunk-in-sequence).
* ``chunk_form_ref``   -- the chunk-form intermediates A, T = (I + A)^-1, w, u of
                          one chunk, written from their definitions with a numpy
                          solve as the library step.

Citations name the pages by title: the FLA op-kernel correctness-coverage
guide ("FLA 算子内核正确性测试与覆盖矩阵"), the FLA contributor guide
("Flash Linear Attention 贡献者指南") and the KCP accuracy-debugging handbook
("flash-linear-attention KCP 精度失效根因排查手册").

Parity status: every function here is pinned by tests in ``tests/test_oracle_pins.py``
(brute-force matrix products, closed forms, the WY identity, varlen splitting,
the handbook's chunk-boundary example); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_gdr.so")
_lib = None
_lock = threading.Lock()


def build_oracle(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, IEEE semantics, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_oracle_lib(path: str):
    """Open a compiled oracle library (the default one, or a test's copy)."""
    lib = ctypes.CDLL(path)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.gdr_oracle_fwd.restype = ctypes.c_int
    lib.gdr_oracle_fwd.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_int,
                                   p, p, p, p, p, p, p, i64, ctypes.c_int,
                                   p, p, i64, p, p, ctypes.c_int]
    lib.gdr_oracle_bwd.restype = ctypes.c_int
    lib.gdr_oracle_bwd.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_int,
                                   p, p, p, p, p, p, p, i64, ctypes.c_int,
                                   p, p, p, p, p, p, p, p, ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_oracle()
            _lib = load_oracle_lib(_LIB_PATH)
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact widening to fp64 on the CPU
        x = x.detach().to("cpu").double().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def chunk_index_ref(cu_seqlens, chunk_size: int):
    """Varlen chunk map from cumulative sequence lengths.

    Sequence n holds ceil(len_n / C) chunks; chunk j of sequence n starts at
    global token cu[n] + j*C and is cut short at cu[n+1].  Returns
    ``(chunk_indices [NT, 2] int64 of (n, j), chunk_offsets [N+1] int64)``.
    The KCP handbook's worked example (lengths [400, 624], C = 64: the second
    sequence is cut at global tokens 400, 464, 528, 592, ...) pins this.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    n_seq = len(cu) - 1
    offsets = np.zeros(n_seq + 1, dtype=np.int64)
    pairs = []
    for n in range(n_seq):
        length = int(cu[n + 1] - cu[n])
        nc = -(-length // chunk_size)
        offsets[n + 1] = offsets[n] + nc
        for j in range(nc):
            pairs.append((n, j))
    return np.array(pairs, dtype=np.int64).reshape(-1, 2), offsets


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def gdr_fwd_ref(q, k, v, g, beta, h0=None, cu_seqlens=None, use_qk_l2norm=False,
                chunk_size=None, want_v_new=False, threads=0, lib=None, beta_logits=False):
    """Per-token fp64 recurrence over whole inputs.

    Shapes: q, k [B,T,H,K]; v [B,T,HV,V]; g [B,T,HV] (scalar gate, GDN) or
    [B,T,HV,K] (per-key-channel gate, KDA); beta [B,T,HV]; h0 [N,HV,K,V] or None;
    cu_seqlens [N+1] (host) or None.  Returns a dict of numpy fp64 arrays:
    ``o`` [B,T,HV,V], ``ht`` [N,HV,K,V], and when ``chunk_size`` is given
    ``h_chunks`` [NT,HV,K,V] (state entering each chunk), and when
    ``want_v_new`` the per-token write vectors ``v_new`` [B,T,HV,V].
    With ``beta_logits`` the given beta are logits x and beta = 1/(1 + e^-x)
    (the coverage guide's "raw beta" axis, section 三).
    """
    lib = lib or _load()
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    if beta_logits:
        beta = np.ascontiguousarray(_sigmoid(beta))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    gate_per_k = 1 if g.ndim == 4 else 0
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
        N = len(cu) - 1
    else:
        N = B
    o = np.zeros((B, T, HV, V))
    ht = np.zeros((N, HV, K, V))
    h_chunks = None
    C = int(chunk_size or 0)
    if C > 0:
        lens = np.diff(cu) if cu is not None else np.full(N, T)
        NT = int(sum(-(-int(n) // C) for n in lens))
        h_chunks = np.zeros((NT, HV, K, V))
    v_new = np.zeros((B, T, HV, V)) if want_v_new else None
    rc = lib.gdr_oracle_fwd(B, T, H, HV, K, V, gate_per_k, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), _ptr(h0), _ptr(cu), N, int(bool(use_qk_l2norm)),
                            _ptr(o), _ptr(ht), C, _ptr(h_chunks), _ptr(v_new), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with status {rc}")
    out = {"o": o, "ht": ht}
    if h_chunks is not None:
        out["h_chunks"] = h_chunks
    if v_new is not None:
        out["v_new"] = v_new
    return out


def gdr_bwd_ref(q, k, v, g, beta, do, dht=None, h0=None, cu_seqlens=None, use_qk_l2norm=False,
                threads=0, lib=None, beta_logits=False):
    """Reverse recurrence of the per-token forward, fp64.

    For the loss L = sum(o * do) + sum(ht * dht), returns a dict of numpy fp64
    arrays ``dq``, ``dk`` [B,T,H,K], ``dv`` [B,T,HV,V], ``dg`` shaped like g,
    ``dbeta`` [B,T,HV] and ``dh0`` [N,HV,K,V].  Shapes and layouts of the
    inputs are those of ``gdr_fwd_ref``; ``dht`` None means zero.  With
    ``beta_logits`` beta = sigmoid(x) and ``dbeta`` is dL/dx = dL/dbeta *
    beta (1 - beta), the chain rule through the logistic function.
    """
    lib = lib or _load()
    q, k, v, g, beta, h0, do, dht = (_f64(x) for x in (q, k, v, g, beta, h0, do, dht))
    if beta_logits:
        beta = np.ascontiguousarray(_sigmoid(beta))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    gate_per_k = 1 if g.ndim == 4 else 0
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
        N = len(cu) - 1
    else:
        N = B
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v), "dg": np.zeros_like(g),
           "dbeta": np.zeros_like(beta), "dh0": np.zeros((N, HV, K, V))}
    rc = lib.gdr_oracle_bwd(B, T, H, HV, K, V, gate_per_k, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                            _ptr(h0), _ptr(cu), N, int(bool(use_qk_l2norm)), _ptr(do), _ptr(dht),
                            _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                            _ptr(out["dbeta"]), _ptr(out["dh0"]), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with status {rc}")
    if beta_logits:
        out["dbeta"] = out["dbeta"] * beta * (1.0 - beta)
    return out


def gdr_fwd_ref_units(q, k, v, g, beta, units, h0=None, cu_seqlens=None,
                      use_qk_l2norm=False, threads=0):
    """The recurrence on a sampled set of (sequence n, value head hv) units.

    The units are independent (each carries its own state), so a subset can be
    run alone.  Inputs may be torch tensors of any size; only the rows a unit
    reads are widened to fp64.  Returns ``{(n, hv): (o [len, V], ht [K, V])}``.
    """
    H, HV = q.shape[2], v.shape[2]
    G = HV // H
    if cu_seqlens is not None:
        cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    else:
        T = q.shape[1]
    qs, ks, vs, gs, bs, hs, lens = [], [], [], [], [], [], []
    for (n, hv) in units:
        hq = hv // G
        if cu_seqlens is not None:
            b, s0, s1 = 0, cu[n], cu[n + 1]
        else:
            b, s0, s1 = n, 0, T
        qs.append(_f64(q[b, s0:s1, hq:hq + 1]))
        ks.append(_f64(k[b, s0:s1, hq:hq + 1]))
        vs.append(_f64(v[b, s0:s1, hv:hv + 1]))
        gs.append(_f64(g[b, s0:s1, hv:hv + 1]))
        bs.append(_f64(beta[b, s0:s1, hv:hv + 1]))
        hs.append(None if h0 is None else _f64(h0[n, hv:hv + 1]))
        lens.append(s1 - s0)
    cu_u = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    cat = lambda xs: np.concatenate(xs, axis=0)[None]
    h0_u = None if h0 is None else np.concatenate(hs, axis=0)
    res = gdr_fwd_ref(cat(qs), cat(ks), cat(vs), cat(gs), cat(bs), h0=h0_u, cu_seqlens=cu_u,
                      use_qk_l2norm=use_qk_l2norm, threads=threads)
    out = {}
    for i, unit in enumerate(units):
        out[tuple(unit)] = (res["o"][0, cu_u[i]:cu_u[i + 1], 0], res["ht"][i, 0])
    return out


def chunk_form_ref(k, v, g, beta, use_qk_l2norm=False, gate_per_k=False):
    """Chunk-form intermediates of ONE chunk of one (sequence, value head).

    k [C, K], v [C, V], g [C] or [C, K], beta [C] (fp64 numpy).  With
    Gamma the inclusive within-chunk cumsum of g:
      A_ij = beta_i * sum_d k_id k_jd exp(Gamma_id - Gamma_jd)  for i > j, else 0
      T    = (I + A)^-1
      w    = T diag(beta) (K * exp(Gamma))
      u    = T diag(beta) V
    so that, for a chunk entered with state h, the per-token write vectors are
    v_new = u - w h (the UT transform of the delta rule; at g = 0 this is the
    WY form P^r = I - sum_i k^i w^i^T of the coverage guide, section 二).
    Returns dict(Gamma, A, T, w, u, k) with k L2-normalized when requested.
    """
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    if use_qk_l2norm:
        k = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    C, K = k.shape
    Gam = np.cumsum(g, axis=0)
    if not gate_per_k:
        Gam = np.repeat(Gam[:, None], K, axis=1)
    A = np.zeros((C, C))
    for i in range(C):
        for j in range(i):
            A[i, j] = beta[i] * np.sum(k[i] * k[j] * np.exp(Gam[i] - Gam[j]))
    Tm = np.linalg.solve(np.eye(C) + A, np.eye(C))
    w = Tm @ (beta[:, None] * k * np.exp(Gam))
    u = Tm @ (beta[:, None] * v)
    return {"Gamma": Gam, "A": A, "T": Tm, "w": w, "u": u, "k": k}
