"""Python binding of libgdr.so, the GB300 chunked gated delta rule (forward and backward).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI (``include/gdr.h``).  PyTorch supplies device memory
and streams.  There is no CPU path: if the library is missing the import of
this module raises.

    o, ht = fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, chunk_size=64,
                use_qk_l2norm=False, output_final_state=True)
    dq, dk, dv, dg, dbeta, dh0 = bwd(q, k, v, g, beta, do, dht=None, h0=None, ...)

Layouts: q, k [B,T,H,K]; v [B,T,HV,V]; g [B,T,HV] (GDN) or [B,T,HV,K] (KDA),
fp32; beta [B,T,HV]; h0 [N,HV,K,V] fp32; cu_seqlens [N+1] int64 (B == 1).
q, k, v, beta share one dtype, fp32 or bf16; o has that dtype; ht is fp32.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdr.so")

GDR_OK = 0
GDR_ERR_CHUNK_SIZE = -1
GDR_ERR_SHAPE = -2
GDR_ERR_DTYPE = -3
GDR_ERR_NULLPTR = -4
GDR_ERR_ALIGN = -5
GDR_ERR_CUDA = -6
GDR_ERR_TIMEOUT = -7
GDR_ERR_SEQLENS = -8
GDR_ERR_UNSUPPORTED = -9

GDR_F32, GDR_BF16 = 0, 1
GDR_GATE_SCALAR, GDR_GATE_PER_K = 0, 1
GDR_FLAG_BETA_LOGITS = 1
ALGOS = {"auto": 0, "chunked": 1, "fused": 2, "recurrent": 3, "split": 4}

EXPORTED = ["gdr_fwd", "gdr_bwd", "gdr_fwd_noalloc", "gdr_chunked_sizes_get", "gdr_chunk_index", "gdr_chunk_prepare", "gdr_chunk_fwd_h",
            "gdr_chunk_fwd_o", "gdr_device_status", "gdr_last_error", "gdr_launch_count", "gdr_version"]


class GdrDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64), ("HV", ctypes.c_int64),
                ("K", ctypes.c_int64), ("V", ctypes.c_int64), ("N", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("gate", ctypes.c_int32), ("algo", ctypes.c_int32), ("flags", ctypes.c_int32)]


class GdrChunkedSizes(ctypes.Structure):
    _fields_ = [("nt_max", ctypes.c_int64), ("chunk_indices_bytes", ctypes.c_size_t),
                ("chunk_offsets_bytes", ctypes.c_size_t), ("gcum_bytes", ctypes.c_size_t),
                ("w_bytes", ctypes.c_size_t), ("u_bytes", ctypes.c_size_t), ("v_new_bytes", ctypes.c_size_t),
                ("h_bytes", ctypes.c_size_t)]


class GdrError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"gdr error {code}: {msg}")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
                          "(the CUDA library is required; there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I = ctypes.c_void_p, ctypes.c_int
    D = ctypes.POINTER(GdrDesc)
    lib.gdr_fwd.argtypes = [D, P, P, P, P, P, P, P, I, I, P, P, P]
    lib.gdr_fwd_noalloc.argtypes = [D, P, P, P, P, P, P, P, I, I, P, P, P]
    lib.gdr_bwd.argtypes = [D, P, P, P, P, P, P, P, I, I, P, P, P, P, P, P, P, P, P]
    lib.gdr_chunked_sizes_get.argtypes = [D, I, I, ctypes.POINTER(GdrChunkedSizes)]
    lib.gdr_chunk_index.argtypes = [D, P, I, P, P, P]
    lib.gdr_chunk_prepare.argtypes = [D, P, P, P, P, P, P, I, I, P, P, P, P]
    lib.gdr_chunk_fwd_h.argtypes = [D, P, P, P, P, P, P, P, I, I, P, P, P, P]
    lib.gdr_chunk_fwd_o.argtypes = [D, P, P, P, P, P, P, P, I, I, P, P]
    lib.gdr_device_status.argtypes = [P, I]
    for name in EXPORTED:
        getattr(lib, name).restype = ctypes.c_int
    lib.gdr_last_error.restype = ctypes.c_char_p
    lib.gdr_launch_count.restype = ctypes.c_int64
    return lib


_lib = _load()


def lib():
    return _lib


def version() -> int:
    return _lib.gdr_version()


def launch_count() -> int:
    """Kernels the library has launched in this process."""
    return _lib.gdr_launch_count()


def last_error() -> str:
    return _lib.gdr_last_error().decode()


def _check(rc):
    if rc != GDR_OK:
        msg = last_error()
        if rc in (GDR_ERR_CHUNK_SIZE, GDR_ERR_SHAPE):
            raise ValueError(msg)
        raise GdrError(rc, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_desc(q, v, g, cu_seqlens=None, algo="auto", beta_logits=False) -> GdrDesc:
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    dt = {torch.float32: GDR_F32, torch.bfloat16: GDR_BF16}.get(q.dtype)
    if dt is None:
        raise GdrError(GDR_ERR_DTYPE, f"unsupported dtype {q.dtype}")
    gate = GDR_GATE_PER_K if g.dim() == 4 else GDR_GATE_SCALAR
    return GdrDesc(B, T, H, HV, K, V, N, dt, gate, ALGOS[algo], GDR_FLAG_BETA_LOGITS if beta_logits else 0)


def _require(t, name, dtype=None, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise GdrError(GDR_ERR_NULLPTR, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise GdrError(GDR_ERR_SHAPE, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise GdrError(GDR_ERR_DTYPE, f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _check_inputs(q, k, v, g, beta, h0, cu_seqlens):
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k must be [B,T,H,K] and v [B,T,HV,V]")
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    _require(q, "q")
    _require(k, "k", q.dtype, q.shape)
    _require(v, "v", q.dtype, (B, T, HV, V))
    if g.dim() == 4:
        _require(g, "g", torch.float32, (B, T, HV, K))
    else:
        _require(g, "g", torch.float32, (B, T, HV))
    _require(beta, "beta", q.dtype, (B, T, HV))
    _require(h0, "h0", torch.float32, (N, HV, K, V))
    _require(cu_seqlens, "cu_seqlens", torch.int64)
    return B, T, H, K, HV, V, N


def fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, chunk_size=64, use_qk_l2norm=False,
        output_final_state=True, algo="auto", out=None, final_state=None, stream=None, beta_logits=False):
    """Chunked gated delta rule forward; returns ``(o, ht)`` (ht None unless requested).

    ``beta_logits``: beta holds logits and the kernels apply the sigmoid."""
    B, T, H, K, HV, V, N = _check_inputs(q, k, v, g, beta, h0, cu_seqlens)
    desc = make_desc(q, v, g, cu_seqlens, algo, beta_logits)
    o = out if out is not None else torch.empty(B, T, HV, V, dtype=q.dtype, device=q.device)
    _require(o, "out", q.dtype, (B, T, HV, V))
    ht = None
    if output_final_state:
        ht = final_state if final_state is not None else torch.empty(N, HV, K, V, dtype=torch.float32,
                                                                     device=q.device)
        _require(ht, "final_state", torch.float32, (N, HV, K, V))
    rc = _lib.gdr_fwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                      _ptr(cu_seqlens), int(chunk_size), int(bool(use_qk_l2norm)), _ptr(o), _ptr(ht),
                      _stream_ptr(stream))
    _check(rc)
    return o, ht


def bwd(q, k, v, g, beta, do, dht=None, h0=None, cu_seqlens=None, chunk_size=64, use_qk_l2norm=False,
        out=None, stream=None, beta_logits=False):
    """Backward of ``fwd`` for L = sum(o * do) + sum(ht * dht).

    Returns ``(dq, dk, dv, dg, dbeta, dh0)``: dq, dk, dv, dbeta in the input
    dtype, dg (shaped like g) and dh0 ([N,HV,K,V]) in fp32.  ``dht`` None means
    zero.  ``out`` may give the six output tensors.  The forward's
    intermediates are recomputed inside the call.  With ``beta_logits`` the
    gradient in dbeta is with respect to the logits.
    """
    B, T, H, K, HV, V, N = _check_inputs(q, k, v, g, beta, h0, cu_seqlens)
    _require(do, "do", q.dtype, (B, T, HV, V))
    _require(dht, "dht", torch.float32, (N, HV, K, V))
    desc = make_desc(q, v, g, cu_seqlens, "chunked", beta_logits)
    if out is None:
        dq, dk = torch.empty_like(q), torch.empty_like(k)
        dv, dbeta = torch.empty_like(v), torch.empty_like(beta)
        dg = torch.empty_like(g)
        dh0 = torch.empty(N, HV, K, V, dtype=torch.float32, device=q.device)
    else:
        dq, dk, dv, dg, dbeta, dh0 = out
        for t, ref, name in ((dq, q, "dq"), (dk, k, "dk"), (dv, v, "dv"), (dg, g, "dg"), (dbeta, beta, "dbeta")):
            _require(t, name, ref.dtype, ref.shape)
        _require(dh0, "dh0", torch.float32, (N, HV, K, V))
    rc = _lib.gdr_bwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                      _ptr(cu_seqlens), int(chunk_size), int(bool(use_qk_l2norm)), _ptr(do), _ptr(dht), _ptr(dq),
                      _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0), _stream_ptr(stream))
    _check(rc)
    return dq, dk, dv, dg, dbeta, dh0


def fwd_host(q, k, v, g, beta, h0=None, cu_seqlens=None, chunk_size=64, use_qk_l2norm=False,
             output_final_state=True, algo="auto", device="cuda", out_host=None, final_state_host=None,
             dev_buffers=None, stream=None, pieces=4, beta_logits=False):
    """End-to-end call on HOST tensors: copy inputs in, run, copy o (and ht) back.

    Host tensors should be pinned for asynchronous copies.  ``dev_buffers`` may
    hold reusable device tensors (a dict keyed by input name, plus ``o``, ``ht``
    and the side streams); the call returns after the device-to-host copies
    complete.  A dense batch (no cu_seqlens, B > 1) is processed in up to
    ``pieces`` slices of whole sequences, pipelined on three streams: the
    host-to-device copy of slice p+1, the forward of slice p and the
    device-to-host copy of slice p-1 overlap.  Sequences are independent, so
    the results are those of one call on the whole batch.
    """
    s = stream if stream is not None else torch.cuda.current_stream()
    bufs = dev_buffers if dev_buffers is not None else {}
    B = q.shape[0]
    inputs = (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("h0", h0), ("cu_seqlens", cu_seqlens))
    dev = {}
    for name, t in inputs:
        if t is None:
            dev[name] = None
            continue
        d = bufs.get(name)
        if d is None or d.shape != t.shape or d.dtype != t.dtype:
            d = torch.empty(t.shape, dtype=t.dtype, device=device)
            bufs[name] = d
        dev[name] = d
    HV, V, K = v.shape[2], v.shape[3], q.shape[3]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    o = bufs.get("o")
    if o is None or o.shape != v.shape or o.dtype != q.dtype:
        o = torch.empty(v.shape, dtype=q.dtype, device=device)
        bufs["o"] = o
    ht = None
    if output_final_state:
        ht = bufs.get("ht")
        if ht is None or ht.shape != (N, HV, K, V):
            ht = torch.empty(N, HV, K, V, dtype=torch.float32, device=device)
            bufs["ht"] = ht
    o_h = out_host if out_host is not None else torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    ht_h = None
    if ht is not None:
        ht_h = final_state_host if final_state_host is not None else torch.empty(ht.shape, dtype=ht.dtype,
                                                                                pin_memory=True)
    P = max(1, min(int(pieces), B)) if cu_seqlens is None else 1
    if P == 1:
        with torch.cuda.stream(s):
            for name, t in inputs:
                if t is not None:
                    dev[name].copy_(t, non_blocking=True)
            fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], h0=dev["h0"], cu_seqlens=dev["cu_seqlens"],
                chunk_size=chunk_size, use_qk_l2norm=use_qk_l2norm, output_final_state=output_final_state,
                algo=algo, out=o, final_state=ht, stream=s, beta_logits=beta_logits)
            o_h.copy_(o, non_blocking=True)
            if ht is not None:
                ht_h.copy_(ht, non_blocking=True)
        s.synchronize()
        return o_h, ht_h
    s_in = bufs.setdefault("_stream_in", torch.cuda.Stream(device=device))
    s_out = bufs.setdefault("_stream_out", torch.cuda.Stream(device=device))
    s_in.wait_stream(s)
    bounds = [B * p // P for p in range(P + 1)]
    for p in range(P):
        b0, b1 = bounds[p], bounds[p + 1]
        with torch.cuda.stream(s_in):
            for name, t in inputs:
                if t is not None:
                    dev[name][b0:b1].copy_(t[b0:b1], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
        s.wait_event(ev_in)
        fwd(dev["q"][b0:b1], dev["k"][b0:b1], dev["v"][b0:b1], dev["g"][b0:b1], dev["beta"][b0:b1],
            h0=None if dev["h0"] is None else dev["h0"][b0:b1], chunk_size=chunk_size, use_qk_l2norm=use_qk_l2norm,
            output_final_state=output_final_state, algo=algo, out=o[b0:b1],
            final_state=None if ht is None else ht[b0:b1], stream=s, beta_logits=beta_logits)
        ev_c = torch.cuda.Event()
        ev_c.record(s)
        s_out.wait_event(ev_c)
        with torch.cuda.stream(s_out):
            o_h[b0:b1].copy_(o[b0:b1], non_blocking=True)
            if ht is not None:
                ht_h[b0:b1].copy_(ht[b0:b1], non_blocking=True)
    s_out.synchronize()
    s.synchronize()
    return o_h, ht_h


def chunked_sizes(desc: GdrDesc, chunk_size: int, varlen: bool) -> GdrChunkedSizes:
    out = GdrChunkedSizes()
    _check(_lib.gdr_chunked_sizes_get(ctypes.byref(desc), int(chunk_size), int(varlen), ctypes.byref(out)))
    return out


def chunk_stages(q, k, v, g, beta, h0=None, cu_seqlens=None, chunk_size=64, use_qk_l2norm=False, stream=None):
    """Runs the chunked form stage by stage and returns every intermediate.

    Returns a dict with chunk_indices, chunk_offsets (varlen only), gcum, w, u,
    h (state entering each chunk, [NT_max, HV, K, V]), v_new, o and ht.
    """
    B, T, H, K, HV, V, N = _check_inputs(q, k, v, g, beta, h0, cu_seqlens)
    desc = make_desc(q, v, g, cu_seqlens, "chunked")
    sz = chunked_sizes(desc, chunk_size, cu_seqlens is not None)
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    sp = _stream_ptr(stream)
    out = {}
    ci = co = None
    if cu_seqlens is not None:
        ci = torch.empty(sz.nt_max, 2, dtype=torch.int64, device=dev)
        co = torch.empty(N + 1, dtype=torch.int64, device=dev)
        _check(_lib.gdr_chunk_index(ctypes.byref(desc), _ptr(cu_seqlens), int(chunk_size), _ptr(ci), _ptr(co), sp))
        out["chunk_indices"], out["chunk_offsets"] = ci, co
    gcum = torch.empty(*g.shape, **f32)
    w = torch.empty(B, T, HV, K, **f32)
    u = torch.empty(B, T, HV, V, **f32)
    _check(_lib.gdr_chunk_prepare(ctypes.byref(desc), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                  _ptr(ci), int(chunk_size), int(bool(use_qk_l2norm)), _ptr(gcum), _ptr(w), _ptr(u),
                                  sp))
    h = torch.empty(sz.nt_max, HV, K, V, **f32)
    v_new = torch.empty(B, T, HV, V, **f32)
    ht = torch.empty(N, HV, K, V, **f32)
    _check(_lib.gdr_chunk_fwd_h(ctypes.byref(desc), _ptr(k), _ptr(w), _ptr(u), _ptr(gcum), _ptr(h0),
                                _ptr(cu_seqlens), _ptr(co), int(chunk_size), int(bool(use_qk_l2norm)), _ptr(h),
                                _ptr(v_new), _ptr(ht), sp))
    o = torch.empty(B, T, HV, V, dtype=q.dtype, device=dev)
    _check(_lib.gdr_chunk_fwd_o(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v_new), _ptr(h), _ptr(gcum),
                                _ptr(cu_seqlens), _ptr(ci), int(chunk_size), int(bool(use_qk_l2norm)), _ptr(o), sp))
    out.update(gcum=gcum, w=w, u=u, h=h, v_new=v_new, o=o, ht=ht)
    return out


def device_status(stream=None, clear=True) -> int:
    """Synchronizes the stream and returns the library's device status word."""
    return _lib.gdr_device_status(_stream_ptr(stream), int(bool(clear)))
