"""gdr_fwd_noalloc: the chunked forward for callers that cannot allocate device
memory (their framework's allocator owns the device, or allocation calls are
not allowed where they run).  Its scratch is a fixed device array inside the
library instead of memory from an allocator.

This file is collected last on purpose: the GPU test below runs after every
other test in a full run, and also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

import workloads as wl

TOL = {torch.float32: 1e-5, torch.bfloat16: 5e-3}


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


def _noalloc(gdr, d, C, l2):
    """One call of the new entry point through the C ABI on device tensors."""
    B, T, H, K = d["q"].shape
    HV, V = d["v"].shape[2], d["v"].shape[3]
    N = B if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    o = torch.full((B, T, HV, V), float("nan"), dtype=d["q"].dtype, device="cuda")
    ht = torch.full((N, HV, K, V), float("nan"), dtype=torch.float32, device="cuda")
    desc = gdr.make_desc(d["q"], d["v"], d["g"], d["cu_seqlens"], "auto")
    P = gdr._ptr
    rc = gdr.lib().gdr_fwd_noalloc(ctypes.byref(desc), P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]),
                                   P(d["h0"]), P(d["cu_seqlens"]), C, int(l2), P(o), P(ht),
                                   gdr._stream_ptr(None))
    assert rc == 0, gdr.last_error()
    torch.cuda.synchronize()
    return o, ht


def _fwd_chunked(gdr, d, C, l2):
    o, ht = gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
                    chunk_size=C, use_qk_l2norm=l2, algo="chunked")
    torch.cuda.synchronize()
    return o, ht


def _dev(x):
    return {k: (None if t is None else t.cuda()) for k, t in x.items()}


@pytest.mark.gpu
def test_noalloc_matches_gdr_fwd_on_two_calls_in_a_row(gdr):
    """The same kernels on the same inputs as gdr_fwd's chunked form, so the
    results must be identical bit for bit: on two workloads of different shapes,
    then on one shape twice with different inputs (nothing may carry over from
    the previous call's contents of the shared array)."""
    runs = [(wl.GDN_BF16_VARLEN, None), (wl.GDN_BF16_GVA_K60, None), (wl.GDN_BF16_GVA_K60, 7)]
    for w, seed in runs:
        d = _dev(wl.make_inputs(w, seed=seed))
        o_ref, ht_ref = _fwd_chunked(gdr, d, w.chunk_size, w.use_qk_l2norm)
        o, ht = _noalloc(gdr, d, w.chunk_size, w.use_qk_l2norm)
        assert torch.isfinite(o.float()).all() and torch.isfinite(ht).all()
        assert torch.equal(o, o_ref) and torch.equal(ht, ht_ref), (w.name, seed)
        # and within the parity tolerance of the other tests, for the record
        assert _rel(o, o_ref) <= TOL[w.dtype] and _rel(ht, ht_ref) <= TOL[w.dtype]


@pytest.mark.gpu
def test_noalloc_bad_cu_seqlens_leaves_outputs_untouched(gdr):
    """cu_seqlens that decrease: nothing is written (there is no status word on
    this path, so the NaN-filled outputs are the evidence)."""
    w, x = wl.random_case(1, 2000, 1, 1, 32, 32, dtype=torch.float32, lengths=(1500, 500), seed=53)
    d = _dev(x)
    d["cu_seqlens"] = torch.tensor([0, 1600, 1500], dtype=torch.int64, device="cuda")
    o, ht = _noalloc(gdr, d, 64, True)
    assert torch.isnan(o).all() and torch.isnan(ht).all()
    # a good call right after still matches gdr_fwd exactly
    d = _dev(x)
    o_ref, ht_ref = _fwd_chunked(gdr, d, 64, True)
    o, ht = _noalloc(gdr, d, 64, True)
    assert torch.equal(o, o_ref) and torch.equal(ht, ht_ref)


def test_noalloc_rejects_requests_beyond_its_array(gdr):
    """Checked on the host before anything is launched."""
    desc = gdr.GdrDesc(4, 32768, 32, 32, 128, 128, 4, gdr.GDR_BF16, gdr.GDR_GATE_SCALAR, 0, 0)
    fake = ctypes.c_void_p(256)  # never dereferenced: the request is refused first
    rc = gdr.lib().gdr_fwd_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, None, None, 64, 1, fake, None,
                                   None)
    assert rc == gdr.GDR_ERR_SHAPE
    assert "bytes of scratch" in gdr.last_error()
