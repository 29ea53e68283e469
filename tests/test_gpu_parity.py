"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Tolerances: relative L2 error <= 1e-5 for fp32 inputs and <= 5e-3 for bf16
inputs, on o and ht (the 0.005 assert_close bar of the coverage guide,
section 三; the fp32 bar is the tighter one set for fp32 inputs).  The metric is
||x - ref||_2 / ||ref||_2 over the whole tensor (FLA contributor guide,
section Testing: RMS(diff) / RMS(ref)), with any NaN a failure.

Pages cited: the coverage guide = "FLA 算子内核正确性测试与覆盖矩阵" (fla/ops correctness-coverage guide); the contributor guide = "Flash Linear Attention 贡献者指南".
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 5e-3}
ALGOS = ["chunked", "auto"]


def rel_l2(got, want):
    got = got.detach().double().cpu().numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.isfinite(got).all(), "non-finite values in the CUDA output"
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def to_dev(x):
    return {k: (None if v is None else v.cuda()) for k, v in x.items()}


def poisoned_like(shape, dtype):
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


def run_gpu(gdr, x, C, l2, algo, poison=True):
    d = to_dev(x)
    B, T, H, K = d["q"].shape
    HV, V = d["v"].shape[2], d["v"].shape[3]
    N = B if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    o = poisoned_like((B, T, HV, V), d["q"].dtype) if poison else None
    ht = poisoned_like((N, HV, K, V), torch.float32) if poison else None
    o, ht = gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
                    chunk_size=C, use_qk_l2norm=l2, algo=algo, out=o, final_state=ht)
    assert gdr.device_status() == 0, gdr.last_error()
    return o, ht


def run_ref(x, l2, **kw):
    return oracle.gdr_fwd_ref(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], cu_seqlens=x["cu_seqlens"],
                              use_qk_l2norm=l2, **kw)


def assert_parity(o, ht, ref, dtype, what=""):
    tol = TOL[dtype]
    eo, eh = rel_l2(o, ref["o"]), rel_l2(ht, ref["ht"])
    assert eo <= tol and eh <= tol, f"{what}: o err {eo:.2e}, ht err {eh:.2e} (tol {tol:.0e})"
    return eo, eh


# ---------------------------------------------------------------- the five workloads
@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("w", [wl.GDN_FP32_SMALL, wl.GDN_BF16_GVA_K60, wl.GDN_BF16_VARLEN, wl.KDA_BF16_VARLEN],
                         ids=lambda w: w.name)
def test_workload_parity(gdr, w, algo):
    x = wl.make_inputs(w)
    o, ht = run_gpu(gdr, x, w.chunk_size, w.use_qk_l2norm, algo)
    ref = run_ref(x, w.use_qk_l2norm)
    assert_parity(o, ht, ref, w.dtype, w.name)


def test_gva_workload_rejects_chunk_size_16(gdr):
    w = wl.GDN_BF16_GVA_K60
    d = to_dev(wl.make_inputs(w))
    with pytest.raises(ValueError, match="chunk_size must be either 32 or 64"):
        gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], chunk_size=16, use_qk_l2norm=True)


def test_varlen_equals_separate_runs_bitwise(gdr):
    """Sequences of a varlen batch give exactly the bits they give alone."""
    w = wl.GDN_BF16_VARLEN
    x = wl.make_inputs(w)
    for algo in ["chunked", "fused"]:
        o, ht = run_gpu(gdr, x, w.chunk_size, w.use_qk_l2norm, algo)
        cu = w.cu_seqlens
        for n in range(w.N):
            s0, s1 = cu[n], cu[n + 1]
            part = {"q": x["q"][:, s0:s1].contiguous(), "k": x["k"][:, s0:s1].contiguous(),
                    "v": x["v"][:, s0:s1].contiguous(), "g": x["g"][:, s0:s1].contiguous(),
                    "beta": x["beta"][:, s0:s1].contiguous(), "h0": x["h0"][n:n + 1].contiguous(),
                    "cu_seqlens": None}
            op, hp = run_gpu(gdr, part, w.chunk_size, w.use_qk_l2norm, algo)
            assert torch.equal(op, o[:, s0:s1]), f"{algo}: o of sequence {n} differs from its separate run"
            assert torch.equal(hp[0], ht[n]), f"{algo}: ht of sequence {n} differs from its separate run"


@pytest.mark.parametrize("N", [37, 300], ids=["ranked", "beyond_rank_limit"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_many_varied_sequences(gdr, N, dtype):
    """Many sequences of mixed lengths (the state scans launch their blocks
    longest sequence first, ranking up to 256 sequences in the block and
    taking index order beyond that): both paths against the oracle."""
    rng = np.random.default_rng(61 + N)
    lengths = [int(x) for x in rng.integers(1, 200, size=N)]
    lengths[N // 2] = 700  # one long sequence among short ones
    T = sum(lengths)
    _, x = wl.random_case(1, T, 2, 2, 32, 48, dtype=dtype, lengths=lengths, gate_per_k=(N == 37), seed=N)
    o, ht = run_gpu(gdr, x, 64, True, "chunked")
    ref = run_ref(x, True)
    assert_parity(o, ht, ref, dtype, f"{N} sequences")


# ---------------------------------------------------------------- large dense workload, every unit
@pytest.mark.parametrize("algo", ["chunked", "fused"])
def test_large_dense_all_units(gdr, algo):
    """Full-size B=4, T=32768, H=HV=32, K=V=128 bf16 run, in the launch configuration
    the bench times; the oracle checks every one of the 128 (sequence, head) units
    whole, o and ht, and every output is finite."""
    w = wl.GDN_BF16_LARGE
    x = wl.make_inputs(w)
    o, ht = run_gpu(gdr, x, w.chunk_size, w.use_qk_l2norm, algo)
    assert torch.isfinite(o).all() and torch.isfinite(ht).all()
    o, ht = o.cpu(), ht.cpu()
    units = [(n, hv) for n in range(w.B) for hv in range(w.HV)]
    # batches of 16 units keep the oracle's fp64 copies of the inputs to about 2 GB
    num = {"o": 0.0, "ht": 0.0}
    den = {"o": 0.0, "ht": 0.0}
    seen = 0
    for b0 in range(0, len(units), 16):
        ref = oracle.gdr_fwd_ref_units(x["q"], x["k"], x["v"], x["g"], x["beta"], units[b0:b0 + 16],
                                       use_qk_l2norm=True)
        for (n, hv), (ro, rh) in ref.items():
            go, gh = o[n, :, hv].double().numpy(), ht[n, hv].double().numpy()
            eo, eh = rel_l2(go, ro), rel_l2(gh, rh)
            assert eo <= TOL[w.dtype] and eh <= TOL[w.dtype], f"unit {(n, hv)}: o {eo:.2e} ht {eh:.2e}"
            num["o"] += float(np.sum((go - ro) ** 2))
            den["o"] += float(np.sum(ro ** 2))
            num["ht"] += float(np.sum((gh - rh) ** 2))
            den["ht"] += float(np.sum(rh ** 2))
            seen += 1
    assert seen == len(units) == 128
    # the whole tensors too, not only unit by unit
    for key in ("o", "ht"):
        err = (num[key] / den[key]) ** 0.5
        assert err <= TOL[w.dtype], f"whole {key}: {err:.2e}"


# ---------------------------------------------------------------- unit grid
GRID = [
    # B, T, H, HV, K, V, lengths, per_k
    (1, 1, 1, 1, 64, 64, None, False),
    (1, 63, 1, 1, 64, 64, None, False),
    (2, 64, 1, 2, 64, 32, None, False),
    (1, 65, 2, 2, 60, 60, None, False),
    (2, 100, 2, 4, 60, 100, None, False),
    (1, 2000, 1, 1, 128, 128, None, False),
    (1, 300, 1, 3, 32, 48, (1, 64, 0, 170, 65), False),
    (1, 64, 1, 1, 64, 64, None, True),
    (1, 64, 1, 2, 64, 64, None, True),
    (2, 512, 2, 4, 60, 60, None, True),
    (1, 333, 2, 4, 128, 256, (100, 233), True),
]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("C", [32, 64])
@pytest.mark.parametrize("case", GRID, ids=lambda c: "x".join(str(v) for v in c[:6]) + ("_kda" if c[7] else ""))
def test_unit_grid(gdr, case, C, dtype, algo):
    B, T, H, HV, K, V, lengths, per_k = case
    for l2, use_h0 in ((True, True), (False, False)):
        _, x = wl.random_case(B, T, H, HV, K, V, dtype=dtype, lengths=lengths, gate_per_k=per_k,
                              use_h0=use_h0, seed=T + K)
        if not l2:
            # the in-kernel norm is off: q, k arrive normalized, as the coverage guide's
            # use_qk_l2norm_in_kernel=False axis prepares them (section 三)
            x["q"] = torch.nn.functional.normalize(x["q"].float(), dim=-1).to(dtype)
            x["k"] = torch.nn.functional.normalize(x["k"].float(), dim=-1).to(dtype)
        o, ht = run_gpu(gdr, x, C, l2, algo)
        ref = run_ref(x, l2)
        assert_parity(o, ht, ref, dtype, f"{case} C={C} l2={l2} h0={use_h0}")


# ---------------------------------------------------------------- fused form, weak and strong decay
@pytest.mark.parametrize("gate_div", [1.0, 16.0, 256.0])
@pytest.mark.parametrize("lengths", [None, (1000, 17, 64, 300)], ids=["dense", "varlen"])
def test_fused_decay_regimes(gdr, gate_div, lengths):
    """The fused tensor-core kernel where the chunk's off-diagonal blocks of A
    and T carry weight (weak decay: g = logsigmoid(N(0,1)) / 256) as well as
    where they vanish (g = logsigmoid(N(0,1))), with an initial state, the
    in-kernel L2 norm and partial last chunks."""
    B = 1 if lengths else 2
    T = sum(lengths) if lengths else 700
    _, x = wl.random_case(B, T, 2, 4, 128, 128, dtype=torch.bfloat16, lengths=lengths, use_h0=True, seed=61,
                          gate_div=gate_div)
    o, ht = run_gpu(gdr, x, 64, True, "fused")
    assert_parity(o, ht, run_ref(x, True), torch.bfloat16, f"gate_div={gate_div}")


# ---------------------------------------------------------------- over-read detection
@pytest.mark.parametrize("per_k,D", [(False, 60), (True, 60), (False, 128)])
def test_padding_poison_detects_overreads(gdr, per_k, D):
    """Inputs sit at the front of buffers whose tails hold NaN (q, k, v, beta) or
    1e30 (g, the coverage guide's section 七 padding); any read past a tensor's
    end would make the outputs non-finite or wrong.  D = 128 takes the fused form."""
    _, x = wl.random_case(1, 190, 1, 2, D, D, dtype=torch.bfloat16, gate_per_k=per_k, seed=5)
    d = {}
    for name in ("q", "k", "v", "beta", "g"):
        t = x[name]
        pad = 1e30 if name == "g" else float("nan")
        buf = torch.full((t.numel() + 4096,), pad, dtype=t.dtype, device="cuda")
        buf[:t.numel()].copy_(t.reshape(-1))
        d[name] = buf[:t.numel()].view(t.shape)
    h0 = x["h0"].cuda()
    o, ht = gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=h0, chunk_size=64, use_qk_l2norm=True,
                    out=poisoned_like((1, 190, 2, D), torch.bfloat16),
                    final_state=poisoned_like((1, 2, D, D), torch.float32))
    ref = run_ref(x, True)
    assert_parity(o, ht, ref, torch.bfloat16, "padded inputs")


# ---------------------------------------------------------------- intermediates
@pytest.mark.parametrize("per_k", [False, True])
def test_chunk_intermediates(gdr, per_k):
    """h (state entering each chunk) and the per-token v_new against the oracle's
    per-token recurrence; w and u against the oracle's chunk-form helper."""
    lengths = (70, 130)
    _, x = wl.random_case(1, 200, 1, 2, 32, 24, dtype=torch.float32, lengths=lengths, gate_per_k=per_k, seed=9)
    C = 32
    st = gdr.chunk_stages(*[x[k].cuda() for k in ("q", "k", "v", "g", "beta")], h0=x["h0"].cuda(),
                          cu_seqlens=x["cu_seqlens"].cuda(), chunk_size=C, use_qk_l2norm=True)
    torch.cuda.synchronize()
    ref = run_ref(x, True, chunk_size=C, want_v_new=True)
    idx, off = oracle.chunk_index_ref(x["cu_seqlens"].numpy(), C)
    NT = len(idx)
    assert st["chunk_offsets"].cpu().tolist() == off.tolist()
    assert st["chunk_indices"][:NT].cpu().tolist() == idx.tolist()
    assert (st["chunk_indices"][NT:] == -1).all()
    assert rel_l2(st["h"][:NT], ref["h_chunks"]) <= 1e-5
    assert rel_l2(st["v_new"], ref["v_new"]) <= 1e-5
    assert rel_l2(st["o"], ref["o"]) <= 1e-5 and rel_l2(st["ht"], ref["ht"]) <= 1e-5
    cu = x["cu_seqlens"].tolist()
    for (n, j) in idx[:: max(1, NT // 4)]:
        s0 = cu[n] + j * C
        s1 = min(s0 + C, cu[n + 1])
        cf = oracle.chunk_form_ref(x["k"][0, s0:s1, 0].numpy(), x["v"][0, s0:s1, 1].numpy(),
                                   x["g"][0, s0:s1, 1].numpy(), x["beta"][0, s0:s1, 1].numpy(),
                                   use_qk_l2norm=True, gate_per_k=per_k)
        assert rel_l2(st["w"][0, s0:s1, 1], cf["w"]) <= 1e-5
        assert rel_l2(st["u"][0, s0:s1, 1], cf["u"]) <= 1e-5
        gam = cf["Gamma"] if per_k else cf["Gamma"][:, 0]
        assert rel_l2(st["gcum"][0, s0:s1, 1], gam) <= 1e-6


# ---------------------------------------------------------------- semantics
def test_resume_from_final_state(gdr):
    _, x = wl.random_case(2, 300, 1, 2, 64, 64, dtype=torch.float32, seed=3)
    d = to_dev(x)
    o, ht = gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], chunk_size=64, use_qk_l2norm=True)
    t1 = 131
    sl = lambda t, a, b: t[:, a:b].contiguous()
    o1, h1 = gdr.fwd(*[sl(d[k], 0, t1) for k in ("q", "k", "v", "g", "beta")], h0=d["h0"], chunk_size=64,
                     use_qk_l2norm=True)
    o2, h2 = gdr.fwd(*[sl(d[k], t1, 300) for k in ("q", "k", "v", "g", "beta")], h0=h1, chunk_size=64,
                     use_qk_l2norm=True)
    assert rel_l2(torch.cat([o1, o2], 1), o.double().cpu().numpy()) <= 1e-5
    assert rel_l2(h2, ht.double().cpu().numpy()) <= 1e-5


def test_no_final_state_and_zero_length(gdr):
    _, x = wl.random_case(1, 0, 1, 1, 64, 64, dtype=torch.bfloat16, seed=1)
    d = to_dev(x)
    o, ht = gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], chunk_size=64)
    assert o.numel() == 0 and torch.equal(ht, d["h0"])
    _, x = wl.random_case(1, 70, 1, 1, 64, 64, dtype=torch.bfloat16, seed=1)
    d = to_dev(x)
    o, ht = gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], chunk_size=64, output_final_state=False)
    assert ht is None and torch.isfinite(o).all()


def test_bad_cu_seqlens_reported_on_device(gdr):
    _, x = wl.random_case(1, 100, 1, 1, 64, 64, dtype=torch.bfloat16, lengths=(40, 60), seed=2)
    d = to_dev(x)
    d["cu_seqlens"] = torch.tensor([0, 70, 60], dtype=torch.int64, device="cuda")
    o = poisoned_like((1, 100, 1, 64), torch.bfloat16)
    gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"], chunk_size=64, out=o,
            algo="chunked")
    assert gdr.device_status(clear=True) == gdr.GDR_ERR_SEQLENS
    assert torch.isnan(o.float()).all()
    assert gdr.device_status() == 0


def test_deterministic(gdr):
    w = wl.GDN_BF16_GVA_K60
    x = wl.make_inputs(w)
    a = run_gpu(gdr, x, 64, True, "auto")
    b = run_gpu(gdr, x, 64, True, "auto")
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_host_buffers_end_to_end(gdr):
    w = wl.GDN_BF16_VARLEN
    x = wl.make_inputs(w)
    pinned = {k: (None if v is None else v.pin_memory()) for k, v in x.items()}
    o_h, ht_h = gdr.fwd_host(pinned["q"], pinned["k"], pinned["v"], pinned["g"], pinned["beta"], h0=pinned["h0"],
                             cu_seqlens=pinned["cu_seqlens"], chunk_size=64)
    o_d, ht_d = run_gpu(gdr, x, 64, False, "auto", poison=False)
    assert not o_h.is_cuda and torch.equal(o_h, o_d.cpu()) and torch.equal(ht_h, ht_d.cpu())


@pytest.mark.parametrize("algo", ["auto", "chunked"])
def test_host_buffers_pipelined_dense(gdr, algo):
    """A dense batch goes through fwd_host in pipelined slices; results equal one device call bit for bit."""
    w, x = wl.random_case(5, 300, 2, 4, 128, 128, dtype=torch.bfloat16, seed=61)
    pinned = {k: (None if v is None else v.pin_memory()) for k, v in x.items()}
    bufs = {}
    for _ in range(2):  # the second call reuses the device buffers and side streams
        o_h, ht_h = gdr.fwd_host(pinned["q"], pinned["k"], pinned["v"], pinned["g"], pinned["beta"],
                                 h0=pinned["h0"], use_qk_l2norm=True, algo=algo, dev_buffers=bufs, pieces=3)
    o_d, ht_d = run_gpu(gdr, x, 64, True, algo, poison=False)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(ht_h, ht_d.cpu())


# ---------------------------------------------------------------- fused tensor-core form
FUSED_GRID = [
    # B, T, H, HV, lengths
    (1, 64, 1, 1, None),
    (2, 1000, 1, 2, None),
    (1, 1, 1, 1, None),
    (3, 130, 2, 4, None),
    (1, 777, 1, 2, (1, 63, 64, 65, 584)),
    (1, 2048, 4, 4, (0, 1024, 1024)),
]


@pytest.mark.parametrize("case", FUSED_GRID, ids=lambda c: "x".join(str(v) for v in c[:4]) + ("_varlen" if c[4] else ""))
def test_fused_grid(gdr, case):
    B, T, H, HV, lengths = case
    for l2, use_h0 in ((True, True), (False, False)):
        _, x = wl.random_case(B, T, H, HV, 128, 128, dtype=torch.bfloat16, lengths=lengths, use_h0=use_h0,
                              seed=T + HV)
        if not l2:
            x["q"] = torch.nn.functional.normalize(x["q"].float(), dim=-1).to(torch.bfloat16)
            x["k"] = torch.nn.functional.normalize(x["k"].float(), dim=-1).to(torch.bfloat16)
        o, ht = run_gpu(gdr, x, 64, l2, "fused")
        ref = run_ref(x, l2)
        assert_parity(o, ht, ref, torch.bfloat16, f"fused {case} l2={l2} h0={use_h0}")


def test_fused_matches_chunked_form(gdr):
    """The two forms agree with each other as well as with the oracle."""
    w = wl.GDN_BF16_VARLEN
    x = wl.make_inputs(w)
    of, hf = run_gpu(gdr, x, 64, False, "fused")
    oc, hc = run_gpu(gdr, x, 64, False, "chunked")
    assert rel_l2(of, oc.double().cpu().numpy()) <= 5e-3
    assert rel_l2(hf, hc.double().cpu().numpy()) <= 5e-3


@pytest.mark.parametrize("what", ["f32", "K60", "C32", "kda"])
def test_fused_reports_unsupported(gdr, what):
    kw = dict(B=1, T=70, H=1, HV=1, K=128, V=128, dtype=torch.bfloat16)
    C = 64
    if what == "f32":
        kw["dtype"] = torch.float32
    elif what == "K60":
        kw["K"] = 60
    elif what == "C32":
        C = 32
    _, x = wl.random_case(**kw, gate_per_k=(what == "kda"), seed=1)
    with pytest.raises(gdr.GdrError) as ei:
        run_gpu(gdr, x, C, True, "fused")
    assert ei.value.code == gdr.GDR_ERR_UNSUPPORTED
    o, ht = run_gpu(gdr, x, C, True, "auto")  # the dispatcher falls back to the chunked form
    assert_parity(o, ht, run_ref(x, True), kw["dtype"], f"auto fallback {what}")
