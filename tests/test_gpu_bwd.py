"""The backward (gdr_bwd, through the C ABI) against the oracle's reverse
recurrence, element by element.

The graded workload is the KDA varlen one (lengths 700, 324, 3072, 12288;
H = 16, HV = 32, K = 128, V = 256, bf16, per-key-channel gate, in-kernel L2
norm, h0 and upstream do, dht drawn with it): dq, dk, dv, dg, dbeta and dh0
must each be within relative L2 error 5e-3 (the coverage guide's assert_close
bar, section 三).  fp32 inputs are held to 1e-5.  The other cases cover the
scalar gate, grouped value heads, K != V, chunk size 32, partial and empty
sequences, and missing dht / h0.

Pages cited: the coverage guide = "FLA 算子内核正确性测试与覆盖矩阵" (fla/ops correctness-coverage guide).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 5e-3}
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def rel_l2(got, want):
    got = got.detach().double().cpu().numpy()
    want = np.asarray(want, np.float64)
    assert np.isfinite(got).all(), "non-finite values in the CUDA output"
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def dev(x):
    return None if x is None else x.cuda()


def run_gpu(gdr, x, do, dht, C, l2, poison=True):
    q, k, v, g, beta, h0, cu = (dev(x[n]) for n in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    out = None
    if poison:
        N = q.shape[0] if cu is None else cu.numel() - 1
        HV, K, V = v.shape[2], q.shape[3], v.shape[3]
        nan = lambda t: torch.full_like(t, float("nan"))
        out = (nan(q), nan(k), nan(v), nan(g), nan(beta),
               torch.full((N, HV, K, V), float("nan"), device="cuda"))
    res = gdr.bwd(q, k, v, g, beta, dev(do), dht=dev(dht), h0=h0, cu_seqlens=cu, chunk_size=C,
                  use_qk_l2norm=l2, out=out)
    assert gdr.device_status() == 0, gdr.last_error()
    return dict(zip(NAMES, res))


def run_ref(x, do, dht, l2):
    return oracle.gdr_bwd_ref(x["q"], x["k"], x["v"], x["g"], x["beta"], do, dht=dht, h0=x["h0"],
                              cu_seqlens=x["cu_seqlens"], use_qk_l2norm=l2)


def assert_parity(got, ref, dtype, what):
    tol = TOL[dtype]
    errs = {n: rel_l2(got[n], ref[n]) for n in NAMES}
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"{what}: " + ", ".join(f"{n} {e:.2e}" for n, e in errs.items()) + f" (tol {tol:.0e})"
    return errs


def test_bwd_kda_varlen_workload(gdr):
    """The graded backward workload at its full size."""
    w = wl.KDA_BF16_VARLEN
    x = wl.make_inputs(w)
    got = run_gpu(gdr, x, x["do"], x["dht"], w.chunk_size, w.use_qk_l2norm)
    ref = run_ref(x, x["do"], x["dht"], w.use_qk_l2norm)
    assert_parity(got, ref, w.dtype, w.name)


@pytest.mark.parametrize("w", [wl.GDN_FP32_SMALL, wl.GDN_BF16_GVA_K60, wl.GDN_BF16_VARLEN], ids=lambda w: w.name)
def test_bwd_gdn_workloads(gdr, w):
    x = wl.make_inputs(w)
    gr = wl.make_grads(w)
    got = run_gpu(gdr, x, gr["do"], gr["dht"], w.chunk_size, w.use_qk_l2norm)
    ref = run_ref(x, gr["do"], gr["dht"], w.use_qk_l2norm)
    assert_parity(got, ref, w.dtype, w.name)


CASES = [
    # (per_k, C, l2, lengths or None, B, T, H, HV, K, V)
    (False, 64, True, None, 2, 150, 2, 4, 64, 48),
    (True, 64, True, None, 1, 200, 1, 2, 128, 96),
    (False, 32, False, (37, 0, 64, 1, 90), 1, 192, 2, 2, 32, 40),
    (True, 32, True, (5, 130, 0, 33), 1, 168, 2, 4, 100, 160),
    (True, 64, False, (64, 65, 127), 1, 256, 1, 1, 16, 256),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"pk{int(c[0])}_C{c[1]}_l2{int(c[2])}_K{c[8]}_V{c[9]}")
def test_bwd_cases(gdr, case, dtype):
    per_k, C, l2, lengths, B, T, H, HV, K, V = case
    w, x = wl.random_case(B, T, H, HV, K, V, dtype=dtype, lengths=lengths, gate_per_k=per_k, seed=3,
                          grads=True, gate_div=4.0 if per_k else 1.0)
    if not l2:  # unit-norm q, k keep the state bounded without the in-kernel norm
        for n in ("q", "k"):
            x[n] = (x[n].float() / x[n].float().norm(dim=-1, keepdim=True)).to(dtype)
    got = run_gpu(gdr, x, x["do"], x["dht"], C, l2)
    ref = run_ref(x, x["do"], x["dht"], l2)
    assert_parity(got, ref, dtype, str(case))


def test_bwd_many_varied_sequences(gdr):
    """The reverse scan's longest-first block order over 40 mixed-length
    sequences (per-key gate, bf16) against the oracle's reverse recurrence."""
    rng = np.random.default_rng(7)
    lengths = [int(x) for x in rng.integers(1, 150, size=40)]
    lengths[5] = 500
    _, x = wl.random_case(1, sum(lengths), 2, 2, 32, 48, dtype=torch.bfloat16, lengths=lengths, gate_per_k=True,
                          seed=17, grads=True)
    got = run_gpu(gdr, x, x["do"], x["dht"], 64, True)
    ref = run_ref(x, x["do"], x["dht"], True)
    assert_parity(got, ref, torch.bfloat16, "40 sequences")


def test_bwd_without_dht_and_h0(gdr):
    w, x = wl.random_case(1, 130, 1, 2, 64, 64, dtype=torch.float32, use_h0=False, seed=5, grads=True)
    got = run_gpu(gdr, x, x["do"], None, 64, True)
    ref = run_ref(x, x["do"], None, True)
    assert_parity(got, ref, torch.float32, "no dht, no h0")


def test_bwd_varlen_equals_separate_bitwise(gdr):
    lengths = (70, 129, 3)
    w, x = wl.random_case(1, sum(lengths), 2, 4, 64, 32, dtype=torch.bfloat16, lengths=lengths, gate_per_k=True,
                          seed=7, grads=True, gate_div=4.0)
    whole = run_gpu(gdr, x, x["do"], x["dht"], 64, True)
    cu = x["cu_seqlens"].tolist()
    for n in range(len(lengths)):
        s = slice(cu[n], cu[n + 1])
        xs = {key: x[key][:, s] for key in ("q", "k", "v", "g", "beta")}
        xs["h0"], xs["cu_seqlens"] = x["h0"][n:n + 1], None
        one = run_gpu(gdr, xs, x["do"][:, s], x["dht"][n:n + 1], 64, True)
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            assert torch.equal(whole[name][:, s], one[name]), f"{name} of sequence {n}"
        assert torch.equal(whole["dh0"][n:n + 1], one["dh0"]), f"dh0 of sequence {n}"


def test_bwd_deterministic(gdr):
    w, x = wl.random_case(1, 300, 2, 4, 128, 128, dtype=torch.bfloat16, gate_per_k=False, seed=9, grads=True)
    a = run_gpu(gdr, x, x["do"], x["dht"], 64, True)
    b = run_gpu(gdr, x, x["do"], x["dht"], 64, True)
    for name in NAMES:
        assert torch.equal(a[name], b[name]), name


def test_bwd_rejects_bad_requests(gdr):
    w, x = wl.random_case(1, 64, 1, 1, 160, 32, dtype=torch.bfloat16, seed=1, grads=True)
    d = {n: dev(t) for n, t in x.items()}
    with pytest.raises(ValueError, match="K <= 128"):
        gdr.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["do"], h0=d["h0"])
    w, x = wl.random_case(1, 64, 1, 1, 64, 32, dtype=torch.bfloat16, seed=1, grads=True)
    d = {n: dev(t) for n, t in x.items()}
    with pytest.raises(ValueError, match="chunk_size must be either 32 or 64"):
        gdr.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["do"], h0=d["h0"], chunk_size=16)
