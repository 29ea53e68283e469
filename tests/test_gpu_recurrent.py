"""The per-token (recurrent) form of the forward, through the C ABI, against
the oracle; and the decode use it serves (T = 1 steps, state carried in
place).  Tolerances as for the other forms: relative L2 error <= 1e-5 (fp32
inputs) and <= 5e-3 (bf16) on o and ht.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 5e-3}


def rel_l2(got, want):
    got = got.detach().double().cpu().numpy()
    want = np.asarray(want, np.float64)
    assert np.isfinite(got).all(), "non-finite values in the CUDA output"
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def dev(x):
    return None if x is None else x.cuda()


def run(gdr, x, l2, algo="recurrent"):
    d = {n: dev(t) for n, t in x.items()}
    B, T, H, K = d["q"].shape
    HV, V = d["v"].shape[2:]
    o = torch.full((B, T, HV, V), float("nan"), dtype=d["q"].dtype, device="cuda")
    o, ht = gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
                    use_qk_l2norm=l2, algo=algo, out=o)
    assert gdr.device_status() == 0, gdr.last_error()
    return o, ht


def ref_of(x, l2):
    return oracle.gdr_fwd_ref(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], cu_seqlens=x["cu_seqlens"],
                              use_qk_l2norm=l2)


CASES = [
    # (per_k, l2, lengths, B, T, H, HV, K, V, h0)
    (False, True, None, 2, 33, 2, 4, 60, 60, True),
    (True, True, None, 1, 40, 1, 2, 128, 256, True),
    (False, False, (5, 0, 17, 1), 1, 23, 2, 2, 256, 32, False),
    (True, True, (9, 30), 1, 39, 2, 2, 100, 72, True),
    (False, True, None, 3, 1, 1, 1, 16, 8, True),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"pk{int(c[0])}_l2{int(c[1])}_K{c[7]}_V{c[8]}")
def test_recurrent_parity(gdr, case, dtype):
    per_k, l2, lengths, B, T, H, HV, K, V, h0 = case
    w, x = wl.random_case(B, T, H, HV, K, V, dtype=dtype, lengths=lengths, gate_per_k=per_k, use_h0=h0, seed=21,
                          gate_div=4.0 if per_k else 1.0)
    if not l2:  # unit-norm q, k keep the state bounded without the in-kernel norm
        for n in ("q", "k"):
            x[n] = (x[n].float() / x[n].float().norm(dim=-1, keepdim=True)).to(dtype)
    o, ht = run(gdr, x, l2)
    ref = ref_of(x, l2)
    eo, eh = rel_l2(o, ref["o"]), rel_l2(ht, ref["ht"])
    assert eo <= TOL[dtype] and eh <= TOL[dtype], f"o {eo:.2e} ht {eh:.2e}"


def test_recurrent_varlen_workload(gdr):
    w = wl.GDN_BF16_VARLEN
    x = wl.make_inputs(w)
    o, ht = run(gdr, x, w.use_qk_l2norm)
    ref = ref_of(x, w.use_qk_l2norm)
    assert rel_l2(o, ref["o"]) <= 5e-3 and rel_l2(ht, ref["ht"]) <= 5e-3


def test_decode_workload_step(gdr):
    """One decode step (256 sequences x 1 token) equals the oracle; in place
    (ht aliasing h0) gives the same bits as a separate ht."""
    w = wl.GDN_BF16_DECODE
    x = wl.make_inputs(w)
    o, ht = run(gdr, x, True)
    ref = ref_of(x, True)
    assert rel_l2(o, ref["o"]) <= 5e-3 and rel_l2(ht, ref["ht"]) <= 5e-3
    d = {n: dev(t) for n, t in x.items()}
    state = d["h0"].clone()
    o2, ht2 = gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=state, use_qk_l2norm=True, algo="recurrent",
                      final_state=state)
    assert gdr.device_status() == 0
    assert ht2.data_ptr() == state.data_ptr()
    assert torch.equal(o2, o) and torch.equal(state, ht)


def test_decode_steps_equal_one_call(gdr):
    """Twelve in-place decode steps equal the oracle on the whole sequence."""
    w, x = wl.random_case(4, 12, 2, 4, 128, 64, dtype=torch.bfloat16, seed=22)
    d = {n: dev(t) for n, t in x.items()}
    state = d["h0"].clone()
    outs = []
    for t in range(12):
        sl = slice(t, t + 1)
        o, _ = gdr.fwd(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(), d["v"][:, sl].contiguous(),
                       d["g"][:, sl].contiguous(), d["beta"][:, sl].contiguous(), h0=state, use_qk_l2norm=True,
                       algo="recurrent", final_state=state)
        outs.append(o)
    assert gdr.device_status() == 0
    ref = ref_of(x, True)
    assert rel_l2(torch.cat(outs, 1), ref["o"]) <= 5e-3
    assert rel_l2(state, ref["ht"]) <= 5e-3


def test_auto_picks_recurrent_for_short_dense(gdr):
    w, x = wl.random_case(2, 16, 1, 2, 64, 64, dtype=torch.bfloat16, seed=23)
    n0 = gdr.launch_count()
    o_auto, ht_auto = run(gdr, x, True, algo="auto")
    assert gdr.launch_count() - n0 == 1
    o_rec, ht_rec = run(gdr, x, True, algo="recurrent")
    assert torch.equal(o_auto, o_rec) and torch.equal(ht_auto, ht_rec)


def test_recurrent_bad_cu_seqlens_touches_nothing(gdr):
    w, x = wl.random_case(1, 20, 1, 1, 32, 32, dtype=torch.float32, lengths=(12, 8), seed=24)
    d = {n: dev(t) for n, t in x.items()}
    d["cu_seqlens"] = torch.tensor([0, 15, 12], dtype=torch.int64, device="cuda")  # decreasing, ends short of T
    o = torch.full((1, 20, 1, 32), 7.0, device="cuda")
    ht = torch.full((2, 1, 32, 32), 7.0, device="cuda")
    gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], cu_seqlens=d["cu_seqlens"], algo="recurrent",
            out=o, final_state=ht)
    assert gdr.device_status() == gdr.GDR_ERR_SEQLENS
    assert (o == 7.0).all() and (ht == 7.0).all()
