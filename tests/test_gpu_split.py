"""The intra-sequence split (GDR_ALGO_SPLIT), through the C ABI, against the
oracle: sequences cut into 1024-token segments, each segment's transition M
and zero-start end state S_ext, the merge S_in(s+1) = M_s S_in(s) + S_ext,s,
then the segments rescanned from their true entering states (the KCP
handbook's segment merge, on one GPU).  Tolerances as for the other forms.

Pages cited: the KCP handbook = "flash-linear-attention KCP 精度失效根因排查手册".
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


def run(gdr, x, l2, C=64, algo="split"):
    d = {n: dev(t) for n, t in x.items()}
    B, T, H, K = d["q"].shape
    HV, V = d["v"].shape[2:]
    N = B if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    o = torch.full((B, T, HV, V), float("nan"), dtype=d["q"].dtype, device="cuda")
    ht = torch.full((N, HV, K, V), float("nan"), device="cuda")
    o, ht = gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
                    chunk_size=C, use_qk_l2norm=l2, algo=algo, out=o, final_state=ht)
    assert gdr.device_status() == 0, gdr.last_error()
    return o, ht


def ref_of(x, l2):
    return oracle.gdr_fwd_ref(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], cu_seqlens=x["cu_seqlens"],
                              use_qk_l2norm=l2)


CASES = [
    # (per_k, C, lengths or None, B, T, H, HV, K, V, h0)
    (False, 64, None, 2, 3000, 1, 2, 64, 64, True),
    (True, 64, (1023, 1025, 0, 2048, 5), 1, 4101, 1, 2, 64, 48, True),
    (False, 32, (2100, 1), 1, 2101, 2, 2, 32, 80, False),
    (True, 32, None, 1, 1024, 1, 1, 128, 128, True),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"pk{int(c[0])}_C{c[1]}_T{c[4]}_K{c[7]}_V{c[8]}")
def test_split_parity(gdr, case, dtype):
    per_k, C, lengths, B, T, H, HV, K, V, h0 = case
    w, x = wl.random_case(B, T, H, HV, K, V, dtype=dtype, lengths=lengths, gate_per_k=per_k, use_h0=h0, seed=51,
                          gate_div=8.0 if per_k else 4.0)
    o, ht = run(gdr, x, True, C=C)
    ref = ref_of(x, True)
    eo, eh = rel_l2(o, ref["o"]), rel_l2(ht, ref["ht"])
    assert eo <= TOL[dtype] and eh <= TOL[dtype], f"o {eo:.2e} ht {eh:.2e}"


@pytest.mark.parametrize("w", [wl.GDN_BF16_VARLEN, wl.KDA_BF16_VARLEN], ids=lambda w: w.name)
def test_split_workloads(gdr, w):
    x = wl.make_inputs(w)
    o, ht = run(gdr, x, w.use_qk_l2norm)
    ref = ref_of(x, w.use_qk_l2norm)
    eo, eh = rel_l2(o, ref["o"]), rel_l2(ht, ref["ht"])
    assert eo <= 5e-3 and eh <= 5e-3, f"o {eo:.2e} ht {eh:.2e}"


def test_split_long_sequence_sampled_heads(gdr):
    """One 32768-token sequence, 4 heads: 32 segments per head; the oracle on every head."""
    w, x = wl.random_case(1, 32768, 4, 4, 128, 128, dtype=torch.bfloat16, seed=52)
    o, ht = run(gdr, x, True)
    ref = ref_of(x, True)
    eo, eh = rel_l2(o, ref["o"]), rel_l2(ht, ref["ht"])
    assert eo <= 5e-3 and eh <= 5e-3, f"o {eo:.2e} ht {eh:.2e}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("per_k", [False, True], ids=["gdn", "kda"])
@pytest.mark.parametrize("C", [32, 64])
def test_split_single_segment_is_bit_exact(gdr, dtype, per_k, C):
    """A uniform single sequence no longer than one 1024-token segment: there is
    nothing to merge (the segment starts from h0 itself), so the split must give
    exactly the bits of the unsplit chunked form (the KCP handbook, TL;DR step 4:
    a uniform single sequence is bit-perfect between the split and unsplit runs).
    Dense batches of such sequences and a varlen batch of short ones too."""
    for B, T, lengths in ((1, 1024, None), (1, 1000, None), (3, 700, None), (1, 1500, (1024, 5, 0, 471))):
        w, x = wl.random_case(B, T, 2, 4, 64, 48, dtype=dtype, lengths=lengths, gate_per_k=per_k, use_h0=True,
                              seed=55)
        o_s, ht_s = run(gdr, x, True, C=C, algo="split")
        o_c, ht_c = run(gdr, x, True, C=C, algo="chunked")
        assert torch.equal(o_s, o_c), f"B={B} T={T} lengths={lengths}: o differs"
        assert torch.equal(ht_s, ht_c), f"B={B} T={T} lengths={lengths}: ht differs"


def test_split_bad_cu_seqlens_touches_nothing(gdr):
    w, x = wl.random_case(1, 2000, 1, 1, 32, 32, dtype=torch.float32, lengths=(1500, 500), seed=53)
    d = {n: dev(t) for n, t in x.items()}
    cu = torch.tensor([0, 1600, 1500], dtype=torch.int64, device="cuda")
    o = torch.full((1, 2000, 1, 32), 7.0, device="cuda")
    ht = torch.full((2, 1, 32, 32), 7.0, device="cuda")
    gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], cu_seqlens=cu, algo="split", out=o,
            final_state=ht)
    assert gdr.device_status() == gdr.GDR_ERR_SEQLENS
    assert (o == 7.0).all() and (ht == 7.0).all()


def test_auto_takes_split_for_few_long_sequences(gdr):
    """fp32 (not the fused form's), one 8192-token sequence, 2 heads: AUTO = split."""
    w, x = wl.random_case(1, 8192, 1, 2, 64, 64, dtype=torch.float32, seed=54)
    o_a, ht_a = run(gdr, x, True, algo="auto")
    o_s, ht_s = run(gdr, x, True, algo="split")
    assert torch.equal(o_a, o_s) and torch.equal(ht_a, ht_s)
    ref = ref_of(x, True)
    assert rel_l2(o_a, ref["o"]) <= 1e-5 and rel_l2(ht_a, ref["ht"]) <= 1e-5
