"""Seeded synthetic workloads for the chunked gated delta rule forward.

This module only draws random inputs; it holds none of the method's arithmetic.
Both sides of every parity check (the CUDA library and the fp64 oracle) are fed
the same tensors produced here.

Recipe (the same for every workload): one ``torch.Generator`` seeded with the
workload's seed (0 unless stated), drawing on the CPU in fp32 in the order
q, k, v, g, beta, h0, do, dht; then rounding q, k, v, beta to the workload's
dtype.  g and h0 stay fp32.  Where the workload says "q, k L2-normalized", the
normalization (x / ||x||_2 per token and head, fp32) is applied before rounding
and the kernel's own L2 norm is off.  The gate is log-sigmoid of a standard
normal, divided by a per-workload factor; beta is sigmoid of a standard normal.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: torch.dtype
    B: int
    T: int
    H: int
    HV: int
    K: int
    V: int
    chunk_size: int = 64
    lengths: tuple | None = None      # varlen sequence lengths (B == 1)
    use_qk_l2norm: bool = False       # the kernel normalizes q, k
    prenorm_qk: bool = False          # inputs arrive already normalized
    gate_per_k: bool = False          # KDA gate [B,T,HV,K] instead of GDN [B,T,HV]
    gate_div: float = 1.0             # g = logsigmoid(N(0,1)) / gate_div
    h0_scale: float | None = None     # h0 = h0_scale * N(0,1); None -> no initial state
    seed: int = 0
    grads: bool = False               # also draw upstream do, dht

    @property
    def N(self) -> int:
        return len(self.lengths) if self.lengths else self.B

    @property
    def cu_seqlens(self):
        if not self.lengths:
            return None
        cu = [0]
        for n in self.lengths:
            cu.append(cu[-1] + n)
        return cu

    @property
    def tokens(self) -> int:
        return self.B * self.T


# The five workloads of the problem statement, in its order.
GDN_FP32_SMALL = Workload("gdn_fp32_T128_K64", torch.float32, B=1, T=128, H=1, HV=1, K=64, V=64,
                          prenorm_qk=True, gate_div=8.0, h0_scale=None)
GDN_BF16_GVA_K60 = Workload("gdn_bf16_gva_T512_K60", torch.bfloat16, B=2, T=512, H=2, HV=4, K=60, V=60,
                            use_qk_l2norm=True, h0_scale=0.1)
GDN_BF16_VARLEN = Workload("gdn_bf16_varlen_400_624_K128", torch.bfloat16, B=1, T=1024, H=16, HV=16,
                           K=128, V=128, lengths=(400, 624), prenorm_qk=True, h0_scale=0.1)
GDN_BF16_LARGE = Workload("gdn_bf16_B4_T32768_H32_K128", torch.bfloat16, B=4, T=32768, H=32, HV=32,
                          K=128, V=128, use_qk_l2norm=True, h0_scale=None)
KDA_BF16_VARLEN = Workload("kda_bf16_varlen_T16384_HV32_V256", torch.bfloat16, B=1, T=16384, H=16, HV=32,
                           K=128, V=256, lengths=(700, 324, 3072, 12288), use_qk_l2norm=True,
                           gate_per_k=True, gate_div=4.0, h0_scale=0.1, grads=True)

WORKLOADS = [GDN_FP32_SMALL, GDN_BF16_GVA_K60, GDN_BF16_VARLEN, GDN_BF16_LARGE, KDA_BF16_VARLEN]

# A quarter of the large dense workload (B = 1): the same per-unit work on 32
# blocks, with inputs (3 x 256 MB) still larger than L2.  Used for profiler
# captures, which replay a kernel many times.
GDN_BF16_PROFILE = Workload("gdn_bf16_B1_T32768_H32_K128", torch.bfloat16, B=1, T=32768, H=32, HV=32,
                            K=128, V=128, use_qk_l2norm=True, h0_scale=None)

# A decode step for the per-token form: 256 sequences, one new token each,
# state carried in h0 (read) and ht (written); not one of the five workloads.
GDN_BF16_DECODE = Workload("gdn_bf16_decode_N256_T1_H32_K128", torch.bfloat16, B=256, T=1, H=32, HV=32, K=128,
                           V=128, use_qk_l2norm=True, h0_scale=0.1)

# Few (sequence, head) units and a long sequence, fp32 (the chunked family):
# the case the intra-sequence split is for; not one of the five workloads.
GDN_FP32_LONG_FEW = Workload("gdn_fp32_B1_T32768_H4_K128", torch.float32, B=1, T=32768, H=4, HV=4, K=128, V=128,
                             use_qk_l2norm=True, h0_scale=0.1)

# A one-sequence cut of the KDA workload (8192 tokens) for per-kernel ncu
# counters of the backward without the full workload's scratch.
KDA_BF16_PROFILE = Workload("kda_bf16_T8192_HV32_V256", torch.bfloat16, B=1, T=8192, H=16, HV=32, K=128, V=256,
                            lengths=(8192,), use_qk_l2norm=True, gate_per_k=True, gate_div=4.0, h0_scale=0.1,
                            grads=True)

BY_NAME = {w.name: w for w in WORKLOADS + [GDN_BF16_PROFILE, GDN_BF16_DECODE, GDN_FP32_LONG_FEW, KDA_BF16_PROFILE]}


def make_inputs(w: Workload, device="cpu", seed: int | None = None) -> dict:
    """Draw the workload's inputs; returns a dict of tensors on ``device``."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    B, T, H, HV, K, V = w.B, w.T, w.H, w.HV, w.K, w.V

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32)

    q = randn(B, T, H, K)
    k = randn(B, T, H, K)
    if w.prenorm_qk:
        q = q / q.norm(dim=-1, keepdim=True)
        k = k / k.norm(dim=-1, keepdim=True)
    v = randn(B, T, HV, V)
    g = torch.nn.functional.logsigmoid(randn(*((B, T, HV, K) if w.gate_per_k else (B, T, HV)))) / w.gate_div
    beta = torch.sigmoid(randn(B, T, HV))
    h0 = None if w.h0_scale is None else w.h0_scale * randn(w.N, HV, K, V)
    out = {
        "q": q.to(w.dtype), "k": k.to(w.dtype), "v": v.to(w.dtype),
        "g": g.contiguous(), "beta": beta.to(w.dtype), "h0": h0,
        "cu_seqlens": None if w.lengths is None else torch.tensor(w.cu_seqlens, dtype=torch.int64),
    }
    if w.grads:
        out["do"] = randn(B, T, HV, V).to(w.dtype)
        out["dht"] = randn(w.N, HV, K, V)
    if device != "cpu":
        out = {key: (None if t is None else t.to(device)) for key, t in out.items()}
    return out


def make_grads(w: Workload, seed: int = 1, device="cpu") -> dict:
    """Upstream gradients do [B,T,HV,V] (input dtype) and dht [N,HV,K,V] (fp32),
    N(0,1), for a workload whose own recipe has none."""
    gen = torch.Generator().manual_seed(seed)
    do = torch.randn(w.B, w.T, w.HV, w.V, generator=gen).to(w.dtype)
    dht = torch.randn(w.N, w.HV, w.K, w.V, generator=gen)
    return {"do": do.to(device), "dht": dht.to(device)}


def random_case(B, T, H, HV, K, V, dtype=torch.float32, lengths=None, gate_per_k=False,
                use_h0=True, seed=0, gate_div=1.0, grads=False):
    """A small unit-test case of arbitrary shape with the same distributions."""
    w = Workload(f"case_{B}_{T}_{H}_{HV}_{K}_{V}", dtype, B, T, H, HV, K, V,
                 lengths=tuple(lengths) if lengths else None, gate_per_k=gate_per_k,
                 gate_div=gate_div, h0_scale=0.1 if use_h0 else None, seed=seed, grads=grads)
    return w, make_inputs(w)
