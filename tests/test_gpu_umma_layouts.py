"""The tcgen05 shared-memory layout and descriptor conventions of
``gdr_sm100.cuh``, checked one MMA chain at a time against torch.

Operand images are laid out on the host (128-byte swizzle, K-major or
MN-major) and copied verbatim into shared memory by ``tests/cuda/umma_probe.cu``;
D = A B^T is read back from tensor memory.  Every configuration the fused
kernel uses is covered: the stacked [K; Q] K^T product, MN-major A from a
token-major tile, the negated-A accumulate, and the N = 128 state update.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


class ProbeParams(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int), ("N", ctypes.c_int), ("a_mn", ctypes.c_int), ("b_mn", ctypes.c_int),
                ("neg_a", ctypes.c_int), ("nk", ctypes.c_int), ("a_lbo", ctypes.c_uint32),
                ("a_sbo", ctypes.c_uint32), ("b_lbo", ctypes.c_uint32), ("b_sbo", ctypes.c_uint32),
                ("a_step", ctypes.c_uint32 * 16), ("b_step", ctypes.c_uint32 * 16), ("a_bytes", ctypes.c_int),
                ("b_bytes", ctypes.c_int)]


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = tmp_path_factory.mktemp("probe") / "libumma_probe.so"
    src = os.path.join(HERE, "cuda", "umma_probe.cu")
    inc = os.path.join(ROOT, "chunked_gated_delta_08_gb300", "csrc")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", f"-I{inc}", "-o", str(out), src], check=True)
    lib = ctypes.CDLL(str(out))
    lib.umma_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ProbeParams), ctypes.c_void_p]
    lib.umma_probe.restype = ctypes.c_int
    return lib


def sw128_offset(row, col):
    chunk = (col >> 3) ^ (row & 7)
    return (row >> 3) * 1024 + (row & 7) * 128 + chunk * 16 + (col & 7) * 2


def sw128_image(X, sub_stride, nbytes, row_base=0, img=None):
    """Places X[rows, cols] (bf16) at rows row_base.. of 64-column sub-tiles."""
    rows, cols = X.shape
    if img is None:
        img = np.zeros(nbytes, dtype=np.uint8)
    bits = X.contiguous().view(torch.int16).numpy().astype(np.uint16)
    r = np.arange(rows)[:, None] + row_base
    c = np.arange(cols)[None, :]
    off = (c // 64) * sub_stride + sw128_offset(r, c % 64)
    img[off] = (bits & 0xFF).astype(np.uint8)
    img[off + 1] = (bits >> 8).astype(np.uint8)
    return img


def kmajor_steps(nk, sub_stride, base=0):
    return [base + ((16 * j) // 64) * sub_stride + ((16 * j) % 64) * 2 for j in range(nk)]


def mnmajor_steps(nk, base=0):
    return [base + 2048 * j for j in range(nk)]


def run(probe, M, N, kd, a_img, b_img, a_mn, b_mn, a_steps, b_steps, a_lbo, b_lbo, neg_a=0):
    p = ProbeParams()
    p.M, p.N, p.a_mn, p.b_mn, p.neg_a, p.nk = M, N, a_mn, b_mn, neg_a, kd // 16
    p.a_lbo, p.a_sbo, p.b_lbo, p.b_sbo = a_lbo, 1024, b_lbo, 1024
    for j, s in enumerate(a_steps):
        p.a_step[j] = s
    for j, s in enumerate(b_steps):
        p.b_step[j] = s
    p.a_bytes, p.b_bytes = len(a_img), len(b_img)
    d = np.zeros((M, N), dtype=np.float32)
    rc = probe.umma_probe(a_img.ctypes.data, b_img.ctypes.data, ctypes.byref(p), d.ctypes.data)
    assert rc == 0, f"probe returned {rc}"
    return d


def rand(*shape, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def check(d, ref):
    ref = ref.double().numpy()
    err = np.abs(d - ref).max() / (np.abs(ref).max() + 1e-30)
    assert err < 1e-5, f"max relative error {err:.2e}"


def test_stacked_kq_times_kt(probe):
    """D = [K; Q] K^T from the interleaved TMA tile layout (sub-tiles K0|Q0|K1|Q1)."""
    K, Q = rand(64, 128, seed=1), rand(64, 128, seed=2)
    img = sw128_image(K, 16384, 32768)
    sw128_image(Q, 16384, 32768, row_base=64, img=img)
    d = run(probe, 128, 64, 128, img, img.copy(), 0, 0, kmajor_steps(8, 16384), kmajor_steps(8, 16384),
            16, 16)
    check(d, torch.cat([K, Q]).double() @ K.double().T)


def test_mn_major_a_from_token_tile(probe):
    """D = K^T W'^T with A = K^T read MN-major from the [token][d] tile."""
    K, W = rand(64, 128, seed=3), rand(64, 64, seed=4)
    a_img = sw128_image(K, 16384, 32768)
    b_img = sw128_image(W, 8192, 8192)
    d = run(probe, 128, 64, 64, a_img, b_img, 1, 0, mnmajor_steps(4), kmajor_steps(4, 8192), 16384, 16)
    check(d, K.double().T @ W.double().T)


def test_negated_accumulate(probe):
    """D = -(h^T w^T) with A = h^T MN-major from h[d][v]; B = w K-major from w[i][d]."""
    h, w = rand(128, 128, seed=5), rand(64, 128, seed=6)
    a_img = sw128_image(h, 16384, 32768)
    b_img = sw128_image(w, 8192, 16384)
    d = run(probe, 128, 64, 128, a_img, b_img, 1, 0, mnmajor_steps(8), kmajor_steps(8, 8192), 16384, 16,
            neg_a=1)
    check(d, -(h.double().T @ w.double().T))


def test_state_update_n128(probe):
    """D = K^T vt with B = vt K-major from the [v][i] rows (N = 128)."""
    K, vt = rand(64, 128, seed=7), rand(128, 64, seed=8)
    a_img = sw128_image(K, 8192, 16384)
    b_img = sw128_image(vt, 16384, 16384)
    d = run(probe, 128, 128, 64, a_img, b_img, 1, 0, mnmajor_steps(4), kmajor_steps(4, 16384), 8192, 16)
    check(d, K.double().T @ vt.double().T)


def test_kmajor_both_k64(probe):
    """D = v_new^T P^T with both operands K-major (K = 64)."""
    vt, P = rand(128, 64, seed=9), rand(64, 64, seed=10)
    a_img = sw128_image(vt, 16384, 16384)
    b_img = sw128_image(P, 8192, 8192)
    d = run(probe, 128, 64, 64, a_img, b_img, 0, 0, kmajor_steps(4, 16384), kmajor_steps(4, 8192), 16, 16)
    check(d, vt.double() @ P.double().T)


def test_mn_major_b(probe):
    """B read MN-major (for completeness: B^T stored [k][n])."""
    A, B = rand(128, 64, seed=11), rand(64, 64, seed=12)
    a_img = sw128_image(A, 16384, 16384)
    b_img = sw128_image(B.T.contiguous(), 8192, 8192)
    d = run(probe, 128, 64, 64, a_img, b_img, 0, 1, kmajor_steps(4, 16384), mnmajor_steps(4), 16, 8192)
    check(d, A.double() @ B.double().T)
