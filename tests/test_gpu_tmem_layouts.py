"""Tensor-memory conventions of ``gdr_sm100.cuh`` beyond the shared-memory
operands (those are covered by ``test_gpu_umma_layouts.py``), checked against
torch and against tags on a one-CTA probe (``tests/cuda/tmem_probe.cu``):

* an MMA whose A operand sits in tensor memory (lane m = row m, two bf16 per
  32-bit column, the lower half holding the even K index, 8 columns per K step);
* the register layout of a ``tcgen05.ld.16x256b.x2`` load: thread t holds
  lanes base + t/4 and base + 8 + t/4, columns 2 (t % 4) and 2 (t % 4) + 1 of
  each group of 8, the second group in registers 4-7.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

from tests.test_gpu_umma_layouts import kmajor_steps, rand, sw128_image

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


class TaParams(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("nk", ctypes.c_int), ("b_lbo", ctypes.c_uint32), ("b_sbo", ctypes.c_uint32),
                ("b_step", ctypes.c_uint32 * 16), ("b_bytes", ctypes.c_int)]


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = tmp_path_factory.mktemp("tprobe") / "libtmem_probe.so"
    src = os.path.join(HERE, "cuda", "tmem_probe.cu")
    inc = os.path.join(ROOT, "chunked_gated_delta_08_gb300", "csrc")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", f"-I{inc}", "-o", str(out), src], check=True)
    lib = ctypes.CDLL(str(out))
    lib.tmem_a_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(TaParams), ctypes.c_void_p]
    lib.tmem_a_probe.restype = ctypes.c_int
    lib.ld16_probe.argtypes = [ctypes.c_void_p]
    lib.ld16_probe.restype = ctypes.c_int
    return lib


def tmem_words(A):
    """[128, Kd] bf16 -> [128, Kd/2] 32-bit words, even K index in the lower half."""
    bits = A.contiguous().view(torch.int16).numpy().astype(np.uint16).astype(np.uint32)
    return np.ascontiguousarray(bits[:, 0::2] | (bits[:, 1::2] << 16))


@pytest.mark.parametrize("N,Kd", [(64, 64), (128, 64), (64, 128)])
def test_a_operand_in_tensor_memory(probe, N, Kd):
    A, B = rand(128, Kd, seed=21), rand(N, Kd, seed=22)
    words = tmem_words(A)
    b_img = sw128_image(B, N * 128, (Kd // 64) * N * 128)
    p = TaParams()
    p.N, p.nk, p.b_lbo, p.b_sbo = N, Kd // 16, 16, 1024
    for j, s in enumerate(kmajor_steps(Kd // 16, N * 128)):
        p.b_step[j] = s
    p.b_bytes = len(b_img)
    d = np.zeros((128, N), dtype=np.float32)
    rc = probe.tmem_a_probe(words.ctypes.data, b_img.ctypes.data, ctypes.byref(p), d.ctypes.data)
    assert rc == 0, f"probe returned {rc}"
    ref = (A.double() @ B.double().T).numpy()
    err = np.abs(d - ref).max() / np.abs(ref).max()
    assert err < 1e-5, f"max relative error {err:.2e}"


def test_ld_16x256b_register_layout(probe):
    out = np.zeros((4, 2, 32, 8), dtype=np.float32)
    assert probe.ld16_probe(out.ctypes.data) == 0
    for w in range(4):
        for h in range(2):
            base = 32 * w + 16 * h
            for t in range(32):
                want = []
                for grp in range(2):
                    c = 8 * grp + 2 * (t % 4)
                    want += [(base + t // 4, c), (base + t // 4, c + 1), (base + 8 + t // 4, c),
                             (base + 8 + t // 4, c + 1)]
                got = [(int(v) // 1000, int(v) % 1000) for v in out[w, h, t]]
                assert got == want, f"warp {w} half {h} thread {t}: {got} != {want}"
