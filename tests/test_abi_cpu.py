"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol the header declares, and rejects bad requests before launching."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "gdr.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|int64_t|const char \*)\s*(gdr_\w+)\s*\(", src, re.M)))


def test_header_and_exports_agree(gdr):
    names = declared_symbols()
    assert "gdr_fwd" in names and len(names) >= 9
    lib = ctypes.CDLL(gdr.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in gdr.h but not exported"
    assert sorted(gdr.EXPORTED) == names


def test_version(gdr):
    assert gdr.version() >= 100


def _desc(gdr, **kw):
    base = dict(B=1, T=64, H=1, HV=1, K=64, V=64, N=1, dtype=gdr.GDR_BF16, gate=gdr.GDR_GATE_SCALAR, algo=0,
                flags=0)
    base.update(kw)
    return gdr.GdrDesc(**base)


def _call(gdr, desc, chunk_size=64, cu=None):
    lib = gdr.lib()
    return lib.gdr_fwd(ctypes.byref(desc), None, None, None, None, None, None, cu, chunk_size, 0, None, None, None)


@pytest.mark.parametrize("cs", [16, 0, 48, 128, -64])
def test_invalid_chunk_size(gdr, cs):
    assert _call(gdr, _desc(gdr), cs) == gdr.GDR_ERR_CHUNK_SIZE
    assert gdr.last_error() == "chunk_size must be either 32 or 64"


@pytest.mark.parametrize("kw,code", [
    (dict(H=3, HV=4), -2), (dict(K=300), -2), (dict(V=0), -2), (dict(T=-1), -2), (dict(N=2), -2),
    (dict(dtype=7), -3), (dict(gate=5), -3), (dict(algo=9), -3), (dict(flags=2), -3),
])
def test_invalid_shapes(gdr, kw, code):
    assert _call(gdr, _desc(gdr, **kw)) == code
    assert gdr.last_error()


def test_varlen_requires_b1(gdr):
    cu = ctypes.c_void_p(8)  # never dereferenced: rejected on the host first
    assert _call(gdr, _desc(gdr, B=2, N=1), cu=cu) == gdr.GDR_ERR_SHAPE


def test_null_pointers_rejected(gdr):
    assert _call(gdr, _desc(gdr)) == gdr.GDR_ERR_NULLPTR


def test_python_errors_map_to_valueerror(gdr):
    with pytest.raises(ValueError, match="chunk_size must be either 32 or 64"):
        gdr._check(_call(gdr, _desc(gdr), 16))


def test_chunked_sizes(gdr):
    d = _desc(gdr, B=2, T=100, HV=4, H=2, K=60, V=60, N=2)
    s = gdr.chunked_sizes(d, 64, False)
    assert s.nt_max == 4 and s.h_bytes == 4 * 4 * 60 * 60 * 4
    dv = _desc(gdr, B=1, T=1024, N=2)
    sv = gdr.chunked_sizes(dv, 64, True)
    assert sv.nt_max >= 17  # lengths [400, 624] need 7 + 10 chunks


def test_int64_offsets_of_the_large_dense_workload():
    """Byte offsets of the largest tensors exceed 2^31 (int64 addressing needed)."""
    B, T, H, HV, K, V, C = 4, 32768, 32, 32, 128, 128, 64
    assert B * T * H * K * 2 == 2 ** 30
    NT = B * T // C
    assert NT * HV * K * V * 4 >= 2 ** 32
