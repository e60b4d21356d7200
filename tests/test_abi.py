"""Host-side tests of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before launching anything (so these
run without a GPU: no call here reaches a kernel launch)."""

import ctypes
import os
import re

import pytest

import int8_qmv_qmm_gb300 as q
from int8_qmv_qmm_gb300 import build_lib

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADERS = sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h"))
OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return q.lib()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qlin_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("qlin_quantize_affine", "qlin_dequant", "qlin_qmv", "qlin_qmm", "qlin_linear"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    assert L.qlin_status_str(0) == b"QLIN_OK"
    assert L.qlin_status_str(3) == b"QLIN_ERR_MISALIGNED"
    assert L.qlin_version() >= 100


FAKE = 0x10000  # 16-byte aligned fake device address; never dereferenced here


def _qmv(L, fn="qlin_qmv", x=FAKE, wq=FAKE, s=FAKE, b=FAKE, y=FAKE, M=1, N=300, K=512, bits=4,
         g=64, dt=q.QLIN_F16):
    return getattr(L, fn)(ctypes.c_void_p(x), ctypes.c_void_p(wq), ctypes.c_void_p(s),
                          ctypes.c_void_p(b), ctypes.c_void_p(y), M, N, K, bits, g, dt, None)


@pytest.mark.parametrize("fn", ["qlin_qmv", "qlin_qmm", "qlin_linear"])
def test_matmul_argument_validation(L, fn):
    assert _qmv(L, fn, bits=3) == UNSUPPORTED
    assert _qmv(L, fn, bits=2) == UNSUPPORTED
    assert _qmv(L, fn, g=32) == UNSUPPORTED
    assert _qmv(L, fn, g=128) == UNSUPPORTED
    assert _qmv(L, fn, dt=q.QLIN_F32) == UNSUPPORTED
    assert _qmv(L, fn, K=100) == INVALID
    assert _qmv(L, fn, K=0) == INVALID
    assert _qmv(L, fn, K=-64) == INVALID
    assert _qmv(L, fn, M=-1) == INVALID
    assert _qmv(L, fn, N=-1) == INVALID
    assert _qmv(L, fn, x=0) == INVALID
    assert _qmv(L, fn, y=0) == INVALID
    assert _qmv(L, fn, x=FAKE + 8) == MISALIGNED
    assert _qmv(L, fn, wq=FAKE + 4) == MISALIGNED
    assert _qmv(L, fn, y=FAKE + 1) == MISALIGNED
    # empty products launch nothing and succeed, even with null pointers
    assert _qmv(L, fn, M=0, x=0, y=0) == OK
    assert _qmv(L, fn, N=0, wq=0, s=0, b=0, y=0) == OK


def test_error_detail_is_recorded(L):
    assert _qmv(L, bits=5) == UNSUPPORTED
    assert b"bits=5" in L.qlin_last_error()


def test_quantize_and_dequant_validation(L):
    vp = ctypes.c_void_p
    assert L.qlin_quantize_affine(vp(FAKE), 4, 128, 4, 64, q.QLIN_F32, vp(FAKE), vp(FAKE),
                                  vp(FAKE), None) == UNSUPPORTED
    assert L.qlin_quantize_affine(vp(FAKE), 4, 100, 4, 64, q.QLIN_F16, vp(FAKE), vp(FAKE),
                                  vp(FAKE), None) == INVALID
    assert L.qlin_quantize_affine(vp(FAKE + 4), 4, 128, 4, 64, q.QLIN_F16, vp(FAKE), vp(FAKE),
                                  vp(FAKE), None) == MISALIGNED
    assert L.qlin_quantize_affine(vp(0), 0, 128, 4, 64, q.QLIN_F16, vp(0), vp(0), vp(0),
                                  None) == OK
    # dequant: output dtype must be f32 or the scale dtype
    assert L.qlin_dequant(vp(FAKE), vp(FAKE), vp(FAKE), 4, 128, 4, 64, q.QLIN_F16, q.QLIN_BF16,
                          vp(FAKE), None) == UNSUPPORTED
    assert L.qlin_dequant(vp(FAKE), vp(FAKE), vp(FAKE), 4, 128, 8, 64, q.QLIN_BF16, q.QLIN_F32,
                          vp(FAKE + 8), None) == MISALIGNED
    assert L.qlin_dequant(vp(0), vp(FAKE), vp(FAKE), 4, 128, 8, 64, q.QLIN_BF16, q.QLIN_F32,
                          vp(FAKE), None) == INVALID


def test_linear_ex_validation(L):
    vp = ctypes.c_void_p

    def call(y_dt=q.QLIN_F32, lb=FAKE, y=FAKE, dt=q.QLIN_F16, M=1):
        return L.qlin_linear_ex(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(lb), vp(y), M, 300,
                                512, 4, 64, dt, y_dt, None)

    # the output is float32 or the activation dtype
    assert call(y_dt=q.QLIN_BF16) == UNSUPPORTED
    assert call(y_dt=q.QLIN_F16, dt=q.QLIN_BF16) == UNSUPPORTED
    # a float32 y needs 4-byte alignment, the layer bias 2-byte alignment
    assert call(y=FAKE + 2) == MISALIGNED
    assert call(lb=FAKE + 1) == MISALIGNED
    assert call(M=600, lb=FAKE + 1) == MISALIGNED
    # the format checks still come first
    assert L.qlin_linear_ex(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 1, 300, 512,
                            3, 64, q.QLIN_F16, q.QLIN_F32, None) == UNSUPPORTED
    # empty product: nothing launched
    assert call(M=0) == OK


def test_device_status_rejects_null(L):
    assert L.qlin_device_status(None) == INVALID


def test_crossover_env_override(L):
    """QLIN_CROSSOVER_M is read once per process (on the first call), so the
    override is checked in a fresh process."""
    import subprocess
    import sys
    assert L.qlin_crossover_m(8192, 2048, 4) >= 1
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import int8_qmv_qmm_gb300 as q; "
            "print(q.lib().qlin_crossover_m(8192, 2048, 4))")
    out = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                         env=dict(os.environ, QLIN_CROSSOVER_M="7"), timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip().splitlines()[-1] == "7"


def test_testing_chain_entry_validation(L):
    """The test-only stalled-chain entry point refuses bad requests on the host."""
    vp = ctypes.c_void_p
    links = (q.Link * 2)()
    links[0] = q.Link(FAKE, FAKE, FAKE, FAKE, 64, 512, -1, 0)
    links[1] = q.Link(FAKE, FAKE, FAKE, FAKE, 64, 64, 0, 0)

    def call(stalled, limit_us, n=2):
        return L.qlin_testing_qmv_chain_stalled(vp(FAKE), links, n, 4, 64, q.QLIN_F16, vp(FAKE),
                                                256, stalled, limit_us, None)

    assert call(-1, 1000) == INVALID      # out of range
    assert call(2, 1000) == INVALID
    assert call(1, 1000) == INVALID       # nothing reads the last link
    assert call(0, 0) == INVALID          # limit out of range
    assert call(0, 3000000) == INVALID


def test_crossover_by_shape_and_dtype(L):
    """The measured switch: qmm from M = 5 on the larger matrices (from M = 4
    for f16 with K > N), from M = 9 on small ones, whatever the bit width."""
    f16, bf16 = q.QLIN_F16, q.QLIN_BF16
    for bits in (4, 8):
        assert L.qlin_crossover_m_dtype(2048, 8192, bits, f16) == 4
        assert L.qlin_crossover_m_dtype(2048, 8192, bits, bf16) == 5
        assert L.qlin_crossover_m_dtype(8192, 2048, bits, bf16) == 5
        assert L.qlin_crossover_m_dtype(8192, 2048, bits, f16) == 5
        assert L.qlin_crossover_m_dtype(3072, 2048, bits, f16) == 5
        assert L.qlin_crossover_m_dtype(2048, 2048, bits, f16) == 9
        assert L.qlin_crossover_m_dtype(2048, 2048, bits, bf16) == 9
        assert L.qlin_crossover_m_dtype(300, 512, bits, bf16) == 9
    assert L.qlin_crossover_m(2048, 8192, 4) == L.qlin_crossover_m_dtype(2048, 8192, 4, f16)


def test_qmv_split_choice(L, monkeypatch):
    """qmv splits K over a cluster only for few, long row blocks (at least
    32 KB of packed weights each), by the largest factor whose CTAs fit on the
    SMs two at a time with at least 4 KB of the block each."""
    monkeypatch.delenv("QLIN_QMV_SPLIT", raising=False)
    monkeypatch.delenv("QLIN_QMV_R", raising=False)
    f = L.qlin_testing_qmv_split
    assert f(300, 512, 4, 152) == 1          # 2 KB blocks: a split does not pay
    assert f(1029, 2048, 8, 152) == 1        # 16 KB blocks
    assert f(129, 8192, 4, 152) == 8         # 17 blocks of 32 KB
    assert f(37, 16384, 8, 152) == 8
    assert f(513, 8192, 8, 152) == 4         # 65 blocks: 8 would not fit at once
    assert f(1000, 4096, 8, 152) == 2        # 125 blocks
    assert f(2048, 8192, 8, 152) == 1        # 256 blocks already fill the SMs
    assert f(129, 8192, 4, 16) == 1          # 17 blocks on 16 SMs
    assert f(129, 8192, 4, 40) == 4
    # invalid arguments
    assert f(0, 512, 4, 152) == -1
    assert f(300, 100, 4, 152) == -1
    assert f(300, 512, 3, 152) == -1
    assert f(300, 512, 4, 0) == -1
    # the tuning override, where each CTA's share stays whole 16-byte chunks
    monkeypatch.setenv("QLIN_QMV_SPLIT", "4")
    assert f(300, 512, 4, 152) == 4          # 256-byte rows: 64 bytes a CTA
    assert f(3, 192, 4, 152) == 1            # 96-byte rows do not split in 4


def test_qmv_rejects_k_beyond_the_staged_x(L, monkeypatch):
    """qmv keeps x in shared memory as f32: a K whose x cannot fit beside the
    ring is refused on the host (no launch), unless a split of K leaves each
    CTA a slice that fits."""
    monkeypatch.setenv("QLIN_QMV_SPLIT", "1")
    assert _qmv(L, N=300, K=1 << 17, bits=8) == UNSUPPORTED
    assert b"too large" in L.qlin_last_error()
    assert _qmv(L, M=4, N=300, K=1 << 15, bits=8) == UNSUPPORTED
