"""The C ABI: the library loads, exports every symbol include/gemm.h declares,
and its host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

import dense_gemm_03_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_\w+|sgemm_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from dense_gemm_03_gb300 import build
    build.build()
    return g.lib()


def test_header_and_binding_agree():
    assert _declared() == sorted(g.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_no_torch_in_header():
    text = open(HEADER).read()
    assert "torch" not in text.lower() and "at::" not in text


def test_error_codes_without_gpu(L):
    # argument checks run before any CUDA call
    assert L.gemm_f16(None, None, None, -1, 4, 4, 1.0, 0.0, None) == -2
    assert L.gemm_f16_ld(None, None, None, 4, 4, 4, 3, 4, 4, 1.0, 0.0, None) == -3   # lda < K
    assert L.gemm_f16_ld(None, None, None, 4, 4, 4, 4, 3, 4, 1.0, 0.0, None) == -3   # ldb < N
    assert L.gemm_f16_ld(None, None, None, 4, 4, 4, 4, 4, 3, 1.0, 0.0, None) == -3   # ldc < N
    assert L.gemm_f16(None, None, None, 4, 4, 4, 1.0, 0.0, None) == -1               # null C
    assert L.gemm_f16(None, None, 8, 4, 4, 4, 1.0, 0.0, None) == -1                  # null A, B
    assert L.sgemm_f32(None, None, None, 4, -4, 4, 1.0, 0.0, None) == -2
    assert L.sgemm_f32_ld(None, None, None, 4, 4, 4, 4, 4, 2, 1.0, 0.0, None) == -3
    # empty outputs are a successful no-op, even with null pointers
    assert L.gemm_f16(None, None, None, 0, 4, 4, 1.0, 0.0, None) == 0
    assert L.sgemm_f32(None, None, None, 4, 0, 4, 1.0, 0.0, None) == 0
    assert L.gemm_f16_host(None, None, None, 0, 0, 0, 0, 0, 0, 1.0, 0.0, None) == 0


def test_strerror_and_switches(L):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert L.gemm_strerror(code)
    assert g.force_path(3) == 0
    assert g.force_path(0) == 3
    with pytest.raises(g.GemmError):
        g.force_path(18)
    assert g.force_splits(4) == 0 and g.force_splits(0) == 4
    assert g.stage_kblocks(2) == 0 and g.stage_kblocks(0) == 2
    with pytest.raises(g.GemmError):
        g.stage_kblocks(3)
    prev = g.set_wait_limit_ns(12345)
    assert g.set_wait_limit_ns(prev) == 12345
