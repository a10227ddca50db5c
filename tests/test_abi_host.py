"""libqk.so loads, exports what include/qk.h declares, and rejects bad
arguments on the host before touching a GPU (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

import block_scaled_precision_tcgen05_gb300 as qk
from block_scaled_precision_tcgen05_gb300 import build as qkbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qk.h")


@pytest.fixture(scope="module")
def lib():
    qkbuild.build()
    return qk.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qk_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(qk.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(8):
        s = lib.qk_status_string(code).decode()
        assert s.startswith("QK_")
    assert lib.qk_status_string(99).decode() == "QK_ERR_UNKNOWN"
    assert lib.qk_version() >= 100


FAKE = 0x100000  # 16-byte aligned fake device address; never dereferenced by these calls


def _p(v):
    return ctypes.c_void_p(v)


def int8_call(lib, A=FAKE, B=FAKE, sa=FAKE, sb=FAKE, bias=None, out=FAKE, M=128, N=128, K=128):
    return lib.qk_gemm_int8_rowwise(_p(A), _p(B), _p(sa), _p(sb), _p(bias) if bias else None, _p(out), M, N, K, None)


def mx_call(lib, fmt=1, A=FAKE, sA=FAKE, B=FAKE, sB=FAKE, bias=None, out=FAKE, M=128, N=128, K=128):
    return lib.qk_gemm_mx(fmt, _p(A), _p(sA), _p(B), _p(sB), _p(bias) if bias else None, _p(out), M, N, K, None)


def test_int8_argument_errors(lib):
    assert int8_call(lib, A=0) == qk.QK_ERR_ARG
    assert int8_call(lib, sb=0) == qk.QK_ERR_ARG
    assert int8_call(lib, out=0) == qk.QK_ERR_ARG
    assert int8_call(lib, M=-1) == qk.QK_ERR_ARG
    assert int8_call(lib, K=0) == qk.QK_ERR_ARG
    assert int8_call(lib, A=FAKE + 8) == qk.QK_ERR_ALIGN
    assert int8_call(lib, bias=FAKE + 2) == qk.QK_ERR_ALIGN
    assert int8_call(lib, N=100) == qk.QK_ERR_ALIGN
    assert int8_call(lib, K=24) == qk.QK_ERR_ALIGN
    assert int8_call(lib, K=131072) == qk.QK_ERR_RANGE   # int32 accumulator could overflow
    assert int8_call(lib, M=2 ** 31) == qk.QK_ERR_RANGE
    # empty products launch nothing and succeed, even with null pointers
    assert int8_call(lib, M=0, A=0, out=0) == qk.QK_OK
    assert int8_call(lib, N=0) == qk.QK_OK


def test_int8_out_type_argument_errors(lib):
    def call(out_type=qk.QK_OUT_FP32, **kw):
        return lib.qk_gemm_int8_rowwise_out(_p(kw.get("A", FAKE)), _p(FAKE), _p(FAKE), _p(FAKE), None,
                                            _p(kw.get("out", FAKE)), out_type, kw.get("M", 128), kw.get("N", 128),
                                            kw.get("K", 128), None)
    for bad in (-1, 3, 99):
        assert call(out_type=bad) == qk.QK_ERR_ARG       # checked before anything else
        assert call(out_type=bad, M=0) == qk.QK_ERR_ARG
    for ot in (qk.QK_OUT_BF16, qk.QK_OUT_FP16, qk.QK_OUT_FP32):
        assert call(out_type=ot, A=0) == qk.QK_ERR_ARG
        assert call(out_type=ot, out=0) == qk.QK_ERR_ARG
        assert call(out_type=ot, out=FAKE + 8) == qk.QK_ERR_ALIGN
        assert call(out_type=ot, N=100) == qk.QK_ERR_ALIGN
        assert call(out_type=ot, K=131072) == qk.QK_ERR_RANGE
        assert call(out_type=ot, M=0, A=0, out=0) == qk.QK_OK   # empty product: nothing launched


def test_fp8_out_type_argument_errors(lib):
    def call(out_type=qk.QK_OUT_FP32, **kw):
        return lib.qk_gemm_fp8_rowwise_out(_p(kw.get("A", FAKE)), _p(FAKE), _p(FAKE), _p(FAKE), None,
                                           _p(kw.get("out", FAKE)), out_type, kw.get("M", 128), kw.get("N", 128),
                                           kw.get("K", 128), None)
    for bad in (-1, 3, 99):
        assert call(out_type=bad) == qk.QK_ERR_ARG       # checked before anything else
        assert call(out_type=bad, M=0) == qk.QK_ERR_ARG
    for ot in (qk.QK_OUT_BF16, qk.QK_OUT_FP16, qk.QK_OUT_FP32):
        assert call(out_type=ot, A=0) == qk.QK_ERR_ARG
        assert call(out_type=ot, out=0) == qk.QK_ERR_ARG
        assert call(out_type=ot, out=FAKE + 8) == qk.QK_ERR_ALIGN
        assert call(out_type=ot, N=100) == qk.QK_ERR_ALIGN
        assert call(out_type=ot, K=40) == qk.QK_ERR_ALIGN
        assert call(out_type=ot, M=0, A=0, out=0) == qk.QK_OK   # empty product: nothing launched


@pytest.mark.parametrize("entry", ["mx", "nvfp4"])
def test_block_scaled_out_type_argument_errors(lib, entry):
    def call(out_type=qk.QK_OUT_FP32, **kw):
        A, out = _p(kw.get("A", FAKE)), _p(kw.get("out", FAKE))
        M, N, K = kw.get("M", 128), kw.get("N", 128), kw.get("K", 128)
        if entry == "mx":
            return lib.qk_gemm_mx_out(kw.get("fmt", qk.FMT_MXFP8_E4M3), A, _p(FAKE), _p(FAKE), _p(FAKE), None, out,
                                      out_type, M, N, K, None)
        return lib.qk_gemm_nvfp4_out(A, _p(FAKE), _p(FAKE), _p(FAKE), None, None, None, out, out_type, M, N, K,
                                     None)
    for bad in (-1, 3, 99):
        assert call(out_type=bad) == qk.QK_ERR_ARG       # checked before anything else
        assert call(out_type=bad, M=0) == qk.QK_ERR_ARG
    for ot in (qk.QK_OUT_BF16, qk.QK_OUT_FP16, qk.QK_OUT_FP32):
        assert call(out_type=ot, A=0) == qk.QK_ERR_ARG
        assert call(out_type=ot, out=0) == qk.QK_ERR_ARG
        assert call(out_type=ot, out=FAKE + 8) == qk.QK_ERR_ALIGN
        assert call(out_type=ot, N=100) == qk.QK_ERR_ALIGN
        assert call(out_type=ot, K=48) == qk.QK_ERR_ALIGN
        assert call(out_type=ot, M=0, A=0, out=0) == qk.QK_OK   # empty product: nothing launched
        if entry == "mx":
            assert call(out_type=ot, fmt=7) == qk.QK_ERR_ARG


def test_fp8_argument_errors(lib):
    call = lambda **kw: lib.qk_gemm_fp8_rowwise(_p(FAKE), _p(kw.get("B", FAKE)), _p(FAKE), _p(FAKE), None,
                                                _p(FAKE), kw.get("M", 64), kw.get("N", 64), kw.get("K", 64), None)
    assert call(B=0) == qk.QK_ERR_ARG
    assert call(N=12) == qk.QK_ERR_ALIGN
    assert call(K=40) == qk.QK_ERR_ALIGN
    assert call(M=0) == qk.QK_OK


def test_mx_argument_errors(lib):
    assert mx_call(lib, fmt=0) == qk.QK_ERR_ARG
    assert mx_call(lib, fmt=3) == qk.QK_ERR_ARG
    assert mx_call(lib, sA=0) == qk.QK_ERR_ARG
    assert mx_call(lib, K=48) == qk.QK_ERR_ALIGN       # not a multiple of 32
    assert mx_call(lib, N=20) == qk.QK_ERR_ALIGN
    assert mx_call(lib, sB=FAKE + 2) == qk.QK_ERR_ALIGN
    assert mx_call(lib, out=FAKE + 4) == qk.QK_ERR_ALIGN
    assert mx_call(lib, K=-32) == qk.QK_ERR_ARG
    assert mx_call(lib, M=0) == qk.QK_OK


def test_mx_b32_argument_errors(lib):
    def call(fmt=1, sA=FAKE, sB32=FAKE, out=FAKE, M=128, N=128, K=128):
        return lib.qk_gemm_mx_b32(fmt, _p(FAKE), _p(sA), _p(FAKE), _p(sB32), None, _p(out), M, N, K, None)
    assert call(fmt=0) == qk.QK_ERR_ARG
    assert call(fmt=3) == qk.QK_ERR_ARG
    assert call(sB32=0) == qk.QK_ERR_ARG
    assert call(sA=0) == qk.QK_ERR_ARG
    assert call(K=48) == qk.QK_ERR_ALIGN
    assert call(N=20) == qk.QK_ERR_ALIGN
    assert call(sB32=FAKE + 2) == qk.QK_ERR_ALIGN
    assert call(out=FAKE + 4) == qk.QK_ERR_ALIGN
    assert call(K=-32) == qk.QK_ERR_ARG
    assert call(M=0) == qk.QK_OK
    assert call(N=0, sB32=0) == qk.QK_OK


def test_binding_fails_loudly_without_library(tmp_path):
    missing = str(tmp_path / "libqk.so")
    with pytest.raises(OSError):
        qk.load_library(missing)
