"""CPU oracle for the quantized GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package.  The product path
(``block_scaled_precision_tcgen05_gb300``) never imports it, and it never
imports the product path.

The arithmetic lives in ``qk_oracle.c`` (plain C, compiled with gcc
``-O2 -ffp-contract=off``, no fast-math, OpenMP over independent outputs).
This module only builds that file and marshals numpy arrays through ctypes.
Every function cites the passage it follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qk_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

FMT_MXFP8_E4M3 = 1
FMT_MXFP4_E2M1 = 2

OK = 0
ERR_ARG = 1
ERR_INT32 = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False, extra_cflags: tuple[str, ...] = (), out_path: str | None = None) -> str:
    """Compile qk_oracle.c into a shared library and return its path."""
    out = out_path or _LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c99",
           "-Wall", "-shared", "-fPIC", *extra_cflags, "-o", out + ".tmp", _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _declare(lib):
    c = ctypes
    P = c.c_void_p
    i64 = c.c_int64
    lib.qko_init.restype = None
    lib.qko_decode_e4m3.argtypes = [c.c_uint8]
    lib.qko_decode_e4m3.restype = c.c_double
    lib.qko_decode_e2m1.argtypes = [c.c_uint8]
    lib.qko_decode_e2m1.restype = c.c_double
    lib.qko_decode_ue8m0.argtypes = [c.c_uint8]
    lib.qko_decode_ue8m0.restype = c.c_double
    lib.qko_decode_ue4m3.argtypes = [c.c_uint8]
    lib.qko_decode_ue4m3.restype = c.c_double
    lib.qko_f32_to_bf16_rne.argtypes = [c.c_float]
    lib.qko_f32_to_bf16_rne.restype = c.c_uint16
    lib.qko_f32_to_f16_rne.argtypes = [c.c_float]
    lib.qko_f32_to_f16_rne.restype = c.c_uint16
    lib.qko_bf16_to_f32.argtypes = [c.c_uint16]
    lib.qko_bf16_to_f32.restype = c.c_float
    lib.qko_encode_e4m3.argtypes = [c.c_double]
    lib.qko_encode_e4m3.restype = c.c_uint8
    lib.qko_encode_e2m1.argtypes = [c.c_double]
    lib.qko_encode_e2m1.restype = c.c_uint8
    lib.qko_mx_quantize_block.argtypes = [c.c_int, P, P, P]
    lib.qko_mx_quantize_block.restype = None
    lib.qko_ptpc_quantize_row.argtypes = [P, i64, P, P]
    lib.qko_ptpc_quantize_row.restype = None
    lib.qko_gemm_int8_rowwise.argtypes = [P, P, P, P, P, P, i64, i64, i64, i64, i64, i64, i64, i64, P]
    lib.qko_gemm_int8_rowwise.restype = c.c_int
    lib.qko_gemm_int8_rowwise_out.argtypes = [P, P, P, P, P, P, c.c_int, i64, i64, i64, i64, i64, i64, i64, i64, P]
    lib.qko_gemm_int8_rowwise_out.restype = c.c_int
    lib.qko_gemm_fp8_rowwise.argtypes = [P, P, P, P, P, P, i64, i64, i64, i64, i64, i64, i64, i64]
    lib.qko_gemm_fp8_rowwise.restype = c.c_int
    lib.qko_gemm_mx.argtypes = [c.c_int, P, P, P, P, P, P, i64, i64, i64, i64, i64, i64, i64, i64]
    lib.qko_gemm_mx.restype = c.c_int
    lib.qko_gemm_mx_b32.argtypes = [c.c_int, P, P, P, P, P, P, i64, i64, i64, i64, i64, i64, i64, i64]
    lib.qko_gemm_mx_b32.restype = c.c_int
    lib.qko_gemm_nvfp4.argtypes = [P, P, P, P, c.c_float, c.c_float, P, P, i64, i64, i64, i64, i64, i64, i64, i64]
    lib.qko_gemm_nvfp4.restype = c.c_int
    lib.qko_gemm_fp8_blockscale.argtypes = [P, P, P, P, P, P, i64, i64, i64, i64, i64, i64, i64, i64]
    lib.qko_gemm_fp8_blockscale.restype = c.c_int
    lib.qko_num_threads.restype = c.c_int
    lib.qko_init()


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
        _declare(lib)
        return lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            _declare(lib)
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def num_threads(lib=None) -> int:
    return int((lib or load()).qko_num_threads())


def decode_e4m3(codes, lib=None):
    lib = lib or load()
    return np.array([lib.qko_decode_e4m3(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


def decode_e2m1(codes, lib=None):
    lib = lib or load()
    return np.array([lib.qko_decode_e2m1(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


def decode_ue8m0(codes, lib=None):
    lib = lib or load()
    return np.array([lib.qko_decode_ue8m0(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


def decode_ue4m3(codes, lib=None):
    lib = lib or load()
    return np.array([lib.qko_decode_ue4m3(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


def f32_to_bf16(x, lib=None):
    lib = lib or load()
    return np.array([lib.qko_f32_to_bf16_rne(float(v)) for v in np.ravel(np.asarray(x, np.float32))],
                    dtype=np.uint16).reshape(np.shape(x))


def f32_to_f16(x, lib=None):
    """IEEE binary16 bits (uint16) of fp32 values, round to nearest even."""
    lib = lib or load()
    return np.array([lib.qko_f32_to_f16_rne(float(v)) for v in np.ravel(np.asarray(x, np.float32))],
                    dtype=np.uint16).reshape(np.shape(x))


def bf16_to_f32(b, lib=None):
    lib = lib or load()
    return np.array([lib.qko_bf16_to_f32(int(v)) for v in np.ravel(b)], dtype=np.float32).reshape(np.shape(b))


def encode_e4m3(x, lib=None):
    lib = lib or load()
    return np.array([lib.qko_encode_e4m3(float(v)) for v in np.ravel(x)], dtype=np.uint8).reshape(np.shape(x))


def encode_e2m1(x, lib=None):
    lib = lib or load()
    return np.array([lib.qko_encode_e2m1(float(v)) for v in np.ravel(x)], dtype=np.uint8).reshape(np.shape(x))


def mx_quantize_block(fmt: int, v, lib=None):
    """Quantize one block of 32 values; returns (codes[32] one per byte, scale_code)."""
    lib = lib or load()
    v = np.ascontiguousarray(np.asarray(v, np.float32).reshape(32))
    codes = np.zeros(32, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib.qko_mx_quantize_block(int(fmt), _ptr(v), _ptr(codes), _ptr(sc))
    return codes, int(sc[0])


def ptpc_quantize(x, lib=None):
    """Per-row E4M3 codes and fp32 scales of a [rows, K] float32 matrix."""
    lib = lib or load()
    x = _c(np.asarray(x, np.float32), np.float32)
    rows, K = x.shape
    codes = np.zeros((rows, K), np.uint8)
    scales = np.zeros(rows, np.float32)
    for r in range(rows):
        lib.qko_ptpc_quantize_row(_ptr(x[r]), K, codes[r].ctypes.data_as(ctypes.c_void_p),
                                  scales[r:].ctypes.data_as(ctypes.c_void_p))
    return codes, scales


def mx_quantize(fmt, x, lib=None):
    """MX codes (one per byte, E2M1 unpacked) and scale bytes of a [rows, K] float32 matrix."""
    lib = lib or load()
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    rows, K = x.shape
    codes = np.zeros((rows, K), np.uint8)
    scales = np.zeros((rows, K // 32), np.uint8)
    for r in range(rows):
        for b in range(K // 32):
            c, sc = mx_quantize_block(fmt, x[r, 32 * b:32 * b + 32], lib)
            codes[r, 32 * b:32 * b + 32] = c
            scales[r, b] = sc
    return codes, scales


def _region(M, N, m0, m1, n0, n1):
    m1 = M if m1 is None else m1
    n1 = N if n1 is None else n1
    return m0, m1, n0, n1


OUT_TYPES = {"bf16": 0, "fp16": 1, "fp32": 2}


def gemm_int8_rowwise(A, B, sa, sb, bias=None, m0=0, m1=None, n0=0, n1=None, return_acc=False, lib=None,
                      out_dtype="bf16"):
    """The INT8 row/column-scaled GEMM over rows [m0,m1) x cols [n0,n1): bf16 or
    fp16 bits (uint16, round to nearest even) or the fp32 values themselves
    (out_dtype "bf16", "fp16" or "fp32")."""
    lib = lib or load()
    A = _c(A, np.int8)
    B = _c(B, np.int8)
    sa = _c(sa, np.float32)
    sb = _c(sb, np.float32)
    bias = _c(bias, np.uint16)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K and sa.shape == (M,) and sb.shape == (N,)
    m0, m1, n0, n1 = _region(M, N, m0, m1, n0, n1)
    out = np.zeros((m1 - m0, n1 - n0), np.float32 if out_dtype == "fp32" else np.uint16)
    acc = np.zeros((m1 - m0, n1 - n0), np.int64) if return_acc else None
    if out_dtype == "bf16":
        rc = lib.qko_gemm_int8_rowwise(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias), _ptr(out),
                                       n1 - n0, M, N, K, m0, m1, n0, n1, _ptr(acc))
    else:
        rc = lib.qko_gemm_int8_rowwise_out(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias), _ptr(out),
                                           OUT_TYPES[out_dtype], n1 - n0, M, N, K, m0, m1, n0, n1, _ptr(acc))
    if rc != OK:
        raise ValueError(f"oracle int8 gemm failed with code {rc}")
    return (out, acc) if return_acc else out


def gemm_fp8_rowwise(A, B, sa, sb, bias=None, m0=0, m1=None, n0=0, n1=None, lib=None):
    """fp64 value, before bf16 rounding, of the FP8 E4M3 per-token x per-channel GEMM."""
    lib = lib or load()
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(sa, np.float32)
    sb = _c(sb, np.float32)
    bias = _c(bias, np.uint16)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K and sa.shape == (M,) and sb.shape == (N,)
    m0, m1, n0, n1 = _region(M, N, m0, m1, n0, n1)
    ref = np.zeros((m1 - m0, n1 - n0), np.float64)
    rc = lib.qko_gemm_fp8_rowwise(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias), _ptr(ref),
                                  n1 - n0, M, N, K, m0, m1, n0, n1)
    if rc != OK:
        raise ValueError(f"oracle fp8 gemm failed with code {rc}")
    return ref


def gemm_mx(fmt, A, sA, B, sB, bias=None, K=None, m0=0, m1=None, n0=0, n1=None, lib=None):
    """fp64 value, before bf16 rounding, of the MX block-scaled GEMM.

    ``A``/``B`` are the raw operand bytes ([M,K] for MXFP8, [M,K/2] packed for
    MXFP4), ``sA``/``sB`` the raw [rows, K/32] ue8m0 bytes.
    """
    lib = lib or load()
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sA = _c(sA, np.uint8)
    sB = _c(sB, np.uint8)
    bias = _c(bias, np.uint16)
    M = A.shape[0]
    N = B.shape[0]
    if K is None:
        K = A.shape[1] * (2 if fmt == FMT_MXFP4_E2M1 else 1)
    assert sA.shape == (M, K // 32) and sB.shape == (N, K // 32)
    m0, m1, n0, n1 = _region(M, N, m0, m1, n0, n1)
    ref = np.zeros((m1 - m0, n1 - n0), np.float64)
    rc = lib.qko_gemm_mx(int(fmt), _ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(bias), _ptr(ref),
                         n1 - n0, M, N, K, m0, m1, n0, n1)
    if rc != OK:
        raise ValueError(f"oracle mx gemm failed with code {rc}")
    return ref


def gemm_mx_b32(fmt, A, sA, B, sB32, bias=None, K=None, m0=0, m1=None, n0=0, n1=None, lib=None):
    """fp64 value, before bf16 rounding, of the MX GEMM whose B scales cover 32x32
    blocks: ``sA`` [M, K/32] as in gemm_mx, ``sB32`` [ceil(N/32), K/32], row n of B
    taking scale row n // 32 (ROCm/mori PR #806, "What": the mxfp8_raw form)."""
    lib = lib or load()
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sA = _c(sA, np.uint8)
    sB32 = _c(sB32, np.uint8)
    bias = _c(bias, np.uint16)
    M = A.shape[0]
    N = B.shape[0]
    if K is None:
        K = A.shape[1] * (2 if fmt == FMT_MXFP4_E2M1 else 1)
    assert sA.shape == (M, K // 32) and sB32.shape == ((N + 31) // 32, K // 32)
    m0, m1, n0, n1 = _region(M, N, m0, m1, n0, n1)
    ref = np.zeros((m1 - m0, n1 - n0), np.float64)
    rc = lib.qko_gemm_mx_b32(int(fmt), _ptr(A), _ptr(sA), _ptr(B), _ptr(sB32), _ptr(bias), _ptr(ref),
                             n1 - n0, M, N, K, m0, m1, n0, n1)
    if rc != OK:
        raise ValueError(f"oracle mx b32 gemm failed with code {rc}")
    return ref


def gemm_nvfp4(A, sA, B, sB, global_a=1.0, global_b=1.0, bias=None, m0=0, m1=None, n0=0, n1=None, lib=None):
    """fp64 value, before bf16 rounding, of the NVFP4 GEMM (see qko_gemm_nvfp4).

    ``A``/``B`` are packed E2M1 bytes [rows, K/2], ``sA``/``sB`` raw UE4M3
    bytes [rows, K/16], ``global_a``/``global_b`` the per-tensor fp32 scales.
    """
    lib = lib or load()
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sA = _c(sA, np.uint8)
    sB = _c(sB, np.uint8)
    bias = _c(bias, np.uint16)
    M, N = A.shape[0], B.shape[0]
    K = 2 * A.shape[1]
    assert B.shape[1] == K // 2 and sA.shape == (M, K // 16) and sB.shape == (N, K // 16)
    m0, m1, n0, n1 = _region(M, N, m0, m1, n0, n1)
    ref = np.zeros((m1 - m0, n1 - n0), np.float64)
    rc = lib.qko_gemm_nvfp4(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), float(np.float32(global_a)),
                            float(np.float32(global_b)), _ptr(bias), _ptr(ref), n1 - n0, M, N, K, m0, m1, n0, n1)
    if rc != OK:
        raise ValueError(f"oracle nvfp4 gemm failed with code {rc}")
    return ref


def gemm_fp8_blockscale(A, B, sa, sb, bias=None, m0=0, m1=None, n0=0, n1=None, lib=None):
    """fp64 value, before bf16 rounding, of the FP8 blockscale GEMM (see qko_gemm_fp8_blockscale).

    ``sa`` is [M, ceil(K/128)] and ``sb`` [ceil(N/128), ceil(K/128)] fp32.
    """
    lib = lib or load()
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(sa, np.float32)
    sb = _c(sb, np.float32)
    bias = _c(bias, np.uint16)
    M, K = A.shape
    N = B.shape[0]
    KB, NB = -(-K // 128), -(-N // 128)
    assert B.shape[1] == K and sa.shape == (M, KB) and sb.shape == (NB, KB)
    m0, m1, n0, n1 = _region(M, N, m0, m1, n0, n1)
    ref = np.zeros((m1 - m0, n1 - n0), np.float64)
    rc = lib.qko_gemm_fp8_blockscale(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias), _ptr(ref),
                                     n1 - n0, M, N, K, m0, m1, n0, n1)
    if rc != OK:
        raise ValueError(f"oracle fp8 blockscale gemm failed with code {rc}")
    return ref
