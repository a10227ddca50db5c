"""Block-scaled / quantized GEMM for GB300 (sm_103a).

Python binding of ``libqk.so`` (C ABI declared in ``include/qk.h``).  This
module only marshals arguments: shape/dtype/device checks, raw pointers and
the current CUDA stream.  Every step of the GEMM runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and every call fails loudly when
the library has not been built.

    out = gemm_int8_rowwise(A, B, sa, sb, bias=None, out=None)
    out = gemm_fp8_rowwise(A, B, sa, sb, bias=None, out=None)
    out = gemm_mx(fmt, A, sA, B, sB, bias=None, out=None)

Operands follow the ABI: A [M, K] and B [N, K] K-major (MXFP4: [rows, K/2]
packed bytes), out [M, N] bf16.  E4M3/E2M1/UE8M0 bytes are passed as uint8
tensors.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB as LIB_PATH

QK_OK = 0
QK_ERR_ARG = 1
QK_ERR_ALIGN = 2
QK_ERR_RANGE = 3
QK_ERR_ARCH = 4
QK_ERR_CUDA = 5
QK_ERR_TIMEOUT = 6
QK_ERR_NOMEM = 7
QK_ERR_SCRATCH = 8

QK_OUT_BF16 = 0
QK_OUT_FP16 = 1
QK_OUT_FP32 = 2

FMT_MXFP8_E4M3 = 1
FMT_MXFP4_E2M1 = 2

# every symbol include/qk.h declares
EXPORTS = (
    "qk_gemm_int8_rowwise",
    "qk_gemm_int8_rowwise_out",
    "qk_gemm_int8_rowwise_noalloc",
    "qk_gemm_mx",
    "qk_gemm_mx_out",
    "qk_gemm_mx_b32",
    "qk_gemm_fp8_rowwise",
    "qk_gemm_fp8_rowwise_out",
    "qk_gemm_nvfp4",
    "qk_gemm_nvfp4_out",
    "qk_gemm_fp8_blockscale",
    "qk_quantize_mx",
    "qk_quantize_ptpc",
    "qk_status_string",
    "qk_device_status",
    "qk_set_wait_timeout_ns",
    "qk_wait_timeout_probe",
    "qk_launch_count",
    "qk_profile_enable",
    "qk_profile_read",
    "qk_release",
    "qk_version",
)


class QkError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lib = None


class KernelStats(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_uint64), ("total_ms", ctypes.c_double)]


def _declare(lib):
    c = ctypes
    P = c.c_void_p
    i64 = c.c_int64
    lib.qk_gemm_int8_rowwise.argtypes = [P, P, P, P, P, P, i64, i64, i64, P]
    lib.qk_gemm_int8_rowwise.restype = c.c_int
    lib.qk_gemm_int8_rowwise_out.argtypes = [P, P, P, P, P, P, c.c_int, i64, i64, i64, P]
    lib.qk_gemm_int8_rowwise_out.restype = c.c_int
    lib.qk_gemm_int8_rowwise_noalloc.argtypes = [P, P, P, P, P, P, i64, i64, i64, P]
    lib.qk_gemm_int8_rowwise_noalloc.restype = c.c_int
    lib.qk_gemm_fp8_rowwise.argtypes = [P, P, P, P, P, P, i64, i64, i64, P]
    lib.qk_gemm_fp8_rowwise.restype = c.c_int
    lib.qk_gemm_fp8_rowwise_out.argtypes = [P, P, P, P, P, P, c.c_int, i64, i64, i64, P]
    lib.qk_gemm_fp8_rowwise_out.restype = c.c_int
    lib.qk_gemm_mx.argtypes = [c.c_int, P, P, P, P, P, P, i64, i64, i64, P]
    lib.qk_gemm_mx.restype = c.c_int
    lib.qk_gemm_mx_out.argtypes = [c.c_int, P, P, P, P, P, P, c.c_int, i64, i64, i64, P]
    lib.qk_gemm_mx_out.restype = c.c_int
    lib.qk_gemm_mx_b32.argtypes = [c.c_int, P, P, P, P, P, P, i64, i64, i64, P]
    lib.qk_gemm_mx_b32.restype = c.c_int
    lib.qk_gemm_nvfp4.argtypes = [P, P, P, P, P, P, P, P, i64, i64, i64, P]
    lib.qk_gemm_nvfp4.restype = c.c_int
    lib.qk_gemm_nvfp4_out.argtypes = [P, P, P, P, P, P, P, P, c.c_int, i64, i64, i64, P]
    lib.qk_gemm_nvfp4_out.restype = c.c_int
    lib.qk_gemm_fp8_blockscale.argtypes = [P, P, P, P, P, P, i64, i64, i64, P]
    lib.qk_gemm_fp8_blockscale.restype = c.c_int
    lib.qk_quantize_mx.argtypes = [c.c_int, P, P, P, i64, i64, P]
    lib.qk_quantize_mx.restype = c.c_int
    lib.qk_quantize_ptpc.argtypes = [P, P, P, i64, i64, P]
    lib.qk_quantize_ptpc.restype = c.c_int
    lib.qk_status_string.argtypes = [c.c_int]
    lib.qk_status_string.restype = c.c_char_p
    lib.qk_device_status.argtypes = [c.POINTER(c.c_uint64), c.c_int]
    lib.qk_device_status.restype = c.c_int
    lib.qk_set_wait_timeout_ns.argtypes = [c.c_uint64]
    lib.qk_set_wait_timeout_ns.restype = None
    lib.qk_wait_timeout_probe.argtypes = [c.c_uint64, P]
    lib.qk_wait_timeout_probe.restype = c.c_int
    lib.qk_launch_count.argtypes = []
    lib.qk_launch_count.restype = c.c_uint64
    lib.qk_profile_enable.argtypes = [c.c_int]
    lib.qk_profile_enable.restype = None
    lib.qk_profile_read.argtypes = [c.POINTER(KernelStats), c.c_int, c.POINTER(c.c_int), c.c_int]
    lib.qk_profile_read.restype = c.c_int
    lib.qk_release.argtypes = []
    lib.qk_release.restype = c.c_int
    lib.qk_version.argtypes = []
    lib.qk_version.restype = c.c_int


def load_library(path: str | None = None):
    """The ctypes handle of libqk.so; raises if the library was never built."""
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
        _declare(lib)
        return lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with block_scaled_precision_tcgen05_gb300.build.build(); "
                "there is no fallback implementation")
        lib = ctypes.CDLL(LIB_PATH)
        _declare(lib)
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().qk_status_string(int(status)).decode()


def check(status: int) -> None:
    if status != QK_OK:
        raise QkError(status, status_string(status))


def _stream_handle(device):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _expect(t, name, dtype, shape, device):
    import torch
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _on_device(device):
    """Makes the operands' device current for the call: the library keeps its
    per-device state (SM count, status word, workspace pool, scratch address)
    for the current device and launches on that device's stream."""
    import torch
    return torch.cuda.device(device)


def _out(out, M, N, device):
    import torch
    if out is None:
        return torch.empty((M, N), dtype=torch.bfloat16, device=device)
    _expect(out, "out", torch.bfloat16, (M, N), device)
    return out


def gemm_int8_rowwise(A, B, sa, sb, bias=None, out=None, out_dtype=None):
    """out = bf16(((float)(A @ B^T) * sa[:, None]) * sb[None, :] (+ bias)), bit-exact.  With
    out_dtype torch.float16 or torch.float32 (or an `out` of that dtype) the same value is
    written as fp16 (round to nearest even) or as fp32 itself."""
    import torch
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    M, K = A.shape
    N = B.shape[0]
    dev = A.device
    if dev.type != "cuda":
        raise ValueError("operands must be CUDA tensors")
    _expect(A, "A", torch.int8, (M, K), dev)
    _expect(B, "B", torch.int8, (N, K), dev)
    _expect(sa, "sa", torch.float32, (M,), dev)
    _expect(sb, "sb", torch.float32, (N,), dev)
    if bias is not None:
        _expect(bias, "bias", torch.bfloat16, (N,), dev)
    if out_dtype is None:
        out_dtype = torch.bfloat16 if out is None else out.dtype
    codes = {torch.bfloat16: QK_OUT_BF16, torch.float16: QK_OUT_FP16, torch.float32: QK_OUT_FP32}
    if out_dtype not in codes:
        raise ValueError(f"out_dtype must be bfloat16, float16 or float32, not {out_dtype}")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    _expect(out, "out", out_dtype, (M, N), dev)
    if out_dtype == torch.bfloat16:
        with _on_device(dev):
            check(load_library().qk_gemm_int8_rowwise(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias), _ptr(out),
                                                      M, N, K, _stream_handle(dev)))
    else:
        with _on_device(dev):
            check(load_library().qk_gemm_int8_rowwise_out(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias),
                                                          _ptr(out), codes[out_dtype], M, N, K, _stream_handle(dev)))
    return out


def gemm_int8_rowwise_noalloc(A, B, sa, sb, bias=None, out=None):
    """gemm_int8_rowwise without any allocation inside the library: the operands are widened in a
    fixed 32 MiB scratch array ((M + N) * K * 2 bytes at most).  For callers that cannot let a library
    allocate device memory.  Calls that can overlap on the GPU share that array and race; `out` must be
    passed in by the caller (the binding does not allocate it either)."""
    import torch
    if out is None:
        raise ValueError("out must be provided: this entry point allocates nothing")
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    M, K = A.shape
    N = B.shape[0]
    dev = A.device
    if dev.type != "cuda":
        raise ValueError("operands must be CUDA tensors")
    _expect(A, "A", torch.int8, (M, K), dev)
    _expect(B, "B", torch.int8, (N, K), dev)
    _expect(sa, "sa", torch.float32, (M,), dev)
    _expect(sb, "sb", torch.float32, (N,), dev)
    if bias is not None:
        _expect(bias, "bias", torch.bfloat16, (N,), dev)
    _expect(out, "out", torch.bfloat16, (M, N), dev)
    with _on_device(dev):
        check(load_library().qk_gemm_int8_rowwise_noalloc(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias), _ptr(out),
                                                          M, N, K, _stream_handle(dev)))
    return out


def _out_typed(out, out_dtype, M, N, dev):
    """The output tensor and its QK_OUT_* code: `out` (its dtype must agree with out_dtype when both
    are given) or a new [M, N] tensor of out_dtype (bf16 by default)."""
    import torch
    if out_dtype is None:
        out_dtype = torch.bfloat16 if out is None else out.dtype
    codes = {torch.bfloat16: QK_OUT_BF16, torch.float16: QK_OUT_FP16, torch.float32: QK_OUT_FP32}
    if out_dtype not in codes:
        raise ValueError(f"out_dtype must be bfloat16, float16 or float32, not {out_dtype}")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    _expect(out, "out", out_dtype, (M, N), dev)
    return out, codes[out_dtype]


def gemm_fp8_rowwise(A, B, sa, sb, bias=None, out=None, out_dtype=None):
    """FP8 E4M3 GEMM with per-token sa[M] and per-channel sb[N] fp32 scales (uint8 E4M3 bytes in).
    With out_dtype torch.float16 or torch.float32 (or an `out` of that dtype) the same value is
    written as fp16 (round to nearest even) or as fp32 itself."""
    import torch
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    M, K = A.shape
    N = B.shape[0]
    dev = A.device
    if dev.type != "cuda":
        raise ValueError("operands must be CUDA tensors")
    _expect(A, "A", torch.uint8, (M, K), dev)
    _expect(B, "B", torch.uint8, (N, K), dev)
    _expect(sa, "sa", torch.float32, (M,), dev)
    _expect(sb, "sb", torch.float32, (N,), dev)
    if bias is not None:
        _expect(bias, "bias", torch.bfloat16, (N,), dev)
    out, code = _out_typed(out, out_dtype, M, N, dev)
    with _on_device(dev):
        if code == QK_OUT_BF16:
            check(load_library().qk_gemm_fp8_rowwise(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias), _ptr(out),
                                                     M, N, K, _stream_handle(dev)))
        else:
            check(load_library().qk_gemm_fp8_rowwise_out(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias),
                                                         _ptr(out), code, M, N, K, _stream_handle(dev)))
    return out


def gemm_mx(fmt, A, sA, B, sB, bias=None, out=None, out_dtype=None):
    """MX block-scaled GEMM.  fmt FMT_MXFP8_E4M3 ([rows, K] bytes) or FMT_MXFP4_E2M1 ([rows, K/2] bytes);
    sA [M, K/32], sB [N, K/32] raw UE8M0 bytes.  With out_dtype torch.float16 or torch.float32 (or an
    `out` of that dtype) the value is written as fp16 (round to nearest even) or as fp32 itself."""
    import torch
    if fmt not in (FMT_MXFP8_E4M3, FMT_MXFP4_E2M1):
        raise ValueError("unknown MX format")
    M, kbytes = A.shape
    N = B.shape[0]
    K = kbytes * (2 if fmt == FMT_MXFP4_E2M1 else 1)
    dev = A.device
    if dev.type != "cuda":
        raise ValueError("operands must be CUDA tensors")
    _expect(A, "A", torch.uint8, (M, kbytes), dev)
    _expect(B, "B", torch.uint8, (N, kbytes), dev)
    _expect(sA, "sA", torch.uint8, (M, K // 32), dev)
    _expect(sB, "sB", torch.uint8, (N, K // 32), dev)
    if bias is not None:
        _expect(bias, "bias", torch.bfloat16, (N,), dev)
    out, code = _out_typed(out, out_dtype, M, N, dev)
    with _on_device(dev):
        if code == QK_OUT_BF16:
            check(load_library().qk_gemm_mx(int(fmt), _ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(bias), _ptr(out),
                                            M, N, K, _stream_handle(dev)))
        else:
            check(load_library().qk_gemm_mx_out(int(fmt), _ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(bias),
                                                _ptr(out), code, M, N, K, _stream_handle(dev)))
    return out


def gemm_mx_b32(fmt, A, sA, B, sB32, bias=None, out=None):
    """MX GEMM with B's scales per 32x32 block: sA [M, K/32], sB32 [ceil(N/32), K/32] raw UE8M0
    bytes (row n of B takes scale row n // 32); operands as for gemm_mx."""
    import torch
    if fmt not in (FMT_MXFP8_E4M3, FMT_MXFP4_E2M1):
        raise ValueError("unknown MX format")
    M, kbytes = A.shape
    N = B.shape[0]
    K = kbytes * (2 if fmt == FMT_MXFP4_E2M1 else 1)
    dev = A.device
    if dev.type != "cuda":
        raise ValueError("operands must be CUDA tensors")
    _expect(A, "A", torch.uint8, (M, kbytes), dev)
    _expect(B, "B", torch.uint8, (N, kbytes), dev)
    _expect(sA, "sA", torch.uint8, (M, K // 32), dev)
    _expect(sB32, "sB32", torch.uint8, ((N + 31) // 32, K // 32), dev)
    if bias is not None:
        _expect(bias, "bias", torch.bfloat16, (N,), dev)
    out = _out(out, M, N, dev)
    with _on_device(dev):
        check(load_library().qk_gemm_mx_b32(int(fmt), _ptr(A), _ptr(sA), _ptr(B), _ptr(sB32), _ptr(bias), _ptr(out),
                                            M, N, K, _stream_handle(dev)))
    return out


def gemm_fp8_blockscale(A, B, sa, sb, bias=None, out=None):
    """FP8 E4M3 GEMM with fp32 block scales: sa [M, ceil(K/128)], sb [ceil(N/128), ceil(K/128)]."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    dev = A.device
    if dev.type != "cuda":
        raise ValueError("operands must be CUDA tensors")
    KB, NB = -(-K // 128), -(-N // 128)
    _expect(A, "A", torch.uint8, (M, K), dev)
    _expect(B, "B", torch.uint8, (N, K), dev)
    _expect(sa, "sa", torch.float32, (M, KB), dev)
    _expect(sb, "sb", torch.float32, (NB, KB), dev)
    if bias is not None:
        _expect(bias, "bias", torch.bfloat16, (N,), dev)
    out = _out(out, M, N, dev)
    with _on_device(dev):
        check(load_library().qk_gemm_fp8_blockscale(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias), _ptr(out), M, N, K,
                                                    _stream_handle(dev)))
    return out


def gemm_nvfp4(A, sA, B, sB, global_a=None, global_b=None, bias=None, out=None, out_dtype=None):
    """NVFP4 GEMM.  A [M, K/2], B [N, K/2] packed E2M1 bytes; sA [M, K/16], sB [N, K/16] raw UE4M3
    bytes; global_a / global_b optional one-element fp32 CUDA tensors (per-tensor scales).  With
    out_dtype torch.float16 or torch.float32 (or an `out` of that dtype) the value is written as fp16
    (round to nearest even) or as fp32 itself."""
    import torch
    M, kbytes = A.shape
    N = B.shape[0]
    K = 2 * kbytes
    dev = A.device
    if dev.type != "cuda":
        raise ValueError("operands must be CUDA tensors")
    _expect(A, "A", torch.uint8, (M, kbytes), dev)
    _expect(B, "B", torch.uint8, (N, kbytes), dev)
    _expect(sA, "sA", torch.uint8, (M, K // 16), dev)
    _expect(sB, "sB", torch.uint8, (N, K // 16), dev)
    for name, g in (("global_a", global_a), ("global_b", global_b)):
        if g is not None:
            _expect(g, name, torch.float32, (1,), dev)
    if bias is not None:
        _expect(bias, "bias", torch.bfloat16, (N,), dev)
    out, code = _out_typed(out, out_dtype, M, N, dev)
    with _on_device(dev):
        check(load_library().qk_gemm_nvfp4_out(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(global_a),
                                               _ptr(global_b), _ptr(bias), _ptr(out), code, M, N, K,
                                               _stream_handle(dev)))
    return out


def quantize_mx(fmt, x, q=None, scales=None):
    """MX-quantize a bf16 [rows, K] CUDA tensor along K: returns (q, scales) as uint8 tensors
    ([rows, K] E4M3 or [rows, K/2] packed E2M1, and [rows, K/32] UE8M0)."""
    import torch
    if fmt not in (FMT_MXFP8_E4M3, FMT_MXFP4_E2M1):
        raise ValueError("unknown MX format")
    rows, K = x.shape
    dev = x.device
    _expect(x, "x", torch.bfloat16, (rows, K), dev)
    width = K if fmt == FMT_MXFP8_E4M3 else K // 2
    q = torch.empty((rows, width), dtype=torch.uint8, device=dev) if q is None else q
    scales = torch.empty((rows, K // 32), dtype=torch.uint8, device=dev) if scales is None else scales
    _expect(q, "q", torch.uint8, (rows, width), dev)
    _expect(scales, "scales", torch.uint8, (rows, K // 32), dev)
    with _on_device(dev):
        check(load_library().qk_quantize_mx(int(fmt), _ptr(x), _ptr(q), _ptr(scales), rows, K, _stream_handle(dev)))
    return q, scales


def quantize_ptpc(x, q=None, scales=None):
    """Per-row E4M3 quantization of a bf16 [rows, K] CUDA tensor: returns (q uint8 [rows, K], scales fp32 [rows])."""
    import torch
    rows, K = x.shape
    dev = x.device
    _expect(x, "x", torch.bfloat16, (rows, K), dev)
    q = torch.empty((rows, K), dtype=torch.uint8, device=dev) if q is None else q
    scales = torch.empty((rows,), dtype=torch.float32, device=dev) if scales is None else scales
    _expect(q, "q", torch.uint8, (rows, K), dev)
    _expect(scales, "scales", torch.float32, (rows,), dev)
    with _on_device(dev):
        check(load_library().qk_quantize_ptpc(_ptr(x), _ptr(q), _ptr(scales), rows, K, _stream_handle(dev)))
    return q, scales


def device_status(clear: bool = True) -> int:
    w = ctypes.c_uint64(0)
    check(load_library().qk_device_status(ctypes.byref(w), 1 if clear else 0))
    return int(w.value)


def set_wait_timeout_ns(ns: int) -> None:
    load_library().qk_set_wait_timeout_ns(int(ns))


def launch_count() -> int:
    return int(load_library().qk_launch_count())


def profile_enable(on: bool = True) -> None:
    """Record a CUDA event pair around every kernel the library launches."""
    load_library().qk_profile_enable(1 if on else 0)


def profile_read(reset: bool = True) -> dict:
    """{kernel name: (launches, total ms)} for the kernels timed so far."""
    lib = load_library()
    arr = (KernelStats * 16)()
    n = ctypes.c_int(0)
    check(lib.qk_profile_read(arr, 16, ctypes.byref(n), 1 if reset else 0))
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms)) for i in range(min(n.value, 16))}
