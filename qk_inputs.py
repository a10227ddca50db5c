"""Seeded synthetic inputs for the quantized GEMM workloads.

This module is shared by the tests, the smoke check and the benchmark.  It
holds the workload recipes (shapes, value distributions, seeds) and the
input-side encoders that turn real-valued draws into operand bytes (E4M3,
packed E2M1, UE8M0 scales, int8).  It contains none of the GEMM's arithmetic,
imports neither the oracle nor the CUDA package, and the oracle and the GPU
consume exactly the bytes produced here.

Recipes (the model-projection shapes of the pages, with synthetic values):

* INT8 row/column-scaled: A, B int8 uniform in [-127, 127]; sa[M], sb[N]
  fp32 uniform in [1e-3, 1e-2]; bias bf16 from N(0, 1).
* MXFP8: A from bf16 N(0, 1) with 1% of entries (seeded uniform mask) x20;
  B from bf16 N(0, 0.02); both MX-quantized to E4M3 + UE8M0 per 32 along K.
* MXFP4: A, B from bf16 N(0, 1), MX-quantized to packed E2M1 + UE8M0.
* FP8 per-token x per-channel: A N(0, 1), W N(0, 0.02); per-row scale
  s = amax/448 (1 for an all-zero row), q = E4M3(x / s).
* FP8 blockscale: A N(0, 1) with fp32 scales per 1x128 (row, K-block),
  W N(0, 0.02) with fp32 scales per 128x128 block; s = amax/448 over the
  group (1 for an all-zero group), q = E4M3(x / s).
* NVFP4: A, B from bf16 N(0, 1); per-tensor fp32 scale g = amax/(448*6)
  over the whole operand; per 16 K-elements a UE4M3 scale
  s = E4M3((amax_block/6)/g) (saturating), elements E2M1(x/(s*g)).

Every generator is a pure function of (shape, seed).  Each operand draws from
its own stream, numpy default_rng([seed, tag]) with tag 0 = A, 1 = B, 2 = sa,
3 = sb, 4 = bias, so a weight matrix does not depend on M.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

FMT_MXFP8_E4M3 = 1
FMT_MXFP4_E2M1 = 2

_ROW_CHUNK = 2048  # rows drawn per chunk; part of the recipe (fixes the stream order)


# ----------------------------------------------------------------------------
# input-side encoders
# ----------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    u = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return u.astype(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _round_mantissa(a: np.ndarray, keep_bits: int) -> np.ndarray:
    """Round non-negative float32 values to `keep_bits` mantissa bits, ties to
    even, on the bit pattern; returns the rounded bit patterns (uint32)."""
    drop = 23 - keep_bits
    u = a.view(np.uint32)
    lsb = (u >> np.uint32(drop)) & np.uint32(1)
    r = u + (np.uint32((1 << (drop - 1)) - 1) + lsb)
    return r & np.uint32(~((1 << drop) - 1) & 0xFFFFFFFF)


def encode_e4m3(q: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3FN value (ties to even), saturating at 448."""
    q = np.asarray(q, np.float32)
    sign = (q.view(np.uint32) >> np.uint32(31)).astype(np.uint8) << np.uint8(7)
    a = np.minimum(np.abs(q), np.float32(448.0))
    r = _round_mantissa(a, 3)
    exp = (r >> np.uint32(23)).astype(np.int32) - 127
    normal_code = (((exp + 7) << 3) | ((r >> np.uint32(20)) & np.uint32(7)).astype(np.int32))
    sub_code = np.rint(a * np.float32(512.0)).astype(np.int32)        # multiples of 2^-9; 8 -> 2^-6
    code = np.where(a < np.float32(2.0 ** -6), sub_code, normal_code).astype(np.uint8)
    return code | sign


def round_e4m3_value(a: np.ndarray) -> np.ndarray:
    """The nearest E4M3FN value (ties to even) of non-negative float32 values, saturating at 448."""
    a = np.minimum(np.asarray(a, np.float32), np.float32(448.0))
    normal = _round_mantissa(a.copy(), 3).view(np.float32)
    sub = (np.rint(a * np.float32(512.0)) / np.float32(512.0)).astype(np.float32)
    return np.where(a < np.float32(2.0 ** -6), sub, normal).astype(np.float32)


# E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6: the code of |q| is the number of
# midpoints it passes.  At a midpoint the tie goes to the even code, i.e.
# down at 0.25, 1.25, 2.5, 5 (to 0, 1, 2, 4) and up at 0.75, 1.75, 3.5 (to 1, 2, 4).
_E2M1_MIDPOINTS = ((0.25, False), (0.75, True), (1.25, False), (1.75, True), (2.5, False), (3.5, True), (5.0, False))


def encode_e2m1(q: np.ndarray) -> np.ndarray:
    """Round to the nearest E2M1 value (ties to even), saturating at 6; one code per byte."""
    q = np.asarray(q, np.float32)
    a = np.abs(q)
    code = np.zeros(q.shape, np.uint8)
    for t, up in _E2M1_MIDPOINTS:
        code += (a >= np.float32(t)) if up else (a > np.float32(t))
    return code | (np.signbit(q).astype(np.uint8) << np.uint8(3))


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """[rows, K] nibble codes -> [rows, K/2] bytes; element 2i in the low nibble."""
    codes = np.asarray(codes, np.uint8)
    return (codes[:, 0::2] & 0xF) | ((codes[:, 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, np.uint8)
    out = np.empty((packed.shape[0], packed.shape[1] * 2), np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def mx_quantize(x: np.ndarray, fmt: int):
    """MX-quantize [rows, K] reals along K in blocks of 32.

    Returns (operand bytes, scale bytes [rows, K/32]).  Shared exponent
    floor(log2(amax)) - emax (8 for E4M3, 2 for E2M1) clamped to [-127, 127],
    code 0 for an all-zero block; elements x / 2^s rounded to nearest even
    and saturated.  MXFP4 operands come back packed two per byte.
    """
    x = np.asarray(x, np.float32)
    rows, K = x.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    blk = x.reshape(rows, K // 32, 32)
    amax = np.abs(blk).max(axis=2)
    _, e = np.frexp(amax.astype(np.float64))
    emax = 8 if fmt == FMT_MXFP8_E4M3 else 2
    sexp = np.clip(e - 1 - emax, -127, 127)
    sexp = np.where(amax == 0.0, -127, sexp).astype(np.int32)
    inv = np.ldexp(np.float32(1.0), -sexp).astype(np.float32)  # always a normal float32
    q = (blk * inv[:, :, None]).reshape(rows, K)                 # exact power-of-two scaling
    if fmt == FMT_MXFP8_E4M3:
        codes = encode_e4m3(q)
    else:
        codes = pack_e2m1(encode_e2m1(q))
    return codes, (sexp + 127).astype(np.uint8)


def ptpc_quantize(x: np.ndarray):
    """Per-row E4M3 quantization with scale amax/448 (1 for an all-zero row)."""
    x = np.asarray(x, np.float32)
    amax = np.abs(x).max(axis=1)
    s = (amax / np.float32(448.0)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    q = (x / s[:, None]).astype(np.float32)
    return encode_e4m3(q), s


def blockscale_quantize(x: np.ndarray, rows_per_block: int):
    """E4M3 codes and fp32 scales per (rows_per_block x 128) group of [rows, K].

    Scales are [ceil(rows/rows_per_block), ceil(K/128)]: s = amax/448 over the
    group (1 for an all-zero group), q = E4M3(x / s) with x / s in fp32.
    """
    x = np.asarray(x, np.float32)
    rows, K = x.shape
    RB, KB = -(-rows // rows_per_block), -(-K // 128)
    pad = np.zeros((RB * rows_per_block, KB * 128), np.float32)
    pad[:rows, :K] = x
    g = np.abs(pad.reshape(RB, rows_per_block, KB, 128)).max(axis=(1, 3))
    s = (g / np.float32(448.0)).astype(np.float32)
    s = np.where(g == 0, np.float32(1.0), s).astype(np.float32)
    full = np.repeat(np.repeat(s, rows_per_block, axis=0), 128, axis=1)[:rows, :K]
    q = (x / full).astype(np.float32)
    return encode_e4m3(q), s


def nvfp4_quantize(x: np.ndarray, global_scale: np.float32):
    """NVFP4-quantize [rows, K] reals along K in blocks of 16 under a per-tensor scale.

    Returns (packed E2M1 bytes [rows, K/2], UE4M3 scale bytes [rows, K/16]).
    Block scale s = E4M3((amax/6)/g) saturating at 448; a block whose scale
    rounds to zero gets zero elements; elements E2M1(x / (s*g)) in fp32.
    """
    x = np.asarray(x, np.float32)
    rows, K = x.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    g = np.float32(global_scale)
    blk = x.reshape(rows, K // 16, 16)
    amax = np.abs(blk).max(axis=2)
    want = ((amax / np.float32(6.0)) / g).astype(np.float32)
    sval = round_e4m3_value(want)
    scodes = encode_e4m3(sval)
    denom = (sval * g).astype(np.float32)
    safe = np.where(denom > 0, denom, np.float32(1.0)).astype(np.float32)
    q = (blk / safe[:, :, None]).astype(np.float32)
    q = np.where((denom > 0)[:, :, None], q, np.float32(0.0)).reshape(rows, K)
    return pack_e2m1(encode_e2m1(q)), scodes


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------

@dataclass
class Int8Problem:
    A: np.ndarray      # int8 [M, K]
    B: np.ndarray      # int8 [N, K]
    sa: np.ndarray     # fp32 [M]
    sb: np.ndarray     # fp32 [N]
    bias: np.ndarray | None  # bf16 bits [N]
    M: int
    N: int
    K: int


@dataclass
class Fp8Problem:
    A: np.ndarray      # e4m3 bytes [M, K]
    B: np.ndarray      # e4m3 bytes [N, K]
    sa: np.ndarray
    sb: np.ndarray
    bias: np.ndarray | None
    M: int
    N: int
    K: int


@dataclass
class MxProblem:
    fmt: int
    A: np.ndarray      # [M, K] (MXFP8) or [M, K/2] (MXFP4) bytes
    sA: np.ndarray     # ue8m0 [M, K/32]
    B: np.ndarray
    sB: np.ndarray
    bias: np.ndarray | None
    M: int
    N: int
    K: int


@dataclass
class BlockscaleProblem:
    A: np.ndarray      # e4m3 bytes [M, K]
    B: np.ndarray      # e4m3 bytes [N, K]
    sa: np.ndarray     # fp32 [M, ceil(K/128)]
    sb: np.ndarray     # fp32 [ceil(N/128), ceil(K/128)]
    bias: np.ndarray | None
    M: int
    N: int
    K: int


@dataclass
class Nvfp4Problem:
    A: np.ndarray      # packed e2m1 [M, K/2]
    sA: np.ndarray     # ue4m3 [M, K/16]
    B: np.ndarray
    sB: np.ndarray
    global_a: float    # per-tensor fp32 scales
    global_b: float
    bias: np.ndarray | None
    M: int
    N: int
    K: int


def _normal_rows(rng, rows, K, std, fn):
    """Draw [rows, K] N(0, std^2) in fixed row chunks, rounded to bf16, then fn(chunk)."""
    outs = []
    for r0 in range(0, rows, _ROW_CHUNK):
        r = min(_ROW_CHUNK, rows - r0)
        x = rng.standard_normal((r, K), dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        outs.append(fn(x))
    return outs


TAG_A, TAG_B, TAG_SA, TAG_SB, TAG_BIAS = 0, 1, 2, 3, 4


def _rng(seed: int, tag: int):
    return np.random.default_rng([int(seed), int(tag)])


def bias_bits(N: int, seed: int) -> np.ndarray:
    return to_bf16_bits(_rng(seed, TAG_BIAS).standard_normal(N).astype(np.float32))


def int8_problem(M: int, N: int, K: int, seed: int = 0, bias: bool = True) -> Int8Problem:
    A = _rng(seed, TAG_A).integers(-127, 128, size=(M, K), dtype=np.int8)
    B = _rng(seed, TAG_B).integers(-127, 128, size=(N, K), dtype=np.int8)
    sa = _rng(seed, TAG_SA).uniform(1e-3, 1e-2, size=M).astype(np.float32)
    sb = _rng(seed, TAG_SB).uniform(1e-3, 1e-2, size=N).astype(np.float32)
    return Int8Problem(A, B, sa, sb, bias_bits(N, seed) if bias else None, M, N, K)


def _cat(parts, idx, empty_shape, dtype):
    return np.concatenate([p[idx] for p in parts]) if parts else np.zeros(empty_shape, dtype)


def mx_operand(fmt: int, rows: int, K: int, seed: int, tag: int):
    """(bytes, scales) of one MX operand of the recipe: tag TAG_A or TAG_B."""
    rng = _rng(seed, tag)

    def quant(x):
        return mx_quantize(from_bf16_bits(to_bf16_bits(x)), fmt)

    if fmt == FMT_MXFP8_E4M3 and tag == TAG_A:
        def chunk(x):
            mask = rng.uniform(size=x.shape) < 0.01
            x[mask] *= np.float32(20.0)
            return quant(x)
        parts = _normal_rows(rng, rows, K, 1.0, chunk)
    elif fmt == FMT_MXFP8_E4M3:
        parts = _normal_rows(rng, rows, K, 0.02, quant)
    elif fmt == FMT_MXFP4_E2M1:
        parts = _normal_rows(rng, rows, K, 1.0, quant)
    else:
        raise ValueError("unknown MX format")
    width = K if fmt == FMT_MXFP8_E4M3 else K // 2
    return _cat(parts, 0, (0, width), np.uint8), _cat(parts, 1, (0, K // 32), np.uint8)


def mx_problem(fmt: int, M: int, N: int, K: int, seed: int = 0, bias: bool = False) -> MxProblem:
    A, sA = mx_operand(fmt, M, K, seed, TAG_A)
    B, sB = mx_operand(fmt, N, K, seed, TAG_B)
    return MxProblem(fmt, A, sA, B, sB, bias_bits(N, seed) if bias else None, M, N, K)


def fp8_operand(rows: int, K: int, seed: int, tag: int):
    """(E4M3 bytes, fp32 row scales) of one per-token / per-channel operand: A ~ N(0,1), W ~ N(0,0.02)."""
    rng = _rng(seed, tag)
    parts = _normal_rows(rng, rows, K, 1.0 if tag == TAG_A else 0.02, ptpc_quantize)
    return _cat(parts, 0, (0, K), np.uint8), _cat(parts, 1, (0,), np.float32).astype(np.float32)


def fp8_problem(M: int, N: int, K: int, seed: int = 0, bias: bool = False, weights=None) -> Fp8Problem:
    """weights: an optional precomputed fp8_operand(N, K, seed, TAG_B)."""
    A, sa = fp8_operand(M, K, seed, TAG_A)
    B, sb = weights if weights is not None else fp8_operand(N, K, seed, TAG_B)
    return Fp8Problem(A, B, sa, sb, bias_bits(N, seed) if bias else None, M, N, K)


def sample_tiles(M: int, N: int, count: int, seed: int, tile: int = 128):
    """A seeded sample of output tiles plus every ragged edge tile.

    Returns a sorted list of (m0, m1, n0, n1): `count` seeded random tiles,
    the first and the last (corner) tile, every tile of the last row-block
    when M is not a multiple of `tile`, every tile of the last column-block
    when N is not, and otherwise one seeded tile of that last block."""
    rng = np.random.default_rng(seed + 7919)
    mt = (M + tile - 1) // tile
    nt = (N + tile - 1) // tile
    picks = set()
    for _ in range(count):
        picks.add((int(rng.integers(mt)), int(rng.integers(nt))))
    picks.add((0, 0))
    picks.add((mt - 1, nt - 1))
    if M % tile:
        picks.update((mt - 1, bn) for bn in range(nt))
    else:
        picks.add((mt - 1, int(rng.integers(nt))))
    if N % tile:
        picks.update((bm, nt - 1) for bm in range(mt))
    else:
        picks.add((int(rng.integers(mt)), nt - 1))
    out = []
    for bm, bn in sorted(picks):
        out.append((bm * tile, min(M, bm * tile + tile), bn * tile, min(N, bn * tile + tile)))
    return out


def blockscale_operand(rows: int, K: int, seed: int, tag: int):
    """(E4M3 bytes, fp32 scales) of one blockscale operand: A ~ N(0,1) per 1x128, W ~ N(0,0.02) per 128x128."""
    rng = _rng(seed, tag)
    rpb = 1 if tag == TAG_A else 128
    parts = _normal_rows(rng, rows, K, 1.0 if tag == TAG_A else 0.02, lambda x: blockscale_quantize(x, rpb))
    KB = -(-K // 128)
    return _cat(parts, 0, (0, K), np.uint8), _cat(parts, 1, (0, KB), np.float32).astype(np.float32)


def blockscale_problem(M: int, N: int, K: int, seed: int = 0, bias: bool = False) -> BlockscaleProblem:
    A, sa = blockscale_operand(M, K, seed, TAG_A)
    B, sb = blockscale_operand(N, K, seed, TAG_B)
    return BlockscaleProblem(A, B, sa, sb, bias_bits(N, seed) if bias else None, M, N, K)


def nvfp4_operand(rows: int, K: int, seed: int, tag: int):
    """(packed E2M1, UE4M3 scales, per-tensor scale) of one NVFP4 operand from bf16 N(0, 1).

    Two passes over the same seeded stream: the first finds the operand's
    amax for the per-tensor scale amax/(448*6), the second quantizes.
    """
    def bf16(x):
        return from_bf16_bits(to_bf16_bits(x))

    # rounding to bf16 is monotonic, so the amax of the rounded operand is the rounded amax
    amax = max([float(np.abs(x).max()) for x in _normal_rows(_rng(seed, tag), rows, K, 1.0, lambda x: x)] or [0.0])
    amax = float(bf16(np.array([amax], np.float32))[0])
    g = np.float32(amax) / np.float32(448.0 * 6.0) if amax > 0 else np.float32(1.0)
    parts = _normal_rows(_rng(seed, tag), rows, K, 1.0, lambda x: nvfp4_quantize(bf16(x), g))
    return (_cat(parts, 0, (0, K // 2), np.uint8), _cat(parts, 1, (0, K // 16), np.uint8), float(g))


def nvfp4_problem(M: int, N: int, K: int, seed: int = 0, bias: bool = False) -> Nvfp4Problem:
    A, sA, ga = nvfp4_operand(M, K, seed, TAG_A)
    B, sB, gb = nvfp4_operand(N, K, seed, TAG_B)
    return Nvfp4Problem(A, sA, B, sB, ga, gb, bias_bits(N, seed) if bias else None, M, N, K)
