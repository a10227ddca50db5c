"""MX GEMM with B's scales per 32x32 block (ROCm/mori PR #806, "What": the
mxfp8_raw form, B's scales [N/32, K/32]) on the GPU against the oracle,
within |gpu - ref| <= 1e-2*|ref| + 1e-2*rms(ref) element-wise and cosine
>= 0.99999, for MXFP8 and MXFP4.

Shapes after the page's tests: K = 256, 512, 640, 1280, 2048 (one chunk,
only the prologue's chunks, chunks refilled in the loop), any M unpadded
(1, 100, 1000), N with a ragged last 32-row scale group and a ragged last
tile.  A closed form with constant elements pins which scale row each B row
takes; every raw-scale staging mode (TMA, cp.async, per-stage loads) runs;
a sampled full-size 16384x7168x2048 (mori's shape) closes it.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import oracle
import qk_inputs as qi
from gpu_util import assert_close, bias_dev, host_bits, nan_out, to_dev

pytestmark = pytest.mark.gpu

FMTS = [qi.FMT_MXFP8_E4M3, qi.FMT_MXFP4_E2M1]
FMT_IDS = ["mxfp8", "mxfp4"]


def _b32_scales(sB, N, K, rng):
    """A [ceil(N/32), K/32] scale grid in the range of the operand's own codes."""
    lo, hi = int(sB.min()), int(sB.max())
    return rng.integers(max(lo - 2, 0), min(hi + 3, 255), ((N + 31) // 32, K // 32), dtype=np.uint8)


def _run(fmt, A, sA, B, sB32, bias=None, out=None, shift=0):
    M, N = A.shape[0], B.shape[0]
    out = nan_out(M, N) if out is None else out
    sb = to_dev(sB32)
    if shift:
        # scale rows at an offset of `shift` bytes (cp.async staging when not 16-byte aligned)
        flat = torch.zeros(sB32.size + 64, dtype=torch.uint8, device="cuda")
        sb = flat[shift:shift + sB32.size].view(sB32.shape)
        sb.copy_(to_dev(sB32))
    qk.gemm_mx_b32(fmt, to_dev(A), to_dev(sA), to_dev(B), sb, bias_dev(bias), out)
    torch.cuda.synchronize()
    return out


SHAPES = [(1, 8, 256), (100, 136, 512), (130, 264, 640), (1000, 520, 1280), (256, 1000, 2048), (300, 1040, 1792)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_mx_b32_matches_oracle(fmt, shape):
    M, N, K = shape
    p = qi.mx_problem(fmt, M, N, K, seed=M + K + 5)
    sB32 = _b32_scales(p.sB, N, K, np.random.default_rng(K))
    got = host_bits(_run(fmt, p.A, p.sA, p.B, sB32))
    ref = oracle.gemm_mx_b32(fmt, p.A, p.sA, p.B, sB32)
    assert_close(got, ref, f"fmt {fmt} {shape}")


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_mx_b32_with_bias(fmt):
    M, N, K = 200, 264, 512
    p = qi.mx_problem(fmt, M, N, K, seed=19, bias=True)
    sB32 = _b32_scales(p.sB, N, K, np.random.default_rng(3))
    got = host_bits(_run(fmt, p.A, p.sA, p.B, sB32, bias=p.bias))
    assert_close(got, oracle.gemm_mx_b32(fmt, p.A, p.sA, p.B, sB32, bias=p.bias), "bias")


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_mx_b32_closed_form(fmt):
    # every element 1.0, sA[m,b] = 127 + da(m,b), sB32[g,b] = 127 + db(g,b):
    # out[m,n] = sum_b 32 * 2^(da(m,b) + db(n/32,b)), exact; N = 296 leaves a
    # last 32-row group of 8 rows and a ragged last tile
    M, N, K = 256, 296, 1024
    nb, ng = K // 32, (N + 31) // 32
    if fmt == qi.FMT_MXFP8_E4M3:
        A, B = np.full((M, K), 0x38, np.uint8), np.full((N, K), 0x38, np.uint8)
    else:
        A, B = np.full((M, K // 2), 0x22, np.uint8), np.full((N, K // 2), 0x22, np.uint8)
    da = (np.arange(M)[:, None] * 7 + np.arange(nb)[None, :] * 3) % 5 - 2
    db = (np.arange(ng)[:, None] * 5 + np.arange(nb)[None, :]) % 7 - 3
    sA = (127 + da).astype(np.uint8)
    sB32 = (127 + db).astype(np.uint8)
    ref = oracle.gemm_mx_b32(fmt, A, sA, B, sB32)
    want = (32.0 * np.exp2(da[:, None, :] + db[np.arange(N) // 32][None, :, :])).sum(axis=2)
    assert np.array_equal(ref, want)
    got = host_bits(_run(fmt, A, sA, B, sB32))
    assert np.array_equal(got, qi.to_bf16_bits(ref.astype(np.float32))), "powers of two must round exactly"


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("K,shift", [(1024, 0), (1024, 4), (896, 0), (96, 0)],
                         ids=["tma", "async-misaligned", "async", "loads"])
def test_mx_b32_scale_staging_modes(fmt, K, shift):
    M, N = 300, 264
    p = qi.mx_problem(fmt, M, N, K, seed=K + shift + 1)
    sB32 = _b32_scales(p.sB, N, K, np.random.default_rng(K + shift))
    got = host_bits(_run(fmt, p.A, p.sA, p.B, sB32, shift=shift))
    assert_close(got, oracle.gemm_mx_b32(fmt, p.A, p.sA, p.B, sB32), f"K={K} shift={shift}")


def test_mx_b32_equals_row_replicated_scales():
    # the same GEMM through qk_gemm_mx with each group's scale row repeated for
    # its 32 rows: both kernels sum the same products in the same order
    M, N, K = 384, 776, 2048
    for fmt in FMTS:
        p = qi.mx_problem(fmt, M, N, K, seed=23)
        sB32 = _b32_scales(p.sB, N, K, np.random.default_rng(23))
        sB = np.ascontiguousarray(np.repeat(sB32, 32, axis=0)[:N])
        got32 = host_bits(_run(fmt, p.A, p.sA, p.B, sB32))
        out = nan_out(M, N)
        qk.gemm_mx(fmt, to_dev(p.A), to_dev(p.sA), to_dev(p.B), to_dev(sB), None, out)
        torch.cuda.synchronize()
        assert np.array_equal(got32, host_bits(out)), fmt


@pytest.mark.slow
def test_mxfp8_b32_full_16384x7168x2048():
    M, N, K = 16384, 7168, 2048
    fmt = qi.FMT_MXFP8_E4M3
    p = qi.mx_problem(fmt, M, N, K, seed=0)
    sB32 = _b32_scales(p.sB, N, K, np.random.default_rng(0))
    out = _run(fmt, p.A, p.sA, p.B, sB32)
    gots, refs = [], []
    for (m0, m1, n0, n1) in qi.sample_tiles(M, N, 12, 5):
        gots.append(host_bits(out[m0:m1, n0:n1]).ravel())
        refs.append(oracle.gemm_mx_b32(fmt, p.A, p.sA, p.B, sB32, m0=m0, m1=m1, n0=n0, n1=n1).ravel())
    assert not torch.isnan(out).any().item()
    assert_close(np.concatenate(gots)[None, :], np.concatenate(refs)[None, :], "mxfp8 b32 16384x7168x2048")
