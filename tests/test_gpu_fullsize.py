"""Full-size workloads (the configurations the benchmark times, and the
few-row decode shapes), checked on a seeded sample of 128x128 output tiles
plus every ragged edge tile, which the oracle computes one by one: INT8
bit-exact, MX/FP8 within tolerance (the rms in the bound is taken over the
sampled outputs)."""
import functools

import numpy as np
import pytest
import torch

import oracle
import qk_inputs as qi
from gpu_util import assert_bit_exact, assert_close, host_bits, run_fp8, run_int8, run_mx

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_TILES = 12


def _tiles(M, N, seed):
    return qi.sample_tiles(M, N, N_TILES, seed)


@pytest.mark.parametrize("bias", [False, True], ids=["nobias", "bias"])
def test_int8_30000x21504x5376(bias):
    M, N, K = 30000, 21504, 5376
    p = qi.int8_problem(M, N, K, seed=0, bias=bias)
    out = run_int8(p)
    for (m0, m1, n0, n1) in _tiles(M, N, 1):
        got = host_bits(out[m0:m1, n0:n1])
        ref = oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias, m0=m0, m1=m1, n0=n0, n1=n1)
        assert_bit_exact(got, ref, f"tile {m0}:{m1}, {n0}:{n1}")
    assert not torch.isnan(out).any().item()
    del out
    torch.cuda.empty_cache()


def _mx_sampled(fmt, M, N, K):
    p = qi.mx_problem(fmt, M, N, K, seed=0)
    out = run_mx(p)
    gots, refs = [], []
    for (m0, m1, n0, n1) in _tiles(M, N, 2):
        gots.append(host_bits(out[m0:m1, n0:n1]).ravel())
        refs.append(oracle.gemm_mx(fmt, p.A, p.sA, p.B, p.sB, m0=m0, m1=m1, n0=n0, n1=n1).ravel())
    assert not torch.isnan(out).any().item()
    assert_close(np.concatenate(gots)[None, :], np.concatenate(refs)[None, :], f"fmt {fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("shape", [(16384, 7168, 2048), (32768, 7168, 1792)], ids=lambda s: "x".join(map(str, s)))
def test_mxfp8_full(shape):
    _mx_sampled(qi.FMT_MXFP8_E4M3, *shape)


@pytest.mark.parametrize("shape", [(8192, 8192, 8192), (8192, 8192, 16384), (16384, 16384, 8192),
                                   (16384, 16384, 16384)],
                         ids=lambda s: "x".join(map(str, s)))
def test_mxfp4_full(shape):
    _mx_sampled(qi.FMT_MXFP4_E2M1, *shape)


@pytest.mark.parametrize("shape", [(8192, 8192, 16384), (16384, 16384, 8192)], ids=lambda s: "x".join(map(str, s)))
def test_nvfp4_full(shape):
    from gpu_util import run_nvfp4
    M, N, K = shape
    p = qi.nvfp4_problem(M, N, K, seed=0)
    out = run_nvfp4(p)
    gots, refs = [], []
    for (m0, m1, n0, n1) in _tiles(M, N, 3):
        gots.append(host_bits(out[m0:m1, n0:n1]).ravel())
        refs.append(oracle.gemm_nvfp4(p.A, p.sA, p.B, p.sB, p.global_a, p.global_b, m0=m0, m1=m1, n0=n0,
                                      n1=n1).ravel())
    assert not torch.isnan(out).any().item()
    assert_close(np.concatenate(gots)[None, :], np.concatenate(refs)[None, :], f"nvfp4 {M}x{N}x{K}")


@pytest.mark.parametrize("shape", [(16384, 7168, 2048), (30000, 21504, 5376)], ids=lambda s: "x".join(map(str, s)))
def test_fp8_blockscale_full(shape):
    from gpu_util import run_blockscale
    M, N, K = shape
    p = qi.blockscale_problem(M, N, K, seed=0)
    out = run_blockscale(p)
    gots, refs = [], []
    for (m0, m1, n0, n1) in _tiles(M, N, 4):
        gots.append(host_bits(out[m0:m1, n0:n1]).ravel())
        refs.append(oracle.gemm_fp8_blockscale(p.A, p.B, p.sa, p.sb, m0=m0, m1=m1, n0=n0, n1=n1).ravel())
    assert not torch.isnan(out).any().item()
    assert_close(np.concatenate(gots)[None, :], np.concatenate(refs)[None, :], f"blockscale {M}x{N}x{K}")


FP8_SWEEP = [(M, N, K) for (N, K) in ((2112, 7168), (7168, 1792), (21504, 5376)) for M in (64, 1024, 4096, 16384, 30000)]


@functools.lru_cache(maxsize=1)
def _fp8_weights(N, K):
    return qi.fp8_operand(N, K, 0, qi.TAG_B)


@pytest.mark.parametrize("shape", FP8_SWEEP, ids=lambda s: "x".join(map(str, s)))
def test_fp8_ptpc_sweep(shape):
    M, N, K = shape
    p = qi.fp8_problem(M, N, K, seed=0, weights=_fp8_weights(N, K))
    out = run_fp8(p)
    gots, refs = [], []
    for (m0, m1, n0, n1) in qi.sample_tiles(M, N, 4, 3):
        gots.append(host_bits(out[m0:m1, n0:n1]).ravel())
        refs.append(oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, p.sb, m0=m0, m1=m1, n0=n0, n1=n1).ravel())
    assert not torch.isnan(out).any().item()
    assert_close(np.concatenate(gots)[None, :], np.concatenate(refs)[None, :], f"fp8 {shape}")


# MXFP8 with few rows at the decode shapes: every dispatch the few-row logic
# can take (cluster split-K, stream-K, tile kernel) across M = 1 .. 128.
MX_FEWROW = [(M, N, K) for (N, K) in ((2112, 7168), (7168, 2048), (8192, 1280), (21504, 5376))
             for M in (1, 16, 64, 128)]


@functools.lru_cache(maxsize=1)
def _mx_weights(N, K):
    return qi.mx_operand(qi.FMT_MXFP8_E4M3, N, K, 0, qi.TAG_B)


@pytest.mark.parametrize("shape", MX_FEWROW, ids=lambda s: "x".join(map(str, s)))
def test_mxfp8_fewrow_sweep(shape):
    M, N, K = shape
    A, sA = qi.mx_operand(qi.FMT_MXFP8_E4M3, M, K, 0, qi.TAG_A)
    B, sB = _mx_weights(N, K)
    p = qi.MxProblem(qi.FMT_MXFP8_E4M3, A, sA, B, sB, None, M, N, K)
    out = run_mx(p)
    gots, refs = [], []
    for (m0, m1, n0, n1) in qi.sample_tiles(M, N, 4, 3):
        gots.append(host_bits(out[m0:m1, n0:n1]).ravel())
        refs.append(oracle.gemm_mx(p.fmt, A, sA, B, sB, m0=m0, m1=m1, n0=n0, n1=n1).ravel())
    assert not torch.isnan(out).any().item()
    assert_close(np.concatenate(gots)[None, :], np.concatenate(refs)[None, :], f"mxfp8 few-row {shape}")
