"""The tail split of the 2-SM tile kernels (FP8 per-token and the block-scaled
formats): when the last wave of tiles would leave at least half of the SM
pairs idle, its tiles run as K-parts; every part writes its fp32 partial to a
workspace, and per epilogue warp the part that finishes last adds the parts in
K order and runs the epilogue on the sum.

QK_TAIL_SPLIT=n (a test switch) splits the last min(tiles, pairs) tiles into
n parts whatever it costs, so small problems reach every epilogue the split
runs through: FP8 with 16 epilogue warps (K <= 2048), with 8 (K > 2048) and
on 256 x 128 pair tiles, MXFP8, MXFP4 and NVFP4; 2, 3 and 4 parts, with a
short last part where the K-blocks do not divide evenly, and a last K-block
shorter than a ring stage; ragged M and N; a
problem with more tiles than pairs, where whole tiles and K-parts mix.  Checked
on sampled tiles (every ragged edge tile included) against the oracle within
the FP8 / MX tolerance.  With small-integer operands every partial sum is an
exact integer in fp32, so the split result equals the oracle bit for bit.
Repeated calls and CUDA graph replays (FP8 and MXFP4) repeat the bits: the
reduction order is fixed, and the last arrival leaves its arrival word
cleared.  Split calls on two streams at once repeat the bits of the same
calls made alone: each call draws its own workspace and tag."""
import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import oracle
import qk_inputs as qi
from gpu_util import assert_close, host_bits, run_fp8, run_mx, run_nvfp4, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[2, 3, 4], ids=lambda n: f"parts{n}")
def split(request, monkeypatch):
    monkeypatch.setenv("QK_TAIL_SPLIT", str(request.param))
    return request.param


def _sampled(out, ref_fn, M, N, what, seed=5, count=6):
    gots, refs = [], []
    for (m0, m1, n0, n1) in qi.sample_tiles(M, N, count, seed):
        gots.append(host_bits(out[m0:m1, n0:n1]).ravel())
        refs.append(ref_fn(m0, m1, n0, n1).ravel())
    assert not torch.isnan(out).any().item(), f"{what}: unwritten outputs"
    assert_close(np.concatenate(gots)[None, :], np.concatenate(refs)[None, :], what)


# (M, N, K): 256 x 256 pair tiles with 16 epilogue warps (K <= 2048, 15
# K-blocks) and with 8 (K > 2048, 18 K-blocks); 100 tiles, more than the
# pairs; 256 x 128 pair tiles (the narrow configuration wins at 600 x 776);
# 19 K-blocks, the last one 16 elements long
FP8_SHAPES = [(1536, 1792, 1920), (1536, 1792, 2304), (2560, 2560, 1920), (600, 776, 2304),
              (1536, 1792, 2320)]  # a ragged last K-block (16 of 128) in the last K-part


@pytest.mark.parametrize("shape", FP8_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fp8_tail_split_matches_oracle(split, shape):
    M, N, K = shape
    p = qi.fp8_problem(M, N, K, seed=M + K, bias=True)
    out = run_fp8(p)
    _sampled(out, lambda m0, m1, n0, n1: oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias, m0=m0, m1=m1,
                                                                  n0=n0, n1=n1), M, N, f"fp8 {shape} parts {split}")
    assert qk.device_status() == 0


@pytest.mark.parametrize("fmt,K", [(qi.FMT_MXFP8_E4M3, 1920), (qi.FMT_MXFP4_E2M1, 3840), (qi.FMT_MXFP4_E2M1, 3872)],
                         ids=["mxfp8", "mxfp4", "mxfp4-ragged-k"])
def test_mx_tail_split_matches_oracle(split, fmt, K):
    M, N = 600, 776
    p = qi.mx_problem(fmt, M, N, K, seed=K, bias=True)
    out = run_mx(p)
    _sampled(out, lambda m0, m1, n0, n1: oracle.gemm_mx(fmt, p.A, p.sA, p.B, p.sB, bias=p.bias, m0=m0, m1=m1,
                                                         n0=n0, n1=n1), M, N, f"fmt {fmt} parts {split}")
    assert qk.device_status() == 0


@pytest.mark.parametrize("K", [3840, 3872], ids=["k3840", "ragged-k"])
def test_nvfp4_tail_split_matches_oracle(split, K):
    M, N = 600, 776
    p = qi.nvfp4_problem(M, N, K, seed=3, bias=True)
    out = run_nvfp4(p)
    _sampled(out, lambda m0, m1, n0, n1: oracle.gemm_nvfp4(p.A, p.sA, p.B, p.sB, p.global_a, p.global_b, bias=p.bias,
                                                            m0=m0, m1=m1, n0=n0, n1=n1), M, N, f"nvfp4 parts {split}")
    assert qk.device_status() == 0


def test_tail_split_exact_small_integers(split):
    # E4M3 integers with unit scales: every K-part's partial and their sum are
    # exact integers in fp32, so no bit may differ from the oracle's
    M, N, K = 1536, 1792, 2304
    rng = np.random.default_rng(4)
    vals = np.array([0.0, 1.0, -1.0, 2.0, -2.0], np.float32)
    A = qi.encode_e4m3(vals[rng.integers(0, 5, (M, K))])
    B = qi.encode_e4m3(vals[rng.integers(0, 5, (N, K))])
    p = qi.Fp8Problem(A, B, np.ones(M, np.float32), np.ones(N, np.float32), None, M, N, K)
    out = run_fp8(p)
    for (m0, m1, n0, n1) in qi.sample_tiles(M, N, 6, 1):
        got = host_bits(out[m0:m1, n0:n1])
        ref = oracle.gemm_fp8_rowwise(A, B, p.sa, p.sb, m0=m0, m1=m1, n0=n0, n1=n1)
        assert np.array_equal(got, qi.to_bf16_bits(ref.astype(np.float32))), f"tile {m0}:{m1}, {n0}:{n1}"


def test_mxfp4_tail_split_exact_powers_of_two(split):
    # E2M1 elements in {0, +-1, +-2} and scales 2^e with |e| <= 3: every
    # scaled product is a multiple of 2^-6 and the sums stay far below 2^18
    M, N, K = 600, 776, 4096
    rng = np.random.default_rng(6)
    codes = np.array([0x0, 0x2, 0xA, 0x4, 0xC], np.uint8)  # 0, 1, -1, 2, -2
    a = codes[rng.integers(0, 5, (M, K))]
    b = codes[rng.integers(0, 5, (N, K))]
    A = (a[:, 0::2] | (a[:, 1::2] << 4)).astype(np.uint8)
    B = (b[:, 0::2] | (b[:, 1::2] << 4)).astype(np.uint8)
    sA = (127 + rng.integers(-3, 4, (M, K // 32))).astype(np.uint8)
    sB = (127 + rng.integers(-3, 4, (N, K // 32))).astype(np.uint8)
    p = qi.MxProblem(qi.FMT_MXFP4_E2M1, A, sA, B, sB, None, M, N, K)
    out = run_mx(p)
    for (m0, m1, n0, n1) in qi.sample_tiles(M, N, 6, 2):
        got = host_bits(out[m0:m1, n0:n1])
        ref = oracle.gemm_mx(p.fmt, A, sA, B, sB, m0=m0, m1=m1, n0=n0, n1=n1)
        assert np.array_equal(got, qi.to_bf16_bits(ref.astype(np.float32))), f"tile {m0}:{m1}, {n0}:{n1}"


def test_tail_split_repeats_and_replays(monkeypatch):
    # three parts (a short last one); plain calls, then one CUDA graph of the
    # call replayed three times into a NaN-filled output
    monkeypatch.setenv("QK_TAIL_SPLIT", "3")
    M, N, K = 1536, 1792, 2304
    p = qi.fp8_problem(M, N, K, seed=8)
    A, B, sa, sb = (to_dev(x) for x in (p.A, p.B, p.sa, p.sb))
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qk.gemm_fp8_rowwise(A, B, sa, sb, None, out)
    torch.cuda.synchronize()
    first = host_bits(out)
    for _ in range(2):
        out.fill_(float("nan"))
        qk.gemm_fp8_rowwise(A, B, sa, sb, None, out)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(out), first), "the fixed-order sum must repeat its bits"
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
        qk.gemm_fp8_rowwise(A, B, sa, sb, None, out)
    for replay in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(out), first), f"replay {replay} differs from the plain call"
    assert qk.device_status() == 0


@pytest.mark.parametrize("case", ["fp8-1024x7168x5120", "mxfp4-512x14336x10240", "nvfp4-512x14336x10240"])
def test_tail_split_default_rule(case):
    # without the switch: 112 pair tiles on 76 pairs (one full wave, then 36
    # tiles) with 40 K-blocks -> the last 36 tiles as two K-parts each
    kind, shape = case.split("-")
    M, N, K = (int(x) for x in shape.split("x"))
    if kind == "fp8":
        p = qi.fp8_problem(M, N, K, seed=2)
        out = run_fp8(p)
        ref_fn = lambda m0, m1, n0, n1: oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, p.sb, m0=m0, m1=m1, n0=n0, n1=n1)
    elif kind == "mxfp4":
        p = qi.mx_problem(qi.FMT_MXFP4_E2M1, M, N, K, seed=2)
        out = run_mx(p)
        ref_fn = lambda m0, m1, n0, n1: oracle.gemm_mx(p.fmt, p.A, p.sA, p.B, p.sB, m0=m0, m1=m1, n0=n0, n1=n1)
    else:
        p = qi.nvfp4_problem(M, N, K, seed=2)
        out = run_nvfp4(p)
        ref_fn = lambda m0, m1, n0, n1: oracle.gemm_nvfp4(p.A, p.sA, p.B, p.sB, p.global_a, p.global_b, m0=m0, m1=m1,
                                                          n0=n0, n1=n1)
    # the split tiles are the last 36 of the grouped-M raster: sample there too
    tiles = qi.sample_tiles(M, N, 4, 5) + [(M - 128, M, N - 128 * (1 + i), N - 128 * i) for i in range(1, 8, 3)]
    gots, refs = [], []
    for (m0, m1, n0, n1) in sorted(set(tiles)):
        gots.append(host_bits(out[m0:m1, n0:n1]).ravel())
        refs.append(ref_fn(m0, m1, n0, n1).ravel())
    assert not torch.isnan(out).any().item(), f"{case}: unwritten outputs"
    assert_close(np.concatenate(gots)[None, :], np.concatenate(refs)[None, :], case)
    assert qk.device_status() == 0


def test_tail_split_on_two_streams(monkeypatch):
    # split calls on two streams at once draw separate workspaces and tags:
    # each result repeats the bits of the same call made alone
    monkeypatch.setenv("QK_TAIL_SPLIT", "2")
    shapes = [(1536, 1792, 2304), (2560, 2560, 1920)]
    probs = [qi.fp8_problem(M, N, K, seed=20 + i) for i, (M, N, K) in enumerate(shapes)]
    devs = [[to_dev(x) for x in (p.A, p.B, p.sa, p.sb)] for p in probs]
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for (M, N, K) in shapes]
    alone = []
    for (A, B, sa, sb), out in zip(devs, outs):
        qk.gemm_fp8_rowwise(A, B, sa, sb, None, out)
        torch.cuda.synchronize()
        alone.append(host_bits(out))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for rep in range(3):
        for o in outs:
            o.fill_(float("nan"))
        torch.cuda.synchronize()
        for s, (A, B, sa, sb), out in zip(streams, devs, outs):
            with torch.cuda.stream(s):
                for _ in range(2):
                    qk.gemm_fp8_rowwise(A, B, sa, sb, None, out)
        torch.cuda.synchronize()
        for o, bits, shape in zip(outs, alone, shapes):
            assert np.array_equal(host_bits(o), bits), f"{shape} on two streams, repetition {rep}"
    assert qk.device_status() == 0


def test_mxfp4_tail_split_graph_replay(monkeypatch):
    # a block-scaled split call (scale pre-pass + GEMM) captured once and
    # replayed: every replay repeats the plain call's bits
    monkeypatch.setenv("QK_TAIL_SPLIT", "3")
    M, N, K = 600, 776, 3872
    p = qi.mx_problem(qi.FMT_MXFP4_E2M1, M, N, K, seed=31)
    A, sA, B, sB = (to_dev(x) for x in (p.A, p.sA, p.B, p.sB))
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qk.gemm_mx(p.fmt, A, sA, B, sB, None, out)
    torch.cuda.synchronize()
    first = host_bits(out)
    assert_close(first, oracle.gemm_mx(p.fmt, p.A, p.sA, p.B, p.sB), "plain split call")
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
        qk.gemm_mx(p.fmt, A, sA, B, sB, None, out)
    for replay in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(out), first), f"replay {replay} differs from the plain call"
    assert qk.device_status() == 0
