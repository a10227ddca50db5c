"""The few-row kernels between calls.

* Graph replay.  A captured stream-K call reuses its recorded epoch on every
  replay; the tile owners clear the flags they consumed, so a replay must
  give the bits of the uncaptured call.  Stream-K and cluster split-K calls
  are captured together in one CUDA graph, which is replayed three times;
  every replay's outputs equal the uncaptured calls' outputs bit for bit, and
  those match the oracle.
* Producer -> consumer.  The few-row kernels launch with programmatic
  dependent launch and wait for the previous kernel of the stream before
  their first global access.  A quantizer writes the activations and the GEMM
  reads them with nothing in between on the stream; the result matches the
  oracle on the quantizer's own outputs.
* The switches QK_FP8_SKINNY=1 and QK_MX_SKINNY=1 send few rows to the 2-SM
  tile kernels instead; their results match the oracle as well.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import oracle
import qk_inputs as qi
from gpu_util import assert_close, host_bits, run_fp8, run_mx, run_nvfp4, to_dev

pytestmark = pytest.mark.gpu


def test_fewrow_graph_replay_matches_plain_calls():
    # 168 and 224 weight tiles (no cluster wave fits: stream-K) and 17 tiles (cluster split-K)
    shapes = [(64, 21504, 2048), (48, 28672, 1024), (64, 2112, 7168)]
    probs = [qi.fp8_problem(M, N, K, seed=i + 1) for i, (M, N, K) in enumerate(shapes)]
    devs = [[to_dev(x) for x in (p.A, p.B, p.sa, p.sb)] for p in probs]
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for (M, N, K) in shapes]

    def calls():
        for (A, B, sa, sb), out in zip(devs, outs):
            qk.gemm_fp8_rowwise(A, B, sa, sb, None, out)

    calls()
    torch.cuda.synchronize()
    plain = [host_bits(o) for o in outs]
    for p, bits in zip(probs, plain):
        assert_close(bits, oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, p.sb), f"plain call {p.M}x{p.N}x{p.K}")
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
        calls()
    for replay in range(3):
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for o, bits, (M, N, K) in zip(outs, plain, shapes):
            assert np.array_equal(host_bits(o), bits), f"replay {replay} of {M}x{N}x{K} differs from the plain call"
    assert qk.device_status() == 0


@pytest.mark.parametrize("shape", [(64, 21504, 2048), (64, 2112, 7168)], ids=["streamk", "cluster"])
def test_quantizer_then_fewrow_gemm(shape):
    M, N, K = shape
    gen = torch.Generator(device="cuda")
    gen.manual_seed(M + N)
    x = torch.randn((M, K), generator=gen, device="cuda").to(torch.bfloat16)
    p = qi.fp8_problem(M, N, K, seed=7)
    B, sb = to_dev(p.B), to_dev(p.sb)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    q, sa = qk.quantize_ptpc(x)                   # writes the activations ...
    qk.gemm_fp8_rowwise(q, B, sa, sb, None, out)  # ... which the next kernel reads
    torch.cuda.synchronize()
    qh = q.cpu().numpy()
    sah = sa.cpu().numpy()
    assert_close(host_bits(out), oracle.gemm_fp8_rowwise(qh, p.B, sah, p.sb), f"quantize -> gemm {shape}")
    assert qk.device_status() == 0


def test_mx_quantizer_then_fewrow_gemm():
    M, N, K = 64, 7168, 2048
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    x = torch.randn((M, K), generator=gen, device="cuda").to(torch.bfloat16)
    p = qi.mx_problem(qi.FMT_MXFP4_E2M1, M, N, K, seed=13)
    B, sB = to_dev(p.B), to_dev(p.sB)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    A, sA = qk.quantize_mx(qi.FMT_MXFP4_E2M1, x)
    qk.gemm_mx(qi.FMT_MXFP4_E2M1, A, sA, B, sB, None, out)
    torch.cuda.synchronize()
    ref = oracle.gemm_mx(qi.FMT_MXFP4_E2M1, A.cpu().numpy(), sA.cpu().numpy(), p.B, p.sB)
    assert_close(host_bits(out), ref, "quantize_mx -> few-row MXFP4 gemm")
    assert qk.device_status() == 0


@pytest.mark.parametrize("shape", [(7, 4096, 4096), (100, 2112, 4096)], ids=["M7", "M100"])
def test_tile_kernel_forced_for_few_rows(monkeypatch, shape):
    # QK_FP8_SKINNY=1 / QK_MX_SKINNY=1: few rows through the 2-SM tile kernels
    # (one 256-row tile, mostly zero-filled rows) instead of the few-row kernels
    monkeypatch.setenv("QK_FP8_SKINNY", "1")
    monkeypatch.setenv("QK_MX_SKINNY", "1")
    M, N, K = shape
    p = qi.fp8_problem(M, N, K, seed=M, bias=True)
    assert_close(host_bits(run_fp8(p)), oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias), f"fp8 {shape}")
    for fmt in (qi.FMT_MXFP8_E4M3, qi.FMT_MXFP4_E2M1):
        q = qi.mx_problem(fmt, M, N, K, seed=M + 1)
        assert_close(host_bits(run_mx(q)), oracle.gemm_mx(fmt, q.A, q.sA, q.B, q.sB), f"fmt {fmt} {shape}")
    r = qi.nvfp4_problem(M, N, K, seed=M + 2)
    assert_close(host_bits(run_nvfp4(r)), oracle.gemm_nvfp4(r.A, r.sA, r.B, r.sB, r.global_a, r.global_b),
                 f"nvfp4 {shape}")
    assert qk.device_status() == 0
