"""INT8 row/column-scaled GEMM with fp16 and fp32 outputs on the GPU against
the oracle: bit-exact.

comfy-kitchen PR #174, update "rebased onto v0.2.38": the page's INT8 kernel
specialization serves bf16, fp16 and fp32 outputs.  The fp32 epilogue value
x is the same as for bf16; fp16 rounds it to nearest even (+-inf beyond
65504), fp32 stores it.  Outputs are NaN-filled before each call so an
element the kernel never writes cannot pass; fp32 results are compared as
bit patterns (so -0 and +0 differ)."""
import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import oracle
import qk_inputs as qi
from gpu_util import bias_dev, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 8, 16),           # smallest legal problem
    (100, 136, 64),       # ragged M and N inside one tile
    (129, 264, 1040),     # one row and a 16-K chunk past the edges
    (300, 520, 2048),     # several tiles, two chunks
    (77, 2112, 5376),     # skinny M, deep K with a partial last chunk
]
DTYPES = {"fp16": torch.float16, "fp32": torch.float32}


def _run(p, dtype):
    out = torch.full((p.M, p.N), float("nan"), dtype=dtype, device="cuda")
    qk.gemm_int8_rowwise(to_dev(p.A), to_dev(p.B), to_dev(p.sa), to_dev(p.sb), bias_dev(p.bias), out)
    torch.cuda.synchronize()
    return out


def _bits(t):
    if t.dtype == torch.float32:
        return t.contiguous().view(torch.int32).cpu().numpy().view(np.uint32)
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _ref_bits(p, name, **kw):
    ref = oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias, out_dtype=name, **kw)
    return ref.view(np.uint32) if name == "fp32" else ref


def _assert_same(got, ref, what):
    bad = got != ref
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} differ; first: " + str(
        [(int(r), int(c), hex(int(got[r, c])), hex(int(ref[r, c]))) for r, c in np.argwhere(bad)[:4]])


@pytest.mark.parametrize("name", ["fp16", "fp32"])
@pytest.mark.parametrize("bias", [False, True], ids=["nobias", "bias"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_int8_out_types_match_oracle(shape, bias, name):
    M, N, K = shape
    p = qi.int8_problem(M, N, K, seed=M + N + K, bias=bias)
    _assert_same(_bits(_run(p, DTYPES[name])), _ref_bits(p, name), f"int8 {shape} bias={bias} {name}")


def test_int8_fp16_overflow_and_signed_zero():
    # 127*127*K beyond 65504 becomes +-inf in fp16 and stays finite in fp32;
    # -0 from the products survives without bias in both
    M, N, K = 128, 64, 64
    A = np.zeros((M, K), np.int8)
    A[:32] = 127
    A[32:64] = -127
    A[64:96, 0] = -3
    B = np.full((N, K), 127, np.int8)
    sa = np.ones(M, np.float32)
    sa[64:96] = -0.0
    sa[96:] = -2.0                                    # rows 96.. have acc = 0: 0 * -2 = -0
    sb = np.ones(N, np.float32)
    p = qi.Int8Problem(A, B, sa, sb, None, M, N, K)
    for name in ("fp16", "fp32"):
        got = _bits(_run(p, DTYPES[name]))
        ref = _ref_bits(p, name)
        if name == "fp16":
            assert np.all(ref[:32] == 0x7C00) and np.all(ref[32:64] == 0xFC00)
            assert np.all(ref[64:96] == 0x0000)       # (-381 * -0) = +0
            assert np.all(ref[96:] == 0x8000)          # -0 kept without bias
        else:
            assert np.all(ref[96:] == 0x80000000)
        _assert_same(got, ref, f"extremes {name}")


def test_int8_out_type_errors():
    lib = qk.load_library()
    assert lib.qk_gemm_int8_rowwise_out(None, None, None, None, None, None, 3, 1, 8, 16, None) == qk.QK_ERR_ARG
    x = torch.zeros((4, 16), dtype=torch.int8, device="cuda")
    s = torch.ones(4, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        qk.gemm_int8_rowwise(x, x, s, s, out_dtype=torch.float64)


def test_int8_fp32_full_size_sampled():
    # the headline shape with fp32 output, on sampled tiles and every edge tile
    M, N, K = 30000, 21504, 5376
    p = qi.int8_problem(M, N, K, seed=0, bias=True)
    out = _run(p, torch.float32)
    for (m0, m1, n0, n1) in qi.sample_tiles(M, N, 8, 5):
        got = _bits(out[m0:m1, n0:n1])
        ref = oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias, out_dtype="fp32",
                                       m0=m0, m1=m1, n0=n0, n1=n1).view(np.uint32)
        _assert_same(got, ref, f"tile {m0}:{m1}, {n0}:{n1}")
    del out
    torch.cuda.empty_cache()
