"""GPU quantizers (bf16 -> MX E4M3/E2M1 + UE8M0, bf16 -> per-token E4M3 + fp32
scale) against the oracle's quantizers: codes and scales bit-exact.

The inputs mix the MXFP8 recipe's distribution (N(0,1) with 1% of entries
x20) with rows scaled over a wide exponent range, all-zero and negative-zero
blocks, bf16 subnormals and values near the bf16 maximum (saturation); one
per-token case runs every bf16 value through the quotient for a range of
scales."""
import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import oracle
import qk_inputs as qi

pytestmark = pytest.mark.gpu


def _inputs(rows, K, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, K)).astype(np.float32)
    x[rng.uniform(size=x.shape) < 0.01] *= 20.0
    x *= np.exp2(rng.integers(-40, 40, (rows, 1))).astype(np.float32)
    x[0, :32] = 0.0                      # an all-zero block
    x[1, 32:64] = -0.0                   # a negative-zero block
    x[2, :64] = np.float32(3e-40) * rng.standard_normal(64).astype(np.float32)   # subnormal
    x[3, 64:96] = np.float32(3.0e38) * np.sign(rng.standard_normal(32)).astype(np.float32)  # near bf16 max
    bits = qi.to_bf16_bits(x)
    return bits, qi.from_bf16_bits(bits)


def _dev_bf16(bits):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("fmt", [qi.FMT_MXFP8_E4M3, qi.FMT_MXFP4_E2M1], ids=["mxfp8", "mxfp4"])
def test_mx_quantize_matches_oracle(fmt):
    rows, K = 37, 1024
    bits, x = _inputs(rows, K, 5 + fmt)
    q, s = qk.quantize_mx(fmt, _dev_bf16(bits))
    torch.cuda.synchronize()
    q = q.cpu().numpy()
    s = s.cpu().numpy()
    ref_codes, ref_scales = oracle.mx_quantize(fmt, x)
    assert np.array_equal(s, ref_scales)
    got = q if fmt == qi.FMT_MXFP8_E4M3 else qi.unpack_e2m1(q)
    bad = np.argwhere(got != ref_codes)
    assert bad.size == 0, f"{len(bad)} codes differ, first (row, col, gpu, ref): " + str(
        [(int(r), int(c), hex(int(got[r, c])), hex(int(ref_codes[r, c]))) for r, c in bad[:6]])


@pytest.mark.parametrize("rows,K", [(41, 2048), (9, 8208), (6, 16400)],
                         ids=["row-in-4-registers", "row-in-8-registers", "row-read-twice"])
def test_ptpc_quantize_matches_oracle(rows, K):
    # rows up to 8192 / 16384 elements stay in 4 / 8 register vectors per thread between the two
    # passes; longer rows are read twice
    bits, x = _inputs(rows, K, 9)
    x[5] = 0.0                           # an all-zero row takes scale 1
    bits[5] = 0
    q, s = qk.quantize_ptpc(_dev_bf16(bits))
    torch.cuda.synchronize()
    ref_codes, ref_scales = oracle.ptpc_quantize(x)
    assert np.array_equal(s.cpu().numpy(), ref_scales)
    assert np.array_equal(q.cpu().numpy(), ref_codes)


def _all_bf16_up_to(amax_bits, tiny):
    """Every finite bf16 value with magnitude <= the given bf16 amax (both
    signs, both zeros); without `tiny`, none with 0 < |x| < 2^-60."""
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = qi.from_bf16_bits(codes)
    amax = float(qi.from_bf16_bits(np.array([amax_bits], np.uint16))[0])
    keep = np.isfinite(v) & (np.abs(v) <= amax)
    if not tiny:
        keep &= (v == 0) | (np.abs(v) >= 2.0 ** -60)
    return codes[keep]


@pytest.mark.parametrize("tiny", [False, True], ids=["reciprocal-range", "with-tiny"])
def test_ptpc_quantize_every_bf16_value(tiny):
    # Each row holds every bf16 value up to its amax, so for the row's scale s
    # every element's quotient x / s is checked, on both sides of each E4M3
    # rounding boundary.  The amax values span scales inside the reciprocal
    # path's range (2^-60 .. 2^60, rows whose elements all go through the
    # reciprocal and its two corrections) and outside it (the library
    # division), including its edges; one variant leaves out, the other
    # keeps, the elements below 2^-60, where the corrections' residuals stop
    # being exact and only the zero code of the tiny quotient must agree.
    rng = np.random.default_rng(17)
    exps = list(range(-70, 71, 7)) + [-58, -57, -52, 51, 52, 53, 60, 68]
    amax_vals = [np.float32(np.ldexp(1.0 + rng.uniform(), e)) for e in exps]
    amax_vals += [np.float32(448.0), np.float32(1.0), np.float32(np.ldexp(448.0, -60)),
                  np.float32(np.ldexp(448.0, 60)), np.float32(np.ldexp(449.0, -61))]
    amax_bits = [int(b) for b in qi.to_bf16_bits(np.array(amax_vals, np.float32))]
    rows = [_all_bf16_up_to(b, tiny) for b in amax_bits]
    K = (max(len(r) for r in rows) + 15) // 16 * 16
    bits = np.zeros((len(rows), K), np.uint16)
    for i, r in enumerate(rows):
        bits[i, :len(r)] = rng.permutation(r)
    q, s = qk.quantize_ptpc(_dev_bf16(bits))
    torch.cuda.synchronize()
    ref_codes, ref_scales = oracle.ptpc_quantize(qi.from_bf16_bits(bits))
    assert np.array_equal(s.cpu().numpy(), ref_scales)
    got = q.cpu().numpy()
    bad = np.argwhere(got != ref_codes)
    assert bad.size == 0, f"{len(bad)} codes differ, first (row, col, x, gpu, ref): " + str(
        [(int(r), int(c), float(qi.from_bf16_bits(bits[r:r + 1, c])[0]), hex(int(got[r, c])), hex(int(ref_codes[r, c])))
         for r, c in bad[:6]])


def test_quantize_then_gemm_matches_oracle_on_the_same_bytes():
    # the quantizers feed the GEMM: quantize on the GPU, multiply on the GPU, and
    # check the product against the oracle on the very bytes the GPU produced
    from gpu_util import assert_close, host_bits
    rng = np.random.default_rng(3)
    M, N, K = 200, 264, 512
    a = qi.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    b = qi.to_bf16_bits((0.02 * rng.standard_normal((N, K))).astype(np.float32))
    for fmt in (qi.FMT_MXFP8_E4M3, qi.FMT_MXFP4_E2M1):
        qa, sa = qk.quantize_mx(fmt, _dev_bf16(a))
        qb, sb = qk.quantize_mx(fmt, _dev_bf16(b))
        out = qk.gemm_mx(fmt, qa, sa, qb, sb)
        torch.cuda.synchronize()
        ref = oracle.gemm_mx(fmt, qa.cpu().numpy(), sa.cpu().numpy(), qb.cpu().numpy(), sb.cpu().numpy())
        assert_close(host_bits(out), ref, f"quantized fmt {fmt}")
    qa, sa = qk.quantize_ptpc(_dev_bf16(a))
    qb, sb = qk.quantize_ptpc(_dev_bf16(b))
    out = qk.gemm_fp8_rowwise(qa, qb, sa, sb)
    torch.cuda.synchronize()
    ref = oracle.gemm_fp8_rowwise(qa.cpu().numpy(), qb.cpu().numpy(), sa.cpu().numpy(), sb.cpu().numpy())
    assert_close(host_bits(out), ref, "quantized ptpc")


def test_quantize_argument_errors():
    x = torch.zeros((4, 48), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qk.QkError):
        qk.quantize_mx(qi.FMT_MXFP8_E4M3, x)          # K % 32 != 0
    lib = qk.load_library()
    assert lib.qk_quantize_mx(3, None, None, None, 1, 32, None) == qk.QK_ERR_ARG
    assert lib.qk_quantize_ptpc(None, None, None, 0, 32, None) == qk.QK_OK
