"""Pins of the CPU oracle to facts outside itself.

Each ``check_*`` takes a loaded oracle library handle and raises
AssertionError when the oracle disagrees with the fact it pins.  The same
checks run against the real oracle (test_oracle_pins.py) and against
deliberately broken copies of it (test_oracle_mutants.py), which shows that a
plausible mistake anywhere in the oracle fails at least one of them.

What each pin rests on:
* format anchor values of the OCP MX v1.0 element formats (1.0, largest
  normal, smallest normal/subnormal, NaN codes, the E2M1 value list),
  monotonicity and sign symmetry, and PyTorch's independent float8 casts;
* IEEE bf16 round-to-nearest-even, via PyTorch's float32 -> bfloat16 cast and
  the classic tie cases;
* the INT8 contraction against numpy's int64 matmul (a library routine) and
  against closed forms (identity B, constant extremes, hand-worked sums);
* the epilogue association (acc*sa)*sb the comfy-kitchen PR #174 update
  "Keep the cached INT8 epilogue scale order exact" fixes, signed zero
  without bias (same PR, "Preserve signed zero without INT8 bias"), and
  exact power-of-two scale invariance;
* the MX block structure against closed forms (constant elements with
  per-block scale codes), the exact doubling when every scale code of A
  grows by one, and a numpy float64 matmul of independently decoded values;
  the 32x32 B-scale form against a closed form over ragged 32-row groups and
  its exact reduction to the 1x32 form on row-repeated scales;
* NVFP4 (UE4M3 scales per 16 elements, per-tensor scales): the UE4M3 anchor
  values and PyTorch's float8_e4m3fn cast, a closed form over the 16-element
  blocks, a numpy matmul of independently decoded values, and the exact
  reduction to MXFP4 when the scales are powers of two shared by each pair
  of 16-blocks;
* FP8 blockscale (fp32 scales per 1x128 of A and 128x128 of B): a closed
  form over ragged K- and N-blocks, a numpy matmul of the blocks, and the
  reduction to the per-token x per-channel GEMM when the scales do not vary
  along K;
* the quantizers that feed the GEMMs: the MX shared exponent from
  torch.frexp, the elements through PyTorch's float8_e4m3fn cast or a brute
  force over the E2M1 values; the per-token scale and codes through PyTorch's
  fp32 divisions and float8_e4m3fn cast, hand-worked midpoint quotients, and
  searched rows where the fp32 rounding of the quotient (not a division in
  double, not a reciprocal multiply) decides the code.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import qk_inputs

E2M1_OCP_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP MX v1.0, E2M1 magnitudes


def _torch_e4m3(codes):
    return torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def _torch_ue8m0(codes):
    return torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e8m0fnu).double().numpy()


def _torch_bf16_bits(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _same_or_both_nan(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return bool(np.all((a == b) | (np.isnan(a) & np.isnan(b))))


# ---------------------------------------------------------------- formats

def check_e4m3_decode(lib):
    d = oracle.decode_e4m3(np.arange(256), lib)
    assert d[0x38] == 1.0
    assert d[0x7E] == 448.0
    assert d[0x08] == 2.0 ** -6
    assert d[0x01] == 2.0 ** -9
    assert d[0x07] == 7 * 2.0 ** -9
    assert d[0x00] == 0.0 and not np.signbit(d[0x00])
    assert d[0x80] == 0.0 and np.signbit(d[0x80])
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert np.sum(np.isnan(d)) == 2
    pos = d[:0x7F]
    assert np.all(np.diff(pos) > 0), "codes 0x00..0x7E must increase strictly"
    assert _same_or_both_nan(d[0x80:], -d[:0x80])
    assert _same_or_both_nan(d, _torch_e4m3(np.arange(256)))


def check_e2m1_decode(lib):
    d = oracle.decode_e2m1(np.arange(16), lib)
    assert list(d[:8]) == E2M1_OCP_VALUES
    assert list(-d[8:]) == E2M1_OCP_VALUES
    assert np.signbit(d[8])


def check_ue8m0_decode(lib):
    d = oracle.decode_ue8m0(np.arange(256), lib)
    assert d[127] == 1.0 and d[128] == 2.0 and d[126] == 0.5
    assert d[0] == 2.0 ** -127 and d[254] == 2.0 ** 127
    assert np.isnan(d[255])
    assert _same_or_both_nan(d, _torch_ue8m0(np.arange(256)))


def check_bf16_rne(lib):
    f = lambda bits: np.array([bits], np.uint32).view(np.float32)[0]
    assert oracle.f32_to_bf16([f(0x3F808000)], lib)[0] == 0x3F80  # tie, even stays
    assert oracle.f32_to_bf16([f(0x3F818000)], lib)[0] == 0x3F82  # tie, odd rounds up
    assert oracle.f32_to_bf16([f(0x3F808001)], lib)[0] == 0x3F81
    assert oracle.f32_to_bf16([f(0x7F7FFFFF)], lib)[0] == 0x7F80  # overflow -> +Inf
    assert oracle.f32_to_bf16([f(0x80000000)], lib)[0] == 0x8000  # -0 kept
    nanb = oracle.f32_to_bf16([np.float32(np.nan)], lib)[0]
    assert (nanb & 0x7F80) == 0x7F80 and (nanb & 0x7F) != 0
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2 ** 32, size=4000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    assert np.array_equal(oracle.f32_to_bf16(x, lib), _torch_bf16_bits(x))


def check_f16_rne(lib):
    # IEEE 754 binary16: 10 fraction bits, bias 15, subnormal spacing 2^-24, max 65504
    f16 = lambda v: int(oracle.f32_to_f16([v], lib)[0])
    assert f16(1.0) == 0x3C00 and f16(-2.0) == 0xC000 and f16(17.0) == 0x4C40
    assert f16(1 + 2 ** -11) == 0x3C00        # tie, even stays
    assert f16(1 + 3 * 2 ** -11) == 0x3C02    # tie, odd rounds up
    assert f16(65504.0) == 0x7BFF and f16(65519.99) == 0x7BFF
    assert f16(65520.0) == 0x7C00             # the midpoint to 2^16 rounds out of range
    assert f16(2.0 ** -14) == 0x0400 and f16(2.0 ** -24) == 0x0001
    assert f16(2.0 ** -25) == 0x0000 and f16(3 * 2.0 ** -25) == 0x0002  # subnormal ties to even
    assert f16(-0.0) == 0x8000 and f16(float("inf")) == 0x7C00
    nanh = f16(float("nan"))
    assert (nanh & 0x7C00) == 0x7C00 and (nanh & 0x3FF) != 0
    # every finite bf16 value, and random fp32 bit patterns, against numpy's conversion
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = qk_inputs.from_bf16_bits(bits)
    rng = np.random.default_rng(12)
    r = rng.integers(0, 2 ** 32, size=4000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x = np.concatenate([v[np.isfinite(v)], r[np.isfinite(r)]]).astype(np.float32)
    with np.errstate(over="ignore"):
        assert np.array_equal(oracle.f32_to_f16(x, lib), x.astype(np.float16).view(np.uint16))


def check_encoders(lib):
    # every finite code round-trips
    for c in range(256):
        v = oracle.decode_e4m3([c], lib)[0]
        if not np.isnan(v):
            assert oracle.encode_e4m3([v], lib)[0] == c
    for c in range(16):
        assert oracle.encode_e2m1([oracle.decode_e2m1([c], lib)[0]], lib)[0] == c
    # ties to even and saturation
    assert oracle.encode_e4m3([1.0625], lib)[0] == 0x38
    assert oracle.encode_e4m3([1.1875], lib)[0] == 0x3A
    assert oracle.encode_e4m3([2.0 ** -10], lib)[0] == 0x00
    assert oracle.encode_e4m3([15 * 2.0 ** -10], lib)[0] == 0x08
    assert oracle.encode_e4m3([470.0], lib)[0] == 0x7E
    assert oracle.encode_e4m3([-1e9], lib)[0] == 0xFE
    assert list(oracle.encode_e2m1([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 100.0], lib)) == [0, 2, 2, 4, 4, 6, 6, 7]
    # agrees with torch's float8_e4m3fn cast inside the finite range
    rng = np.random.default_rng(5)
    r = rng.standard_normal(3000) * 40
    r = r[np.abs(r) < 448]
    ours = oracle.encode_e4m3(r, lib)
    theirs = torch.tensor(r).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def _e2m1_code_nearest(y):
    """The E2M1 code nearest to y by brute force over the OCP value list, ties
    to the even code (the value with an even significand), saturating at 6."""
    mag = abs(float(y))
    best, best_err = 0, float("inf")
    for c, v in enumerate(E2M1_OCP_VALUES):
        err = abs(v - mag)
        if err < best_err or (err == best_err and c % 2 == 0):
            best, best_err = c, err
    return (0x8 if y < 0 else 0) | best


def check_mx_quantize_block(lib):
    codes, sc = oracle.mx_quantize_block(oracle.FMT_MXFP8_E4M3, np.ones(32), lib)
    assert sc == 127 - 8 and np.all(codes == 0x78)          # 1.0 * 2^8 = 256
    codes, sc = oracle.mx_quantize_block(oracle.FMT_MXFP4_E2M1, np.ones(32), lib)
    assert sc == 127 - 2 and np.all(codes == 0x6)           # 1.0 * 2^2 = 4
    codes, sc = oracle.mx_quantize_block(oracle.FMT_MXFP8_E4M3, np.zeros(32), lib)
    assert sc == 0 and np.all(codes == 0)
    # Independent pin: the shared exponent from torch.frexp (amax = f * 2^e,
    # f in [0.5, 1): floor(log2 amax) = e - 1), the elements x * 2^-s exactly
    # (a power-of-two scaling) and then PyTorch's float8_e4m3fn cast after
    # saturation at +-448, or the nearest E2M1 value by brute force.
    rng = np.random.default_rng(3)
    for fmt, emax in ((oracle.FMT_MXFP8_E4M3, 8), (oracle.FMT_MXFP4_E2M1, 2)):
        x = (rng.standard_normal((6, 32)) * np.exp(rng.uniform(-8, 8, (6, 1)))).astype(np.float32)
        x[0, 5] *= 30.0
        for r in range(6):
            c, s = oracle.mx_quantize_block(fmt, x[r], lib)
            xt = torch.from_numpy(x[r].copy())
            _, e = torch.frexp(xt.abs().max())
            sexp = min(max(int(e) - 1 - emax, -127), 127)
            assert s == sexp + 127
            y = torch.ldexp(xt, torch.tensor(-sexp, dtype=torch.int32))
            if fmt == oracle.FMT_MXFP8_E4M3:
                want = y.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            else:
                want = np.array([_e2m1_code_nearest(v) for v in y.numpy()], np.uint8)
            assert np.array_equal(c, want), (fmt, r)


def _e4m3_neighbours(t):
    """The E4M3 values just below and above t (t strictly inside the normal range)."""
    vals = sorted(v for v in oracle.decode_e4m3(np.arange(0x7F, dtype=np.uint8)) if np.isfinite(v))
    lo = max(v for v in vals if v < t)
    hi = min(v for v in vals if v > t)
    return lo, hi


def _division_rounding_cases():
    """Rows (amax, x) whose fp32 quotient x / fl(amax / 448) lands exactly on the
    midpoint of two E4M3 values while the exact quotient lies strictly on one
    side: rounding the fp32 quotient gives the even neighbour, rounding the
    exact quotient (a division in double) may give the other one.  Found by a
    seeded search; the exact side is decided with rationals."""
    from fractions import Fraction
    rng = np.random.default_rng(29)
    mids = [1.0625, 1.1875, 1.3125, 2.125, 2.375, 0.53125, 17.0, 19.0, 0.0390625]
    cases = []
    for _ in range(4000):
        amax = np.float32(rng.uniform(1.0, 100.0))
        s = np.float32(amax / np.float32(448.0))
        for t in mids:
            x0 = np.float32(s * np.float32(t))
            for k in range(-3, 4):
                x = x0
                for _ in range(abs(k)):
                    x = np.nextafter(x, np.float32(np.inf if k > 0 else -np.inf), dtype=np.float32)
                if not abs(x) < amax:
                    continue
                if np.float32(x / s) != np.float32(t):
                    continue
                exact = Fraction(float(x)) / Fraction(float(s))
                if exact == Fraction(t):
                    continue
                lo, hi = _e4m3_neighbours(t)
                cases.append((amax, x, t, lo if exact < Fraction(t) else hi))
        if len(cases) >= 12:
            break
    return cases


def _reciprocal_differs_cases():
    """Rows (amax, x) where the code of the fp32 quotient x / s differs from the
    code of x * fl(1 / s) (a reciprocal multiply, one rounding more), s =
    fl(amax / 448); found by a seeded search near E4M3 midpoints."""
    rng = np.random.default_rng(31)
    mids = [1.0625, 1.1875, 1.3125, 2.125, 2.375, 0.53125, 17.0, 19.0, 0.0390625, 5.25, 88.0]
    to_code = lambda v: int(torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])
    cases = []
    for _ in range(20000):
        amax = np.float32(rng.uniform(0.5, 300.0))
        s = np.float32(amax / np.float32(448.0))
        r = np.float32(np.float32(1.0) / s)
        for t in mids:
            x0 = np.float32(s * np.float32(t))
            for k in (-2, -1, 1, 2):
                x = x0
                for _ in range(abs(k)):
                    x = np.nextafter(x, np.float32(np.inf if k > 0 else -np.inf), dtype=np.float32)
                if not abs(x) < amax:
                    continue
                qd, qr = np.float32(x / s), np.float32(x * r)
                if qd != qr and to_code(qd) != to_code(qr):
                    cases.append((amax, x, to_code(qd)))
        if len(cases) >= 8:
            break
    return cases


def check_ptpc_quantize(lib):
    # closed forms: the row maximum maps to 448 exactly; an all-zero row takes scale 1
    x = np.array([[0.0, 1.0, -2.0, 7.0], [0.0, 0.0, 0.0, 0.0], [-3.5, 0.25, 1e-6, 3.5]], np.float32)
    codes, s = oracle.ptpc_quantize(x, lib)
    assert s[0] == np.float32(7.0) / np.float32(448.0) and s[1] == 1.0
    assert codes[0, 3] == 0x7E and codes[2, 0] == 0xFE and codes[2, 3] == 0x7E   # +-448
    assert np.all(codes[1] == 0)
    # hand-worked: amax 1344 gives s = 3 exactly; 3.1875 / 3 = 1.0625 and
    # 3.5625 / 3 = 1.1875 are exact E4M3 midpoints, which round to the even
    # neighbours 1.0 (0x38) and 1.25 (0x3A); amax 448 gives s = 1
    x = np.array([[1344.0, 3.1875, 3.5625, -3.1875], [448.0, 1.0625, 1.1875, -0.0]], np.float32)
    codes, s = oracle.ptpc_quantize(x, lib)
    assert s.tolist() == [3.0, 1.0]
    assert codes.tolist() == [[0x7E, 0x38, 0x3A, 0xB8], [0x7E, 0x38, 0x3A, 0x80]]
    # Independent pin (PyTorch): the fp32 row maximum, the fp32 division
    # amax / 448, the fp32 division x / s and PyTorch's float8_e4m3fn cast
    rng = np.random.default_rng(17)
    x = (rng.standard_normal((5, 300)) * np.exp(rng.uniform(-6, 6, (5, 1)))).astype(np.float32)
    x[2, :7] = 0.0
    codes, s = oracle.ptpc_quantize(x, lib)
    xt = torch.from_numpy(x)
    amax = xt.abs().amax(dim=1)
    st = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    assert st.dtype == torch.float32 and np.array_equal(s, st.numpy())
    want = (xt / st[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, want)
    # the division rounds in fp32 before the E4M3 rounding: quotients that
    # land on an E4M3 midpoint only after the fp32 rounding take the even
    # neighbour, as PyTorch's cast of the fp32 quotient does
    cases = _division_rounding_cases()
    assert len(cases) >= 6
    checked_other_side = 0
    for amax_v, xv, t, other in cases:
        row = np.array([[amax_v, xv]], np.float32)
        c, sv = oracle.ptpc_quantize(row, lib)
        tie_code = int(torch.tensor([t], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])
        assert int(c[0, 1]) == tie_code, (amax_v, xv, t)
        other_code = int(torch.tensor([other], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])
        checked_other_side += other_code != tie_code
    assert checked_other_side >= 3
    # a division, not a reciprocal multiply: rows where the two round apart
    rcp = _reciprocal_differs_cases()
    assert len(rcp) >= 4
    for amax_v, xv, code in rcp:
        c, _ = oracle.ptpc_quantize(np.array([[amax_v, xv]], np.float32), lib)
        assert int(c[0, 1]) == code, (amax_v, xv)


# ---------------------------------------------------------------- INT8

def check_int8_acc_vs_numpy(lib):
    rng = np.random.default_rng(21)
    for (M, N, K) in [(3, 5, 16), (17, 9, 48), (33, 40, 160)]:
        A = rng.integers(-128, 128, (M, K), dtype=np.int8)
        B = rng.integers(-128, 128, (N, K), dtype=np.int8)
        A[0, :] = -128
        B[0, :] = -128
        sa = np.ones(M, np.float32)
        sb = np.ones(N, np.float32)
        _, acc = oracle.gemm_int8_rowwise(A, B, sa, sb, return_acc=True, lib=lib)
        ref = A.astype(np.int64) @ B.astype(np.int64).T
        assert np.array_equal(acc, ref)
        # sub-region indexing agrees with the full result
        sub, acc2 = oracle.gemm_int8_rowwise(A, B, sa, sb, m0=1, m1=M, n0=2, n1=N, return_acc=True, lib=lib)
        assert np.array_equal(acc2, ref[1:, 2:])


def check_int8_hand_examples(lib):
    # (M,N,K) = (1,1,16): 1+2+...+16 = 136, exact in bf16
    A = np.arange(1, 17, dtype=np.int8).reshape(1, 16)
    B = np.ones((1, 16), np.int8)
    out = oracle.gemm_int8_rowwise(A, B, np.ones(1, np.float32), np.ones(1, np.float32), lib=lib)
    assert out[0, 0] == 0x4308  # 136.0
    # (2,3,32): rows a0 = +1 x32, a1 = alternating +2,-2; cols b0 = 1s, b1 = k mod 4, b2 = -1 for first 8 else 0
    a = np.zeros((2, 32), np.int8)
    a[0] = 1
    a[1, 0::2] = 2
    a[1, 1::2] = -2
    b = np.zeros((3, 32), np.int8)
    b[0] = 1
    b[1] = np.arange(32) % 4
    b[2, :8] = -1
    # by hand: acc[0] = [32, 48, -8]; acc[1] = [0, 2*(0-1+2-3)*8 = -32, 2*(-1+1)*4 = 0]
    _, acc = oracle.gemm_int8_rowwise(a, b, np.ones(2, np.float32), np.ones(3, np.float32), return_acc=True, lib=lib)
    assert acc.tolist() == [[32, 48, -8], [0, -32, 0]]


def check_int8_identity_and_extremes(lib):
    rng = np.random.default_rng(4)
    K = 64
    A = rng.integers(-128, 128, (7, K), dtype=np.int8)
    out = oracle.gemm_int8_rowwise(A, np.eye(K, dtype=np.int8), np.ones(7, np.float32), np.ones(K, np.float32), lib=lib)
    assert np.array_equal(out, _torch_bf16_bits(A.astype(np.float32)))  # int8 values are exact in bf16
    A = np.full((2, 1024), -128, np.int8)
    B = np.full((2, 1024), -128, np.int8)
    B[1] = 127
    _, acc = oracle.gemm_int8_rowwise(A, B, np.ones(2, np.float32), np.ones(2, np.float32), return_acc=True, lib=lib)
    assert acc[0, 0] == 1024 * 16384 and acc[0, 1] == -1024 * 16256
    # 2^31 does not fit in int32 -> the oracle refuses
    A = np.full((1, 131072), -128, np.int8)
    try:
        oracle.gemm_int8_rowwise(A, A, np.ones(1, np.float32), np.ones(1, np.float32), lib=lib)
    except ValueError:
        pass
    else:
        raise AssertionError("int32 overflow not reported")


def _find_association_witness():
    """A (acc, sa, sb) with bf16((acc*sa)*sb) != bf16(acc*(sa*sb)) in IEEE fp32."""
    rng = np.random.default_rng(12345)
    acc = rng.integers(-2 ** 24, 2 ** 24, 200000).astype(np.float32)
    sa = rng.uniform(1e-3, 1e-2, 200000).astype(np.float32)
    sb = rng.uniform(1e-3, 1e-2, 200000).astype(np.float32)
    left = _torch_bf16_bits((acc * sa) * sb)
    right = _torch_bf16_bits(acc * (sa * sb))
    idx = np.nonzero(left != right)[0]
    assert idx.size > 0
    return [(int(acc[i]), sa[i], sb[i], left[i], right[i]) for i in idx[:8]]


def _int8_rows_for_acc(acc):
    """One A row and one B row of int8 whose dot product is exactly ``acc``."""
    mag = abs(int(acc))
    q, r = divmod(mag, 127)
    q1, q0 = divmod(q, 127)          # mag = 127*127*q1 + 127*q0 + r
    K = ((q1 + 2 + 15) // 16) * 16
    a = np.zeros((1, K), np.int16)
    b = np.zeros((1, K), np.int16)
    a[0, :q1] = 127
    b[0, :q1] = 127
    a[0, q1], b[0, q1] = 127, q0
    a[0, q1 + 1], b[0, q1 + 1] = 1, r
    if acc < 0:
        b = -b
    return a.astype(np.int8), b.astype(np.int8)


def check_int8_epilogue_order(lib):
    for acc, sa, sb, left, right in _find_association_witness():
        a, b = _int8_rows_for_acc(acc)
        out, got = oracle.gemm_int8_rowwise(a, b, np.array([sa], np.float32), np.array([sb], np.float32),
                                            return_acc=True, lib=lib)
        assert got[0, 0] == acc
        assert out[0, 0] == left and out[0, 0] != right


def check_int8_signed_zero(lib):
    a = np.zeros((1, 16), np.int8)
    b = np.ones((1, 16), np.int8)
    out = oracle.gemm_int8_rowwise(a, b, np.array([-0.5], np.float32), np.array([0.25], np.float32), lib=lib)
    assert out[0, 0] == 0x8000  # 0 * (-0.5) = -0, kept without bias
    out = oracle.gemm_int8_rowwise(a, b, np.array([-0.5], np.float32), np.array([0.25], np.float32),
                                   bias=np.array([0x0000], np.uint16), lib=lib)
    assert out[0, 0] == 0x0000  # -0 + +0 = +0 under round-to-nearest
    a[0, 0] = -3
    out = oracle.gemm_int8_rowwise(a, b, np.array([1.0], np.float32), np.array([0.0], np.float32), lib=lib)
    assert out[0, 0] == 0x8000  # (-3 * 1) * (+0) = -0
    out = oracle.gemm_int8_rowwise(a, b, np.array([1.0], np.float32), np.array([1.0], np.float32),
                                   bias=np.array([0x3F80], np.uint16), lib=lib)
    assert out[0, 0] == _torch_bf16_bits(np.array([-2.0], np.float32))[0]


def check_int8_output_types(lib):
    # by hand: 1+2+...+16 = 136, times 0.5 and 0.25 = 17.0 exactly in every type
    A = np.arange(1, 17, dtype=np.int8).reshape(1, 16)
    B = np.ones((1, 16), np.int8)
    half, quarter = np.full(1, 0.5, np.float32), np.full(1, 0.25, np.float32)
    assert oracle.gemm_int8_rowwise(A, B, half, quarter, out_dtype="fp32", lib=lib)[0, 0] == 17.0
    assert oracle.gemm_int8_rowwise(A, B, half, quarter, out_dtype="fp16", lib=lib)[0, 0] == 0x4C40
    # beyond the fp16 range: 127*127*16 = 258064 is +Inf in fp16, finite in bf16
    A = np.full((1, 16), 127, np.int8)
    one = np.ones(1, np.float32)
    assert oracle.gemm_int8_rowwise(A, A, one, one, out_dtype="fp16", lib=lib)[0, 0] == 0x7C00
    assert oracle.gemm_int8_rowwise(A, A, one, one, out_dtype="fp32", lib=lib)[0, 0] == 258064.0
    # the three outputs are roundings of one fp32 value x (with and without bias)
    for bias in (False, True):
        p = qk_inputs.int8_problem(19, 40, 160, seed=23, bias=bias)
        x = oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias, out_dtype="fp32", lib=lib)
        assert x.dtype == np.float32
        bf = oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias, lib=lib)
        h = oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias, out_dtype="fp16", lib=lib)
        assert np.array_equal(bf, _torch_bf16_bits(x))
        with np.errstate(over="ignore"):
            assert np.array_equal(h, x.astype(np.float16).view(np.uint16))


def check_int8_pow2_invariance(lib):
    p = qk_inputs.int8_problem(24, 40, 96, seed=9, bias=False)
    base = oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, lib=lib)
    for k in (1, 3, -2):
        out = oracle.gemm_int8_rowwise(p.A, p.B, p.sa * np.float32(2.0 ** k), p.sb, lib=lib)
        expect = _torch_bf16_bits(qk_inputs.from_bf16_bits(base) * np.float32(2.0 ** k))
        assert np.array_equal(out, expect)
    # bias is added to the scaled product of row m and column n
    bias = qk_inputs.to_bf16_bits(np.linspace(-3, 3, 40).astype(np.float32))
    out = oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=bias, lib=lib)
    zero = oracle.gemm_int8_rowwise(np.zeros_like(p.A), p.B, p.sa, p.sb, bias=bias, lib=lib)
    assert np.array_equal(zero, np.broadcast_to(bias, zero.shape))
    assert not np.array_equal(out, base)


# ---------------------------------------------------------------- FP8 per-token x per-channel

def check_fp8_vs_numpy(lib):
    rng = np.random.default_rng(31)
    M, N, K = 9, 13, 96
    A = rng.integers(0, 256, (M, K), dtype=np.uint8)
    B = rng.integers(0, 256, (N, K), dtype=np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x11  # no NaN codes
    B[(B & 0x7F) == 0x7F] = 0x22
    sa = rng.uniform(0.5, 2, M).astype(np.float32)
    sb = rng.uniform(0.5, 2, N).astype(np.float32)
    bias = qk_inputs.to_bf16_bits(rng.standard_normal(N).astype(np.float32))
    ref = oracle.gemm_fp8_rowwise(A, B, sa, sb, bias=bias, lib=lib)
    acc = _torch_e4m3(A) @ _torch_e4m3(B).T  # exact: every partial sum fits in 53 bits
    expect = acc * sa.astype(np.float64)[:, None] * sb.astype(np.float64)[None, :] \
        + qk_inputs.from_bf16_bits(bias).astype(np.float64)[None, :]
    assert np.allclose(ref, expect, rtol=1e-15, atol=1e-12)
    sub = oracle.gemm_fp8_rowwise(A, B, sa, sb, bias=bias, m0=2, m1=7, n0=3, n1=13, lib=lib)
    assert np.array_equal(sub, ref[2:7, 3:13])


# ---------------------------------------------------------------- MX

def _mx_ones(fmt, M, N, K):
    one = 0x38 if fmt == oracle.FMT_MXFP8_E4M3 else 0x2
    if fmt == oracle.FMT_MXFP8_E4M3:
        A = np.full((M, K), one, np.uint8)
        B = np.full((N, K), one, np.uint8)
    else:
        A = np.full((M, K // 2), one | (one << 4), np.uint8)
        B = np.full((N, K // 2), one | (one << 4), np.uint8)
    return A, B


def check_mx_block_structure(lib):
    for fmt in (oracle.FMT_MXFP8_E4M3, oracle.FMT_MXFP4_E2M1):
        M, N, K = 3, 4, 256
        A, B = _mx_ones(fmt, M, N, K)
        nb = K // 32
        delta_a = np.arange(M)[:, None] * 2 + np.arange(nb)[None, :] - 3     # per row, per block
        delta_b = (np.arange(N)[:, None] - np.arange(nb)[None, :] % 3)       # per column, per block
        sA = (127 + delta_a).astype(np.uint8)
        sB = (127 + delta_b).astype(np.uint8)
        ref = oracle.gemm_mx(fmt, A, sA, B, sB, lib=lib)
        expect = np.zeros((M, N))
        for m in range(M):
            for n in range(N):
                expect[m, n] = sum(32.0 * 2.0 ** (delta_a[m, b] + delta_b[n, b]) for b in range(nb))
        assert np.array_equal(ref, expect)


def check_mx_scale_doubling(lib):
    for fmt in (oracle.FMT_MXFP8_E4M3, oracle.FMT_MXFP4_E2M1):
        p = qk_inputs.mx_problem(fmt, 8, 12, 128, seed=2)
        base = oracle.gemm_mx(fmt, p.A, p.sA, p.B, p.sB, lib=lib)
        up = oracle.gemm_mx(fmt, p.A, p.sA + 1, p.B, p.sB, lib=lib)
        assert np.array_equal(up, 2.0 * base)


def _dequant(fmt, X, sX, K):
    if fmt == oracle.FMT_MXFP8_E4M3:
        v = _torch_e4m3(X)
    else:
        v = np.asarray(E2M1_OCP_VALUES * 2)[qk_inputs.unpack_e2m1(X)]
        v = np.where(qk_inputs.unpack_e2m1(X) >= 8, -v, v)
    return v * np.repeat(_torch_ue8m0(sX), 32, axis=1)


def check_mx_vs_numpy(lib):
    for fmt in (oracle.FMT_MXFP8_E4M3, oracle.FMT_MXFP4_E2M1):
        p = qk_inputs.mx_problem(fmt, 10, 14, 192, seed=8, bias=True)
        ref = oracle.gemm_mx(fmt, p.A, p.sA, p.B, p.sB, bias=p.bias, lib=lib)
        expect = _dequant(fmt, p.A, p.sA, p.K) @ _dequant(fmt, p.B, p.sB, p.K).T \
            + qk_inputs.from_bf16_bits(p.bias).astype(np.float64)[None, :]
        assert np.allclose(ref, expect, rtol=1e-14, atol=1e-14)
        # nibble order: element 2i is the low nibble (0x21 -> 0.5 then 1.0)
    A = np.zeros((1, 16), np.uint8)
    A[0, 0] = 0x21
    B = np.zeros((1, 16), np.uint8)
    B[0, 0] = 0x02   # element 0 = 1.0, element 1 = 0
    ref = oracle.gemm_mx(oracle.FMT_MXFP4_E2M1, A, np.full((1, 1), 127, np.uint8), B,
                         np.full((1, 1), 127, np.uint8), lib=lib)
    assert ref[0, 0] == 0.5


# ---------------------------------------------------------------- NVFP4

def check_mx_b32(lib):
    """MX GEMM with B scales per 32x32 block (ROCm/mori PR #806, "What": B's
    scales [N/32, K/32]): a closed form over ragged 32-row groups, and the
    exact reduction to the 1x32 form when each group's scale row is repeated
    for its 32 rows."""
    for fmt in (oracle.FMT_MXFP8_E4M3, oracle.FMT_MXFP4_E2M1):
        M, N, K = 5, 72, 128            # groups of rows 0-31, 32-63, 64-71
        nb, ng = K // 32, (N + 31) // 32
        A, B = _mx_ones(fmt, M, N, K)
        da = (np.arange(M)[:, None] * 2 + np.arange(nb)[None, :]) % 5 - 2
        db = (np.arange(ng)[:, None] * 3 + np.arange(nb)[None, :] * 2) % 7 - 3
        sA = (127 + da).astype(np.uint8)
        sB32 = (127 + db).astype(np.uint8)
        ref = oracle.gemm_mx_b32(fmt, A, sA, B, sB32, lib=lib)
        n = np.arange(N)
        want = (32.0 * np.exp2(da[:, None, :] + db[n // 32][None, :, :])).sum(axis=2)
        assert np.array_equal(ref, want), fmt
        # random elements: equal to the 1x32 form on row-repeated scales, also
        # on a sub-region with a bias
        rng = np.random.default_rng(13)
        M, N, K = 7, 104, 256
        width = K if fmt == oracle.FMT_MXFP8_E4M3 else K // 2
        A = rng.integers(0, 256, (M, width), dtype=np.uint8)
        B = rng.integers(0, 256, (N, width), dtype=np.uint8)
        if fmt == oracle.FMT_MXFP8_E4M3:   # no NaN codes
            A[(A & 0x7F) == 0x7F] = 0x40
            B[(B & 0x7F) == 0x7F] = 0x40
        sA = rng.integers(110, 140, (M, K // 32), dtype=np.uint8)
        sB32 = rng.integers(110, 140, ((N + 31) // 32, K // 32), dtype=np.uint8)
        sB = np.repeat(sB32, 32, axis=0)[:N]
        bias = qk_inputs.bias_bits(N, 3)
        full = oracle.gemm_mx(fmt, A, sA, B, sB, bias=bias, lib=lib)
        assert np.array_equal(oracle.gemm_mx_b32(fmt, A, sA, B, sB32, bias=bias, lib=lib), full)
        sub = oracle.gemm_mx_b32(fmt, A, sA, B, sB32, bias=bias, m0=2, m1=6, n0=30, n1=97, lib=lib)
        assert np.array_equal(sub, full[2:6, 30:97])


def check_ue4m3_decode(lib):
    d = oracle.decode_ue4m3(np.arange(256), lib)
    assert d[0x38] == 1.0 and d[0x7E] == 448.0
    assert d[0x08] == 2.0 ** -6 and d[0x01] == 2.0 ** -9 and d[0x00] == 0.0
    assert np.isnan(d[0x7F]) and np.all(np.isnan(d[0x80:]))   # bit 7 is not part of the format
    assert np.array_equal(d[:0x7F], _torch_e4m3(np.arange(0x7F)))
    assert np.all(np.diff(d[:0x7F]) > 0)


def _nvfp4_ones(M, N, K):
    return np.full((M, K // 2), 0x22, np.uint8), np.full((N, K // 2), 0x22, np.uint8)   # E2M1 1.0 everywhere


def check_nvfp4_block_structure(lib):
    M, N, K = 3, 5, 128
    A, B = _nvfp4_ones(M, N, K)
    nb = K // 16
    rng = np.random.default_rng(17)
    sA = rng.integers(0x08, 0x7F, (M, nb)).astype(np.uint8)    # normal UE4M3 codes, varied mantissas
    sB = rng.integers(0x01, 0x7F, (N, nb)).astype(np.uint8)
    ga, gb = np.float32(0.75), np.float32(3.0)
    ref = oracle.gemm_nvfp4(A, sA, B, sB, ga, gb, lib=lib)
    dA, dB = _torch_e4m3(sA), _torch_e4m3(sB)
    expect = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            expect[m, n] = sum(16.0 * dA[m, b] * dB[n, b] for b in range(nb)) * 0.75 * 3.0
    assert np.allclose(ref, expect, rtol=1e-15, atol=0)


def _e2m1_values(packed):
    codes = qk_inputs.unpack_e2m1(packed)
    v = np.asarray(E2M1_OCP_VALUES * 2)[codes]
    return np.where(codes >= 8, -v, v)


def check_nvfp4_vs_numpy(lib):
    p = qk_inputs.nvfp4_problem(10, 14, 192, seed=8, bias=True)
    ref = oracle.gemm_nvfp4(p.A, p.sA, p.B, p.sB, p.global_a, p.global_b, bias=p.bias, lib=lib)
    a = _e2m1_values(p.A) * np.repeat(_torch_e4m3(p.sA), 16, axis=1)
    b = _e2m1_values(p.B) * np.repeat(_torch_e4m3(p.sB), 16, axis=1)
    expect = (a @ b.T) * float(np.float32(p.global_a)) * float(np.float32(p.global_b)) \
        + qk_inputs.from_bf16_bits(p.bias).astype(np.float64)[None, :]
    assert np.allclose(ref, expect, rtol=1e-13, atol=1e-13)
    sub = oracle.gemm_nvfp4(p.A, p.sA, p.B, p.sB, p.global_a, p.global_b, bias=p.bias, m0=3, m1=9, n0=2, n1=11,
                            lib=lib)
    assert np.array_equal(sub, ref[3:9, 2:11])


def check_nvfp4_reduces_to_mxfp4(lib):
    # power-of-two UE4M3 scales (mantissa 0), equal over each pair of 16-blocks,
    # with unit per-tensor scales: the same real numbers as MXFP4 with UE8M0
    rng = np.random.default_rng(23)
    M, N, K = 6, 9, 256
    A = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    ea = rng.integers(-6, 9, (M, K // 32))
    eb = rng.integers(-6, 9, (N, K // 32))
    to_ue4m3 = lambda e: ((e + 7) << 3).astype(np.uint8)             # 2^e, e in [-6, 8]
    sA16 = np.repeat(to_ue4m3(ea), 2, axis=1)
    sB16 = np.repeat(to_ue4m3(eb), 2, axis=1)
    nv = oracle.gemm_nvfp4(A, sA16, B, sB16, 1.0, 1.0, lib=lib)
    mx = oracle.gemm_mx(oracle.FMT_MXFP4_E2M1, A, (ea + 127).astype(np.uint8), B, (eb + 127).astype(np.uint8),
                        lib=lib)
    assert np.array_equal(nv, mx)


# ---------------------------------------------------------------- FP8 blockscale

def check_blockscale_block_structure(lib):
    M, N, K = 3, 300, 300             # ragged: K-blocks of 128, 128, 44; N-blocks of 128, 128, 44
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((N, K), 0x38, np.uint8)
    KB, NB = 3, 3
    sa = np.array([[2.0 ** g * (m + 1) for g in range(KB)] for m in range(M)], np.float32)
    sb = np.array([[(nb + 1) * (1 if g != 1 else 0.5) for g in range(KB)] for nb in range(NB)], np.float32)
    ref = oracle.gemm_fp8_blockscale(A, B, sa, sb, lib=lib)
    lens = [128, 128, 44]
    expect = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            expect[m, n] = sum(lens[g] * 2.0 ** g * (m + 1) * (n // 128 + 1) * (1 if g != 1 else 0.5)
                               for g in range(KB))
    assert np.array_equal(ref, expect)


def check_blockscale_vs_numpy(lib):
    rng = np.random.default_rng(37)
    M, N, K = 7, 140, 272
    A = rng.integers(0, 256, (M, K), dtype=np.uint8)
    B = rng.integers(0, 256, (N, K), dtype=np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x19
    B[(B & 0x7F) == 0x7F] = 0x2A
    KB, NB = 3, 2
    sa = rng.uniform(0.5, 2, (M, KB)).astype(np.float32)
    sb = rng.uniform(0.5, 2, (NB, KB)).astype(np.float32)
    bias = qk_inputs.to_bf16_bits(rng.standard_normal(N).astype(np.float32))
    ref = oracle.gemm_fp8_blockscale(A, B, sa, sb, bias=bias, lib=lib)
    a, b = _torch_e4m3(A), _torch_e4m3(B)
    expect = qk_inputs.from_bf16_bits(bias).astype(np.float64)[None, :].repeat(M, 0)
    for g in range(KB):
        ks = slice(128 * g, min(128 * g + 128, K))
        part = a[:, ks] @ b[:, ks].T
        expect = expect + part * sa[:, g].astype(np.float64)[:, None] \
            * np.repeat(sb[:, g].astype(np.float64), 128)[None, :N]
    # random E4M3 codes reach 448, so sums reach 1e6: compare at fp64 precision of that scale
    assert np.allclose(ref, expect, rtol=1e-14, atol=1e-14 * np.abs(expect).max())
    sub = oracle.gemm_fp8_blockscale(A, B, sa, sb, bias=bias, m0=1, m1=6, n0=100, n1=140, lib=lib)
    assert np.array_equal(sub, ref[1:6, 100:140])


def check_blockscale_reduces_to_ptpc(lib):
    p = qk_inputs.fp8_problem(9, 260, 384, seed=5)
    c = np.float32(0.013)
    KB = 3
    sa = np.repeat(p.sa[:, None], KB, axis=1)
    sb = np.full((3, KB), c, np.float32)
    bs = oracle.gemm_fp8_blockscale(p.A, p.B, sa, sb, lib=lib)
    pt = oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, np.full(p.N, c, np.float32), lib=lib)
    # the same real number up to fp64 rounding (scaled per block vs once at the end)
    assert np.allclose(bs, pt, rtol=1e-13, atol=1e-14 * np.abs(pt).max())


ALL_CHECKS = [
    check_e4m3_decode, check_e2m1_decode, check_ue8m0_decode, check_bf16_rne, check_f16_rne, check_encoders,
    check_mx_quantize_block, check_ptpc_quantize, check_int8_acc_vs_numpy, check_int8_hand_examples,
    check_int8_identity_and_extremes, check_int8_epilogue_order, check_int8_signed_zero,
    check_int8_output_types, check_int8_pow2_invariance, check_fp8_vs_numpy, check_mx_block_structure,
    check_mx_scale_doubling, check_mx_vs_numpy, check_ue4m3_decode, check_nvfp4_block_structure,
    check_nvfp4_vs_numpy, check_nvfp4_reduces_to_mxfp4, check_blockscale_block_structure,
    check_blockscale_vs_numpy, check_blockscale_reduces_to_ptpc, check_mx_b32,
]
