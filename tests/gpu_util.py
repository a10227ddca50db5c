"""Helpers for the GPU parity tests: device transfer, NaN-filled outputs, the
bit-exact and tolerance comparisons."""
from __future__ import annotations

import numpy as np
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import qk_inputs as qi

# MX / FP8 tolerance, before the bf16 output rounding (compared against the
# oracle's unrounded fp64 value): |gpu - ref| <= RTOL*|ref| + ATOL_RMS*rms(ref),
# and cosine similarity >= COS_MIN.
RTOL = 1e-2
ATOL_RMS = 1e-2
COS_MIN = 0.99999


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def bias_dev(bits):
    return None if bits is None else to_dev(np.asarray(bits).view(np.int16)).view(torch.bfloat16)


def nan_out(M, N):
    return torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")


def host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_int8(p, out=None):
    out = nan_out(p.M, p.N) if out is None else out
    qk.gemm_int8_rowwise(to_dev(p.A), to_dev(p.B), to_dev(p.sa), to_dev(p.sb), bias_dev(p.bias), out)
    torch.cuda.synchronize()
    return out


def run_fp8(p, out=None):
    out = nan_out(p.M, p.N) if out is None else out
    qk.gemm_fp8_rowwise(to_dev(p.A), to_dev(p.B), to_dev(p.sa), to_dev(p.sb), bias_dev(p.bias), out)
    torch.cuda.synchronize()
    return out


def run_mx(p, out=None):
    out = nan_out(p.M, p.N) if out is None else out
    qk.gemm_mx(p.fmt, to_dev(p.A), to_dev(p.sA), to_dev(p.B), to_dev(p.sB), bias_dev(p.bias), out)
    torch.cuda.synchronize()
    return out


def run_blockscale(p, out=None):
    out = nan_out(p.M, p.N) if out is None else out
    qk.gemm_fp8_blockscale(to_dev(p.A), to_dev(p.B), to_dev(p.sa), to_dev(p.sb), bias_dev(p.bias), out)
    torch.cuda.synchronize()
    return out


def run_nvfp4(p, out=None, global_scales=True):
    out = nan_out(p.M, p.N) if out is None else out
    ga = to_dev(np.array([p.global_a], np.float32)) if global_scales else None
    gb = to_dev(np.array([p.global_b], np.float32)) if global_scales else None
    qk.gemm_nvfp4(to_dev(p.A), to_dev(p.sA), to_dev(p.B), to_dev(p.sB), ga, gb, bias_dev(p.bias), out)
    torch.cuda.synchronize()
    return out


def assert_bit_exact(gpu_bits, ref_bits, what=""):
    gpu_bits = np.asarray(gpu_bits, np.uint16)
    ref_bits = np.asarray(ref_bits, np.uint16)
    bad = gpu_bits != ref_bits
    if bad.any():
        idx = np.argwhere(bad)
        sample = [(int(i), int(j), hex(int(gpu_bits[i, j])), hex(int(ref_bits[i, j]))) for i, j in idx[:8]]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outputs differ; first (row, col, gpu, ref): {sample}")


def tolerance_report(gpu_bits, ref):
    return tolerance_report_values(qi.from_bf16_bits(gpu_bits).astype(np.float64), ref)


def tolerance_report_values(g, ref):
    """The report on output values already widened to fp64 (fp16 / fp32 outputs)."""
    g = np.asarray(g, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = np.abs(g - ref)
    bound = RTOL * np.abs(ref) + ATOL_RMS * rms
    den = float(np.linalg.norm(g) * np.linalg.norm(ref))
    cos = float((g * ref).sum() / den) if den > 0 else (1.0 if not g.any() and not ref.any() else 0.0)
    return {"nan": int(np.isnan(g).sum()), "bad": int((~(err <= bound)).sum()), "max_rel_to_bound":
            float(np.nanmax(err / np.maximum(bound, 1e-300))) if err.size else 0.0, "cos": cos, "rms": rms}


def assert_close(gpu_bits, ref, what=""):
    r = tolerance_report(gpu_bits, ref)
    assert r["nan"] == 0 and r["bad"] == 0 and r["cos"] >= COS_MIN, f"{what}: {r}"
    return r


def assert_close_values(gpu_values, ref, what=""):
    r = tolerance_report_values(gpu_values, ref)
    assert r["nan"] == 0 and r["bad"] == 0 and r["cos"] >= COS_MIN, f"{what}: {r}"
    return r
