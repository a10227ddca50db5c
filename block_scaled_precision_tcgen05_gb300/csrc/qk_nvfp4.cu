// qk_nvfp4.cu -- NVFP4 GEMM: packed E2M1 elements with one UE4M3 scale per 16
// K-elements and one fp32 scale per tensor, on tcgen05.mma
// kind::mxf4nvf4.block_scale.scale_vec::4X (four scale bytes per row per MMA
// of K = 64).  The per-tensor scales are the optional NVFP4 arguments of
// ROCm/aiter PR #6262's gemm_a4w4; the epilogue multiplies the fp32
// accumulator by their fp32 product before the bias.
#include "qk_sf_atoms.cuh"
#include "qk_fewrow_launch.cuh"

namespace qk {

// 256 x 256 tiles on a 2-SM CTA pair, five stages (32 KB of operands and 6 KB
// of scale atoms each), one accumulator drained by 16 epilogue warps into
// registers and released before the epilogue math.  Four stages measured 8%
// slower.  Measured alternatives, slower and not built: the pair with 8
// epilogue warps working from TMEM; 128 x 256 tiles on one CTA.
using CfgNvfp4PairDrain = GemmCfg<Kind::NVF4, 256, 5, 1, true, 16, 1>;
// fp16 / fp32 outputs (the same value, another rounding) run this tile kernel
// for every M (the few-row kernels write bf16 only): fp16 through the same
// staging blocks, fp32 with 16-byte stores straight from registers.
using CfgNvfp4F16 = GemmCfg<Kind::NVF4, 256, 5, 1, true, 16, 1, OutType::F16>;
using CfgNvfp4F32 = GemmCfg<Kind::NVF4, 256, 5, 1, true, 16, 0, OutType::F32>;

}  // namespace qk

using namespace qk;

namespace {
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Checks shared by both entry points.
int check_nvfp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const float* ga,
                const float* gb, const uint16_t* bias, const void* out, int64_t M, int64_t N, int64_t K, bool* empty) {
  *empty = false;
  if (M < 0 || N < 0 || K < 1) return QK_ERR_ARG;
  if (M == 0 || N == 0) {
    *empty = true;
    return QK_OK;
  }
  if (!A || !sA || !B || !sB || !out) return QK_ERR_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(out, 16) || (bias && !aligned(bias, 16)) ||
      (ga && !aligned(ga, 4)) || (gb && !aligned(gb, 4)))
    return QK_ERR_ALIGN;
  if (N % 8 != 0 || K % 32 != 0) return QK_ERR_ALIGN;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return QK_ERR_RANGE;
  if (((M + 127) / 128) * ((N + 31) / 32) > INT32_MAX) return QK_ERR_RANGE;
  return QK_OK;
}
}  // namespace

extern "C" int qk_gemm_nvfp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                             const float* ga, const float* gb, const uint16_t* bias, uint16_t* out, int64_t M,
                             int64_t N, int64_t K, qk_stream_t stream) {
  bool empty;
  int st = check_nvfp4(A, sA, B, sB, ga, gb, bias, out, M, N, K, &empty);
  if (st != QK_OK || empty) return st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  const auto s = static_cast<cudaStream_t>(stream);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  // few rows: the few-row kernels' NVFP4 mode where they are faster
  // (launch_fewrow_block_scaled, qk_fewrow_launch.cuh)
  FewRowArgs args;
  args.sfa = sA;
  args.sfw = sB;
  args.ga = ga;
  args.gb = gb;
  args.bias = bias;
  args.out = out;
  bool launched = false;
  st = launch_fewrow_block_scaled<3>(A, B, args, m, n, k, kKGemmNvfp4, *dev, s, &launched);
  if (launched) return st;
  return launch_block_scaled<CfgNvfp4PairDrain>(A, sA, B, sB, 1, ga, gb, bias, out, m, n, k, *dev, s);
}

extern "C" int qk_gemm_nvfp4_out(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                                 const float* ga, const float* gb, const uint16_t* bias, void* out, int out_type,
                                 int64_t M, int64_t N, int64_t K, qk_stream_t stream) {
  if (out_type != QK_OUT_BF16 && out_type != QK_OUT_FP16 && out_type != QK_OUT_FP32) return QK_ERR_ARG;
  if (out_type == QK_OUT_BF16)
    return qk_gemm_nvfp4(A, sA, B, sB, ga, gb, bias, static_cast<uint16_t*>(out), M, N, K, stream);
  bool empty;
  int st = check_nvfp4(A, sA, B, sB, ga, gb, bias, out, M, N, K, &empty);
  if (st != QK_OK || empty) return st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  const auto s = static_cast<cudaStream_t>(stream);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  if (out_type == QK_OUT_FP16)
    return launch_block_scaled<CfgNvfp4F16>(A, sA, B, sB, 1, ga, gb, bias, out, m, n, k, *dev, s);
  return launch_block_scaled<CfgNvfp4F32>(A, sA, B, sB, 1, ga, gb, bias, out, m, n, k, *dev, s);
}
