// qk_fp8_blockscale.cu -- FP8 E4M3 GEMM with fp32 block scales: one per
// (row, 128-K block) of A and one per (128-row, 128-K) block of B (the
// "blockscale" kind of ROCm/mori PR #806's measurements, read with the
// DeepSeek-V3 block sizes).
//
// The tensor cores cannot apply fp32 scales, so every 128-K block is its own
// accumulation chunk: the MMAs (kind::f8f6f4) fill one of two 256-column TMEM
// accumulators per K-block while 16 epilogue warps drain the other into fp32
// sums in registers, sum += partial * (sa[m, g] * sb[n / 128, g]).
#include "qk_launch.cuh"

namespace qk {

// 128 x 256 tiles on one CTA, two 256-column accumulators, 16 epilogue warps
// with 64 columns each.  Measured alternatives, not built: 256 x 256 tiles on
// a CTA pair (the peer's MMA warp relays each accumulator release to the
// leader; 32 instead of 48 KB of operands per SM and chunk), 1651-1665
// against 1737 TFLOP/s at 16384 x 7168 x 2048 with 4 or 6 stages, and 1643
// with the peer's warps releasing straight on the leader's barrier; pair
// tiles of 256 x 128 with four 128-column accumulators, slower.  A cycle
// probe of the MMA thread puts this kernel's limit in the tensor pipe: with
// the epilogue draining the other accumulator meanwhile, each 128 x 256 x 32
// MMA takes ~281 cycles to issue (~1124 per 128-K block), about half the
// per-SM rate the pair MMAs reach without a drain beside them (~158 cycles
// per 256 x 256 x 32 pair MMA in the FP8 per-token kernel); the pair form
// here is limited by its accumulator turnover every 128 K.
using CfgFp8BlockscaleSingle = GemmCfg<Kind::F8BS, 256, 4, 2, false, 16, 1>;

template <class C>
static int launch_fp8_blockscale_cfg(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                                     const uint16_t* bias, uint16_t* out, int M, int N, int K,
                                     const DeviceInfo& dev, cudaStream_t stream) {
  CUtensorMap ta, tb;
  int st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, C::TMA_K, C::BM);
  if (st == QK_OK) st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, C::TMA_K, C::B_LOAD_ROWS);
  if (st != QK_OK) return st;
  GemmParams p{};
  plan_tiles<C>(p, M, N, K);
  p.sa = sa;
  p.sb = sb;
  p.scale_kb = ceil_div(K, 128);
  p.bias = bias;
  p.out = out;
  p.err = dev.err_word;
  p.timeout_ns = wait_timeout_ns();
  return launch_gemm<C>(ta, tb, ta, tb, p, dev, stream);
}

int launch_fp8_blockscale(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                          const uint16_t* bias, uint16_t* out, int M, int N, int K, const DeviceInfo& dev,
                          cudaStream_t stream) {
  return launch_fp8_blockscale_cfg<CfgFp8BlockscaleSingle>(A, B, sa, sb, bias, out, M, N, K, dev, stream);
}

}  // namespace qk

using namespace qk;

namespace {
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
}  // namespace

extern "C" int qk_gemm_fp8_blockscale(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                                      const uint16_t* bias, uint16_t* out, int64_t M, int64_t N, int64_t K,
                                      qk_stream_t stream) {
  if (M < 0 || N < 0 || K < 1) return QK_ERR_ARG;
  if (M == 0 || N == 0) return QK_OK;
  if (!A || !B || !sa || !sb || !out) return QK_ERR_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(out, 16) || (bias && !aligned(bias, 16)) || !aligned(sa, 4) ||
      !aligned(sb, 4))
    return QK_ERR_ALIGN;
  if (N % 8 != 0 || K % 16 != 0) return QK_ERR_ALIGN;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return QK_ERR_RANGE;
  if (((M + 255) / 256) * ((N + 255) / 256) > INT32_MAX) return QK_ERR_RANGE;
  int st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  return launch_fp8_blockscale(A, B, sa, sb, bias, out, static_cast<int>(M), static_cast<int>(N),
                               static_cast<int>(K), *dev, static_cast<cudaStream_t>(stream));
}
