// qk_fp8.cu -- FP8 E4M3 GEMM with per-token x per-channel fp32 scales
// (ROCm/aiter PR #6262 gemm_a8w8_bpreshuffle semantics; ROCm/mori PR #806
// "ptpc"), on tcgen05.mma kind::f8f6f4 with fp32 accumulation in TMEM.
#include "qk_launch.cuh"

namespace qk {

// 256 x 256 tiles per CTA pair, two accumulators of 256 columns per SM.
using CfgFp8 = GemmCfg<Kind::F8, 256, 6, 2, true>;

int launch_fp8_rowwise(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                       uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  using C = CfgFp8;
  CUtensorMap ta, tb;
  int st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, C::TMA_K, C::BM);
  if (st == QK_OK) st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, C::TMA_K, C::B_ROWS);
  if (st != QK_OK) return st;
  GemmParams p{};
  plan_tiles<C>(p, M, N, K);
  p.sa = sa;
  p.sb = sb;
  p.bias = bias;
  p.out = out;
  p.err = dev.err_word;
  p.timeout_ns = wait_timeout_ns();
  return launch_gemm<C>(ta, tb, ta, tb, p, dev, stream);
}

}  // namespace qk
