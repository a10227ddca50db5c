// qk_nvfp4.cu -- NVFP4 GEMM: packed E2M1 elements with one UE4M3 scale per 16
// K-elements and one fp32 scale per tensor, on tcgen05.mma
// kind::mxf4nvf4.block_scale.scale_vec::4X (four scale bytes per row per MMA
// of K = 64).  The per-tensor scales are the optional NVFP4 arguments of
// ROCm/aiter PR #6262's gemm_a4w4; the epilogue multiplies the fp32
// accumulator by their fp32 product before the bias.
#include "qk_launch.cuh"

namespace qk {

// 256 x 256 tiles on a 2-SM CTA pair, four stages, one accumulator drained
// by 16 epilogue warps into registers and released before the epilogue math.
// Measured alternatives, slower and not built: the pair with five stages and
// 8 epilogue warps working from TMEM; 128 x 256 tiles on one CTA, where the
// 16 scale bytes per row per stage (6 KB of shared memory and 48 TMEM columns
// per slot) leave room for three stages.
using CfgNvfp4PairDrain = GemmCfg<Kind::NVF4, 256, 4, 1, true, 16, 1>;

template <class C>
static int launch_nvfp4_cfg(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                            const float* ga, const float* gb, const uint16_t* bias, uint16_t* out, int M, int N,
                            int K, const DeviceInfo& dev, cudaStream_t stream) {
  CUtensorMap ta, tb;
  const uint64_t kb = static_cast<uint64_t>(K) / 2;  // bytes per row
  int st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, kb, M, kb, C::TMA_K, C::BM);
  if (st == QK_OK) st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kb, N, kb, C::TMA_K, C::B_LOAD_ROWS);
  if (st != QK_OK) return st;
  GemmParams p{};
  plan_tiles<C>(p, M, N, K);
  p.bias = bias;
  p.out = out;
  p.sA = sA;
  p.sB = sB;
  p.sf_cols = K / 16;
  p.ga = ga;
  p.gb = gb;
  p.err = dev.err_word;
  p.timeout_ns = wait_timeout_ns();
  // Raw scale rows (K/16 bytes) through TMA when the pitch and base addresses
  // are 16-byte multiples, through cp.async at 4-byte multiples, else loads.
  CUtensorMap tsa = ta, tsb = tb;
  const bool a16 = ((reinterpret_cast<uintptr_t>(sA) | reinterpret_cast<uintptr_t>(sB)) & 15u) == 0;
  const bool a4 = ((reinterpret_cast<uintptr_t>(sA) | reinterpret_cast<uintptr_t>(sB)) & 3u) == 0;
  p.sf_mode = (p.sf_cols % 16 == 0 && a16) ? kSfTma : ((p.sf_cols % 4 == 0 && a4) ? kSfAsync : kSfLoads);
  if (p.sf_mode == kSfTma) {
    st = encode_tmap_2d_plain(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, sA, p.sf_cols, M, p.sf_cols, 16, C::BM);
    if (st == QK_OK)
      st = encode_tmap_2d_plain(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, sB, p.sf_cols, N, p.sf_cols, 16, C::BN);
    if (st != QK_OK) return st;
  }
  return launch_gemm<C>(ta, tb, tsa, tsb, p, dev, stream);
}

}  // namespace qk

using namespace qk;

namespace {
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
}  // namespace

extern "C" int qk_gemm_nvfp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                             const float* ga, const float* gb, const uint16_t* bias, uint16_t* out, int64_t M,
                             int64_t N, int64_t K, qk_stream_t stream) {
  if (M < 0 || N < 0 || K < 1) return QK_ERR_ARG;
  if (M == 0 || N == 0) return QK_OK;
  if (!A || !sA || !B || !sB || !out) return QK_ERR_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(out, 16) || (bias && !aligned(bias, 16)) ||
      (ga && !aligned(ga, 4)) || (gb && !aligned(gb, 4)))
    return QK_ERR_ALIGN;
  if (N % 8 != 0 || K % 32 != 0) return QK_ERR_ALIGN;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return QK_ERR_RANGE;
  if (((M + 127) / 128) * ((N + 31) / 32) > INT32_MAX) return QK_ERR_RANGE;
  int st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  const auto s = static_cast<cudaStream_t>(stream);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  return launch_nvfp4_cfg<CfgNvfp4PairDrain>(A, sA, B, sB, ga, gb, bias, out, m, n, k, *dev, s);
}
