// qk_mxfp4.cu -- MXFP4 (packed E2M1 elements, one UE8M0 scale per 32 K) GEMM
// on tcgen05.mma kind::mxf4.block_scale.scale_vec::2X, which reads the
// packed 4-bit operands directly (ROCm/FlyDSL PR #990: MXFP4 with per-1x32
// scales).  Operands are [rows, K/2] bytes, element 2i in the low nibble.
#include "qk_sf_atoms.cuh"
#include "qk_fewrow_launch.cuh"

namespace qk {

// 256 x 256 tiles on a 2-SM CTA pair (each SM loads half of B: 32 KB of
// operands per 256-K stage instead of 48), six stages, one accumulator that
// 16 epilogue warps drain into registers (64 columns each) and release before
// the epilogue math, so the next tile's MMAs start after the drain.  The
// output leaves in 32x16 staging blocks (1 KB), which leaves room for the
// sixth stage (no room for alignment slack: the kernel checks its base).  Each CTA
// loads the scale atoms of its own A rows and of all the tile's B rows; the
// leader's two copy threads fill both CTAs' TMEM with cta_group::2 copies
// beside the MMAs.  Measured alternatives (the same pair
// with 8 epilogue warps working from TMEM; one CTA with 128 x 256 tiles) were
// slower and are not built.
using CfgMxfp4PairDrain = GemmCfg<Kind::MXF4, 256, 6, 1, true, 16, 1, OutType::BF16, 16>;
// fp16 / fp32 outputs (the same value, another rounding) run this tile kernel
// for every M (the few-row kernels write bf16 only): fp16 through the same
// 32x16 staging blocks, fp32 with 16-byte stores straight from registers
// (4 KB fp32 staging blocks for 16 warps would cost ring stages).
using CfgMxfp4F16 = GemmCfg<Kind::MXF4, 256, 6, 1, true, 16, 1, OutType::F16, 16>;
using CfgMxfp4F32 = GemmCfg<Kind::MXF4, 256, 6, 1, true, 16, 0, OutType::F32>;

// Few rows (M <= 128): the few-row kernels' MXFP4 mode where they are
// faster (launch_fewrow_block_scaled, qk_fewrow_launch.cuh).
int launch_mxfp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const uint16_t* bias,
                 uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  FewRowArgs args;
  args.sfa = sA;
  args.sfw = sB;
  args.bias = bias;
  args.out = out;
  bool launched = false;
  const int st = launch_fewrow_block_scaled<2>(A, B, args, M, N, K, kKGemmMxfp4, dev, stream, &launched);
  if (launched) return st;
  return launch_block_scaled<CfgMxfp4PairDrain>(A, sA, B, sB, 1, nullptr, nullptr, bias, out, M, N, K, dev, stream);
}

int launch_mxfp4_out(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const uint16_t* bias,
                     void* out, int out_type, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  if (out_type == QK_OUT_FP16)
    return launch_block_scaled<CfgMxfp4F16>(A, sA, B, sB, 1, nullptr, nullptr, bias, out, M, N, K, dev, stream);
  if (out_type == QK_OUT_FP32)
    return launch_block_scaled<CfgMxfp4F32>(A, sA, B, sB, 1, nullptr, nullptr, bias, out, M, N, K, dev, stream);
  return launch_mxfp4(A, sA, B, sB, bias, static_cast<uint16_t*>(out), M, N, K, dev, stream);
}

int launch_mxfp4_b32(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB32,
                     const uint16_t* bias, uint16_t* out, int M, int N, int K, const DeviceInfo& dev,
                     cudaStream_t stream) {
  return launch_block_scaled<CfgMxfp4PairDrain>(A, sA, B, sB32, 32, nullptr, nullptr, bias, out, M, N, K, dev,
                                                stream);
}

}  // namespace qk
