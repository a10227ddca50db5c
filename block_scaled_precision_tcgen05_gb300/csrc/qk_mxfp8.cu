// qk_mxfp8.cu -- MXFP8 (E4M3 elements, one UE8M0 scale per 32 K) GEMM on
// tcgen05.mma kind::mxf8f6f4.block_scale.scale_vec::1X.  The raw row-major
// [rows, K/32] scale bytes (ROCm/mori PR #806, "What") are rearranged once per
// call into the atoms tcgen05.cp reads (qk_sf_atoms.cuh), loaded by TMA with
// each ring stage and moved to TMEM by two copy warps; with few rows the
// few-row kernels' scale warps stage them on chip (qk_fewrow_scales.cuh).
#include "qk_sf_atoms.cuh"
#include "qk_fewrow_launch.cuh"

namespace qk {

// 256 x 256 tiles on a 2-SM CTA pair, six stages, one accumulator drained by
// 16 epilogue warps into registers (64 columns each) and released before the
// epilogue math; the output leaves in 32x16 staging blocks (1 KB each, so the
// sixth stage fits).  Measured alternatives, slower and not built: one CTA with
// 128 x 224 tiles and two TMEM accumulators beside the scale ring; the pair
// with 8 epilogue warps working from TMEM; one CTA with 128 x 256 tiles and
// one accumulator, whose epilogue stalls the MMAs.
using CfgMxfp8PairDrain = GemmCfg<Kind::MXF8, 256, 6, 1, true, 16, 1, OutType::BF16, 16>;
// fp16 / fp32 outputs (the same value, another rounding) run this tile kernel
// for every M (the few-row kernels write bf16 only): fp16 through the same
// 32x16 staging blocks, fp32 with 16-byte stores straight from registers
// (4 KB fp32 staging blocks for 16 warps would cost ring stages).
using CfgMxfp8F16 = GemmCfg<Kind::MXF8, 256, 6, 1, true, 16, 1, OutType::F16, 16>;
using CfgMxfp8F32 = GemmCfg<Kind::MXF8, 256, 6, 1, true, 16, 0, OutType::F32>;

// Few rows (M <= 128): the few-row kernels' MXFP8 mode where they are faster
// (launch_fewrow_block_scaled, qk_fewrow_launch.cuh, with the measurements).
int launch_mxfp8(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const uint16_t* bias,
                 uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  FewRowArgs args;
  args.sfa = sA;
  args.sfw = sB;
  args.bias = bias;
  args.out = out;
  bool launched = false;
  const int st = launch_fewrow_block_scaled<1>(A, B, args, M, N, K, kKGemmMxfp8, dev, stream, &launched);
  if (launched) return st;
  return launch_block_scaled<CfgMxfp8PairDrain>(A, sA, B, sB, 1, nullptr, nullptr, bias, out, M, N, K, dev, stream);
}

int launch_mxfp8_out(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const uint16_t* bias,
                     void* out, int out_type, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  if (out_type == QK_OUT_FP16)
    return launch_block_scaled<CfgMxfp8F16>(A, sA, B, sB, 1, nullptr, nullptr, bias, out, M, N, K, dev, stream);
  if (out_type == QK_OUT_FP32)
    return launch_block_scaled<CfgMxfp8F32>(A, sA, B, sB, 1, nullptr, nullptr, bias, out, M, N, K, dev, stream);
  return launch_mxfp8(A, sA, B, sB, bias, static_cast<uint16_t*>(out), M, N, K, dev, stream);
}

// B scales per 32x32 block (ROCm/mori PR #806's mxfp8_raw form): the scale-atom
// pre-pass places each 32-row group's scale bytes at all 32 rows; the tile
// kernel runs for every M (the few-row kernels stage per-row scales only).
int launch_mxfp8_b32(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB32,
                     const uint16_t* bias, uint16_t* out, int M, int N, int K, const DeviceInfo& dev,
                     cudaStream_t stream) {
  return launch_block_scaled<CfgMxfp8PairDrain>(A, sA, B, sB32, 32, nullptr, nullptr, bias, out, M, N, K, dev,
                                                stream);
}

}  // namespace qk
