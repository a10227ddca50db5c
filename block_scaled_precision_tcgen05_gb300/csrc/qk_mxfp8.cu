// qk_mxfp8.cu -- MXFP8 (E4M3 elements, one UE8M0 scale per 32 K) GEMM on
// tcgen05.mma kind::mxf8f6f4.block_scale.scale_vec::1X.  The raw row-major
// [rows, K/32] scale bytes (ROCm/mori PR #806, "What") are staged per ring
// slot by the kernel's scale warp and moved to TMEM with tcgen05.cp.
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

// Few rows (M <= 128): the few-row kernels' MXFP8 mode (qk_fewrow_launch.cuh).
// Against the tile kernel (us): the cluster split-K kernel, when all tiles'
// clusters fit in one wave, wins with a deep enough K range per CTA (at least
// 6 K-blocks for M <= 64; S >= 4 for more rows) -- 64 x 2112 x 7168
// 16.8 / 33.9, 64 x 4096 x 4096 15.2 / 23.9 (S = 4), 16 x 7168 x 4096
// 18.6 / 24.6 and 1 x 7168 x 2048 12.6 / 18.1 (S = 2), 48 x 12288 x 2048
// 16.8 (S = 1; stream-K 22.8), 128 x 2112 x 7168 20.7 / 33.4 -- and loses
// with a short one:
// 64 x 8192 x 1280 (5 K-blocks per CTA) 17.0 / 15.4, 128 x 7168 x 2048 (S = 2)
// 22.8 / 17.3.  Otherwise the stream-K kernel wins for M <= 64 once the
// weight holds about ten units per SM: 64 x 21504 x 5376 37.2 / 49.8; with
// fewer units or 128 activation rows it loses (64 x 2112 x 7168: 43.7,
// 128 x 21504 x 5376: 51.5 / 49.7).  QK_MX_SKINNY: 1 = always the tile
// kernel, 2 = stream-K, 3 = cluster split-K, whenever M <= 128.
int launch_mxfp8(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const uint16_t* bias,
                 uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  const int skinny = kernel_variant("QK_MX_SKINNY");
  if (M <= 128 && skinny != 1) {
    FewRowArgs args;
    args.sfa = sA;
    args.sfw = sB;
    args.bias = bias;
    args.out = out;
    const long long units = static_cast<long long>(ceil_div(N, 128)) * ceil_div(K, 128);
    if (skinny == 2) {
      if (M <= 64) return launch_streamk<64, true>(A, B, args, M, N, K, kKGemmMxfp8, dev, stream);
      return launch_streamk<128, true>(A, B, args, M, N, K, kKGemmMxfp8, dev, stream);
    }
    bool fits = false;
    if (skinny == 3) {
      if (M <= 64) return launch_cluster<64, true>(A, B, args, M, N, K, kKGemmMxfp8, dev, stream, true, 1, 0, &fits);
      return launch_cluster<128, true>(A, B, args, M, N, K, kKGemmMxfp8, dev, stream, true, 1, 0, &fits);
    }
    if (M <= 64) {
      const int st = launch_cluster<64, true>(A, B, args, M, N, K, kKGemmMxfp8, dev, stream, false, 1,
                                              kClusterMinKb, &fits);
      if (st != QK_ERR_RANGE) return st;
      if (!fits && units >= 10LL * dev.sm_count)
        return launch_streamk<64, true>(A, B, args, M, N, K, kKGemmMxfp8, dev, stream);
    } else {
      const int st = launch_cluster<128, true>(A, B, args, M, N, K, kKGemmMxfp8, dev, stream, false,
                                               kClusterMinSplitWide, 0, &fits);
      if (st != QK_ERR_RANGE) return st;
    }
  }
  return launch_block_scaled<CfgMxfp8PairDrain>(A, sA, B, sB, 1, nullptr, nullptr, bias, out, M, N, K, dev, stream);
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
