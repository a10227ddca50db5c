// qk_fp8.cu -- FP8 E4M3 GEMM with per-token x per-channel fp32 scales
// (ROCm/aiter PR #6262 gemm_a8w8_bpreshuffle semantics; ROCm/mori PR #806
// "ptpc"), on tcgen05.mma kind::f8f6f4 with fp32 accumulation in TMEM.
#include "qk_launch.cuh"

#include "qk_fewrow_launch.cuh"

namespace qk {

// 256 x 256 tiles per CTA pair, two accumulators of 256 columns per SM, 8
// epilogue warps writing through shared-memory staging blocks and bulk
// tensor stores (with K as short as 1792 the epilogue sets the pace: 4 warps
// storing straight to global memory reach 0.55 of this configuration's rate).
using CfgFp8 = GemmCfg<Kind::F8, 256, 6, 2, true, 8, 1>;
// With K <= 2048 a tile's MMAs take about as long as its epilogue, so 16
// epilogue warps drain each accumulator into registers and release it before
// the epilogue math: 2945 / 3068 TFLOP/s against 2840 / 3026 at K = 1792
// (and 1% slower than CfgFp8 at K = 5376 and 8192).
using CfgFp8Drain = GemmCfg<Kind::F8, 256, 6, 2, true, 16, 1>;
// 256 x 128 tiles per CTA pair (each SM loads 24 KB per 128-K stage instead of
// 32 for half the work), eight stages, two 128-column accumulators: twice the
// tiles of CfgFp8, for problems whose 256 x 256 tiles leave pairs idle.
using CfgFp8Narrow = GemmCfg<Kind::F8, 128, 8, 2, true, 8, 1>;
// fp16 / fp32 outputs (the same x, another rounding): CfgFp8's tiles and ring
// with 16-bit or 32-bit staging blocks (the fp32 blocks of 4 KB still leave
// room for six stages)
using CfgFp8F16 = GemmCfg<Kind::F8, 256, 6, 2, true, 8, 1, OutType::F16>;
using CfgFp8F32 = GemmCfg<Kind::F8, 256, 6, 2, true, 8, 1, OutType::F32>;

// Time of a tile configuration in tile periods: whole waves of tiles over the
// SM pairs, plus the last partial wave, which the tail split (qk_launch.cuh)
// shortens to 1/S of a tile plus the partials' round trip (about 7 k-blocks).
static double tile_waves(long long tiles, long long slots, int num_kb) {
  const long long W = tiles / slots, R = tiles % slots;
  if (R == 0) return static_cast<double>(W);
  const int S = tail_split_parts(tiles, slots, num_kb);
  return static_cast<double>(W) + (S > 1 ? 1.0 / S + 7.0 / num_kb : 1.0);
}

// Whether 256 x 128 pair tiles finish sooner than 256 x 256 ones, a narrow
// tile's period costing about 3/4 of a wide one's per SM (24 against 32 KB of
// operands per k-block at the per-SM ingress that bounds both), with a 10%
// margin for the narrow tiles' extra epilogues.
static bool narrow_tiles_win(int M, int N, int K, const DeviceInfo& dev) {
  const long long pairs = dev.sm_count / 2;
  const long long mb = (M + 255) / 256;
  const int num_kb = (K + 127) / 128;
  const double wide = tile_waves(mb * ((N + 255) / 256), pairs, num_kb);
  const double narrow = tile_waves(mb * ((N + 127) / 128), pairs, num_kb);
  return narrow * 0.75 < wide * 0.9;
}

template <class C>
static int launch_fp8_cfg(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                          void* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  CUtensorMap ta, tb;
  int st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, C::TMA_K, C::BM);
  if (st == QK_OK) st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, C::TMA_K, C::B_LOAD_ROWS);
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

// Few rows (M <= 128): if the weight tiles times some split S in {8, 4, 2, 1}
// fit on the GPU in one wave of clusters, the cluster split-K kernel with the
// largest such S (one pass, on-chip reduction); if no split fits, stream-K,
// which keeps every SM streaming whatever the tile count
// (qk_fewrow_launch.cuh).  Tile kernel against cluster (event times, us):
// 64 x 8192 x 1280 14.3 / 12.3, 128 x 7168 x 2048 16.4 / 14.3, 32 x 4096 x
// 2048 16.4 / 11.3, 128 x 2112 x 7168 26.6 / 16.4, 16 x 7168 x 4096 20.5 /
// 16.4.  QK_FP8_SKINNY: 1 = the 2-SM tile kernel, 2 = always stream-K, 3 =
// always cluster split-K.  Returns QK_ERR_RANGE when the tile kernel should run.
std::atomic<unsigned long long> g_streamk_epoch{0};

template <int MT>
static int launch_fewrow_fp8(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                             const uint16_t* bias, uint16_t* out, int M, int N, int K, const DeviceInfo& dev,
                             cudaStream_t stream, int variant) {
  FewRowArgs args;
  args.sa = sa;
  args.sb = sb;
  args.bias = bias;
  args.out = out;
  if (variant != 2) {
    bool fits = false;
    const int st = launch_cluster<MT, 0>(A, B, args, M, N, K, kKGemmFp8, dev, stream, variant == 3, &fits);
    if (st != QK_ERR_RANGE) return st;
  }
  return launch_streamk<MT, 0>(A, B, args, M, N, K, kKGemmFp8, dev, stream);
}

int launch_fp8_rowwise(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                       uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  const int v = kernel_variant("QK_FP8_SKINNY");
  if (M <= 128 && v != 1) {
    const int st = M <= 64 ? launch_fewrow_fp8<64>(A, B, sa, sb, bias, out, M, N, K, dev, stream, v)
                           : launch_fewrow_fp8<128>(A, B, sa, sb, bias, out, M, N, K, dev, stream, v);
    if (st != QK_ERR_RANGE) return st;
  }
  if (narrow_tiles_win(M, N, K, dev)) return launch_fp8_cfg<CfgFp8Narrow>(A, B, sa, sb, bias, out, M, N, K, dev, stream);
  if (K <= 2048) return launch_fp8_cfg<CfgFp8Drain>(A, B, sa, sb, bias, out, M, N, K, dev, stream);
  return launch_fp8_cfg<CfgFp8>(A, B, sa, sb, bias, out, M, N, K, dev, stream);
}

// Output types other than bf16: the 2-SM tile kernel for every M (the
// few-row kernels write bf16 only).
int launch_fp8_rowwise_out(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                           void* out, int out_type, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  if (out_type == QK_OUT_FP32) return launch_fp8_cfg<CfgFp8F32>(A, B, sa, sb, bias, out, M, N, K, dev, stream);
  if (out_type == QK_OUT_FP16) return launch_fp8_cfg<CfgFp8F16>(A, B, sa, sb, bias, out, M, N, K, dev, stream);
  return launch_fp8_rowwise(A, B, sa, sb, bias, static_cast<uint16_t*>(out), M, N, K, dev, stream);
}

}  // namespace qk
