// qk_fp8.cu -- FP8 E4M3 GEMM with per-token x per-channel fp32 scales
// (ROCm/aiter PR #6262 gemm_a8w8_bpreshuffle semantics; ROCm/mori PR #806
// "ptpc"), on tcgen05.mma kind::f8f6f4 with fp32 accumulation in TMEM.
#include "qk_launch.cuh"

#include "qk_skinny_kernel.cuh"
#include "qk_streamk_launch.cuh"

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

template <class C>
static int launch_fp8_cfg(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                          uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
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

// Few rows, few weight tiles: split-K over a cluster of S CTAs with a DSMEM
// reduction (qk_skinny_kernel.cuh), used when every tile's cluster fits on
// the GPU at once.
template <int MT, int S>
static int launch_skinny_cfg(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                             const uint16_t* bias, uint16_t* out, int M, int N, int K, const DeviceInfo& dev,
                             cudaStream_t stream, bool probe_only, int* fits) {
  using C = SkinnyCfg<MT, S, MT <= 64 ? 6 : 4>;
  auto kernel = qk_skinny_fp8_kernel<C>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return QK_ERR_CUDA;
  const int n_tiles = ceil_div(N, C::NT);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_tiles * S, 1, 1);
  cfg.blockDim = dim3(C::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (probe_only) {  // how many clusters of S fit at once (computed once per device)
    static int cached[64];  // value + 1; 0 = not yet known
    int& slot = cached[dev.device >= 0 && dev.device < 64 ? dev.device : 0];
    if (slot == 0) {
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      slot = n + 1;
    }
    *fits = slot - 1;
    return QK_OK;
  }
  CUtensorMap tw, ta;
  int st = encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, 128, C::NT);
  if (st == QK_OK) st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, 128, C::MT);
  if (st != QK_OK) return st;
  SkinnyParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_kb = ceil_div(K, C::K_ELEMS);
  p.kb_per_split = ceil_div(p.num_kb, S);
  p.sa = sa;
  p.sb = sb;
  p.bias = bias;
  p.out = out;
  p.err = dev.err_word;
  p.timeout_ns = wait_timeout_ns();
  LaunchTimer timer(kKGemmFp8, stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tw, ta, p);
  timer.done();
  if (e != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_CUDA;
  }
  count_launches(1);
  return QK_OK;
}

// Few rows (M <= 128): the stream-K weight-streaming kernel in its FP8
// per-token mode.
std::atomic<unsigned long long> g_streamk_epoch{0};

template <int MT>
static int launch_streamk(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                          uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  StreamKParams p{};
  p.sa = sa;
  p.sb = sb;
  p.bias = bias;
  p.out = out;
  return launch_streamk_cfg<StreamKCfg<MT, MT <= 64 ? 8 : 6>>(A, B, p, M, N, K, kKGemmFp8, dev, stream);
}

// Few rows: if the weight tiles times some split S in {8, 4, 2, 1} fit on the
// GPU in one wave of clusters, the cluster split-K kernel with the largest
// such S (one pass, on-chip reduction); otherwise stream-K, which keeps every
// SM streaming whatever the tile count.  QK_FP8_SKINNY: 1 = the 2-SM tile
// kernel, 2 = always stream-K, 3 = always cluster split-K.
template <int MT>
static int launch_skinny(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                         uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream, int variant) {
  const int n_tiles = ceil_div(N, 128);
  const int num_kb = ceil_div(K, 128);
  if (variant != 2) {
    for (int S : {8, 4, 2, 1}) {
      if (S > num_kb && S > 1) continue;
      int fits = 0;
      if (S == 8) launch_skinny_cfg<MT, 8>(A, B, sa, sb, bias, out, M, N, K, dev, stream, true, &fits);
      if (S == 4) launch_skinny_cfg<MT, 4>(A, B, sa, sb, bias, out, M, N, K, dev, stream, true, &fits);
      if (S == 2) launch_skinny_cfg<MT, 2>(A, B, sa, sb, bias, out, M, N, K, dev, stream, true, &fits);
      if (S == 1) launch_skinny_cfg<MT, 1>(A, B, sa, sb, bias, out, M, N, K, dev, stream, true, &fits);
      if (n_tiles > fits && !(variant == 3 && S == 1)) continue;
      switch (S) {
        case 8: return launch_skinny_cfg<MT, 8>(A, B, sa, sb, bias, out, M, N, K, dev, stream, false, nullptr);
        case 4: return launch_skinny_cfg<MT, 4>(A, B, sa, sb, bias, out, M, N, K, dev, stream, false, nullptr);
        case 2: return launch_skinny_cfg<MT, 2>(A, B, sa, sb, bias, out, M, N, K, dev, stream, false, nullptr);
        default: return launch_skinny_cfg<MT, 1>(A, B, sa, sb, bias, out, M, N, K, dev, stream, false, nullptr);
      }
    }
  }
  return launch_streamk<MT>(A, B, sa, sb, bias, out, M, N, K, dev, stream);
}

int launch_fp8_rowwise(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                       uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  const int v = kernel_variant("QK_FP8_SKINNY");
  if (M <= 64 && v != 1) return launch_skinny<64>(A, B, sa, sb, bias, out, M, N, K, dev, stream, v);
  if (M <= 128 && v != 1) return launch_skinny<128>(A, B, sa, sb, bias, out, M, N, K, dev, stream, v);
  if (K <= 2048) return launch_fp8_cfg<CfgFp8Drain>(A, B, sa, sb, bias, out, M, N, K, dev, stream);
  return launch_fp8_cfg<CfgFp8>(A, B, sa, sb, bias, out, M, N, K, dev, stream);
}

}  // namespace qk
