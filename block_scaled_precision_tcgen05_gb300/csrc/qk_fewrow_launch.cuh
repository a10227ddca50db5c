// qk_fewrow_launch.cuh -- host launch of the few-row kernels (M <= 128):
// the cluster split-K kernel (qk_skinny_kernel.cuh) and the stream-K kernel
// (qk_streamk_kernel.cuh), each in its FP8 per-token and MXFP8 modes, and
// the choice between them.
#pragma once
#include <atomic>

#include "qk_launch.cuh"
#include "qk_skinny_kernel.cuh"
#include "qk_streamk_kernel.cuh"

namespace qk {

// The operation's operands beyond A and B: per-token / per-channel fp32
// scales (FP8) or UE8M0 scale rows (MXFP8), bias and output.
struct FewRowArgs {
  const float* sa = nullptr;
  const float* sb = nullptr;
  const uint8_t* sfa = nullptr;
  const uint8_t* sfw = nullptr;
  const uint16_t* bias = nullptr;
  uint16_t* out = nullptr;
};

// One CTA per SM, launched cooperatively so that all CTAs are resident while
// owners wait for their contributors' partials.  The partials and flags come
// from the stream-ordered workspace pool; each call gets a fresh 64-bit epoch
// (shared by both modes, since they draw on the same pool), so flags left in
// reused memory by earlier calls never read as finished.
extern std::atomic<unsigned long long> g_streamk_epoch;

template <class C>
int launch_streamk_cfg(const uint8_t* A, const uint8_t* B, const FewRowArgs& args, int M, int N, int K,
                       int kernel_kind, const DeviceInfo& dev, cudaStream_t stream) {
  auto kernel = qk_streamk_fp8_kernel<C>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return QK_ERR_CUDA;
  const int n_tiles = ceil_div(N, C::NT);
  const int num_kb = ceil_div(K, C::K_ELEMS);
  const long long units = static_cast<long long>(n_tiles) * num_kb;
  const int G = static_cast<int>(units < dev.sm_count ? units : dev.sm_count);
  CUtensorMap tw, ta;
  int st = encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, C::K_ELEMS, C::NT);
  if (st == QK_OK) st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, C::K_ELEMS, C::MT);
  if (st != QK_OK) return st;
  const size_t part_bytes = static_cast<size_t>(G) * C::MT * C::NT * sizeof(float);
  void* ws = nullptr;
  if (cudaMallocFromPoolAsync(&ws, part_bytes + static_cast<size_t>(G) * 4 * sizeof(unsigned long long), dev.pool,
                              stream) != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_NOMEM;
  }
  StreamKParams p{};
  p.sa = args.sa;
  p.sb = args.sb;
  p.sfa = args.sfa;
  p.sfw = args.sfw;
  p.sf_cols = K / 32;
  p.bias = args.bias;
  p.out = args.out;
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_kb = num_kb;
  p.units = units;
  p.partials = static_cast<float*>(ws);
  p.flags = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + part_bytes);
  // the epilogue's bulk stores: the output in [OUT_ROWS x 32] boxes, the
  // partials ([G * MT, 128] fp32) in 32 x 32 boxes
  CUtensorMap tout, tpart;
  st = encode_tmap_2d_plain(&tout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, args.out, N, M,
                            static_cast<uint64_t>(N) * 2, 32, C::OUT_ROWS);
  if (st == QK_OK)
    st = encode_tmap_2d_plain(&tpart, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.partials, C::NT,
                              static_cast<uint64_t>(G) * C::MT, C::NT * 4, 32, 32);
  if (st != QK_OK) {
    cudaFreeAsync(ws, stream);
    return st;
  }
  // a 64-bit value no earlier call used (odd multiplier: a bijection of the counter)
  p.epoch = (g_streamk_epoch.fetch_add(1) + 1) * 0x9E3779B97F4A7C15ull;
  p.err = dev.err_word;
  p.timeout_ns = wait_timeout_ns();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G, 1, 1);
  cfg.blockDim = dim3(C::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  // the prologue may overlap the previous kernel of the stream (the kernel
  // waits for it before touching memory)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  LaunchTimer timer(kernel_kind, stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tw, ta, tout, tpart, p);
  timer.done();
  const cudaError_t f = cudaFreeAsync(ws, stream);
  if (e != cudaSuccess || f != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_CUDA;
  }
  count_launches(1);
  return QK_OK;
}

// Split-K over a cluster of S CTAs with a DSMEM reduction.  With probe_only
// it only reports (in *fits) how many clusters of S fit on the GPU at once,
// computed once per device.
template <class C>
int launch_cluster_cfg(const uint8_t* A, const uint8_t* B, const FewRowArgs& args, int M, int N, int K,
                       int kernel_kind, const DeviceInfo& dev, cudaStream_t stream, bool probe_only, int* fits) {
  auto kernel = qk_skinny_fp8_kernel<C>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return QK_ERR_CUDA;
  const int n_tiles = ceil_div(N, C::NT);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_tiles * C::SPLITS, 1, 1);
  cfg.blockDim = dim3(C::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::SPLITS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (probe_only) {
    // value + 1; 0 = not yet known (threads racing on the first call store the same value)
    static std::atomic<int> cached[64];
    std::atomic<int>& slot = cached[dev.device >= 0 && dev.device < 64 ? dev.device : 0];
    int v = slot.load(std::memory_order_relaxed);
    if (v == 0) {
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      v = n + 1;
      slot.store(v, std::memory_order_relaxed);
    }
    *fits = v - 1;
    return QK_OK;
  }
  // the prologue may overlap the previous kernel of the stream (the kernel
  // waits for it before touching memory)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  CUtensorMap tw, ta, tout;
  int st = encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, C::K_ELEMS, C::NT);
  if (st == QK_OK) st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, C::K_ELEMS, C::MT);
  // the output in [OUT_ROWS x 32] boxes (the epilogue warps' staging blocks)
  if (st == QK_OK)
    st = encode_tmap_2d_plain(&tout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, args.out, N, M, static_cast<uint64_t>(N) * 2, 32,
                              C::OUT_ROWS);
  if (st != QK_OK) return st;
  SkinnyParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_kb = ceil_div(K, C::K_ELEMS);
  p.kb_per_split = ceil_div(p.num_kb, C::SPLITS);
  p.sa = args.sa;
  p.sb = args.sb;
  p.sfa = args.sfa;
  p.sfw = args.sfw;
  p.sf_cols = K / 32;
  p.bias = args.bias;
  p.out = args.out;
  p.err = dev.err_word;
  p.timeout_ns = wait_timeout_ns();
  LaunchTimer timer(kernel_kind, stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tw, ta, tout, p);
  timer.done();
  if (e != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_CUDA;
  }
  count_launches(1);
  return QK_OK;
}

// The cluster split-K kernel with the largest S in {8, 4, 2, 1} (S no larger
// than the K-blocks) whose clusters for all weight tiles fit on the GPU in one
// wave (one pass, on-chip reduction).  Returns QK_ERR_RANGE without launching
// when no S fits (*fits_one_wave = false), or when that S is below min_s or
// leaves a CTA fewer than min_kb K-blocks (*fits_one_wave = true); with
// `force` S = 1 runs in several waves if nothing fits.
template <int MT, bool MX>
int launch_cluster(const uint8_t* A, const uint8_t* B, const FewRowArgs& args, int M, int N, int K,
                   int kernel_kind, const DeviceInfo& dev, cudaStream_t stream, bool force, int min_s,
                   int min_kb, bool* fits_one_wave) {
  constexpr int ST = MT <= 64 ? 6 : 4;
  const int n_tiles = ceil_div(N, 128);
  const int num_kb = ceil_div(K, 128);
  int chosen = 0;
  for (int S : {8, 4, 2, 1}) {
    if (S > num_kb && S > 1) continue;
    int fits = 0;
    if (S == 8) launch_cluster_cfg<SkinnyCfg<MT, 8, ST, MX>>(A, B, args, M, N, K, kernel_kind, dev, stream, true, &fits);
    if (S == 4) launch_cluster_cfg<SkinnyCfg<MT, 4, ST, MX>>(A, B, args, M, N, K, kernel_kind, dev, stream, true, &fits);
    if (S == 2) launch_cluster_cfg<SkinnyCfg<MT, 2, ST, MX>>(A, B, args, M, N, K, kernel_kind, dev, stream, true, &fits);
    if (S == 1) launch_cluster_cfg<SkinnyCfg<MT, 1, ST, MX>>(A, B, args, M, N, K, kernel_kind, dev, stream, true, &fits);
    if (n_tiles <= fits) {
      chosen = S;
      break;
    }
  }
  *fits_one_wave = chosen != 0;
  if (!force) {
    if (chosen == 0 || chosen < min_s || ceil_div(num_kb, chosen) < min_kb) return QK_ERR_RANGE;
  } else if (chosen == 0) {
    chosen = 1;
  }
  switch (chosen) {  // launch_cluster_cfg never returns QK_ERR_RANGE
    case 8:
      return launch_cluster_cfg<SkinnyCfg<MT, 8, ST, MX>>(A, B, args, M, N, K, kernel_kind, dev, stream, false, nullptr);
    case 4:
      return launch_cluster_cfg<SkinnyCfg<MT, 4, ST, MX>>(A, B, args, M, N, K, kernel_kind, dev, stream, false, nullptr);
    case 2:
      return launch_cluster_cfg<SkinnyCfg<MT, 2, ST, MX>>(A, B, args, M, N, K, kernel_kind, dev, stream, false, nullptr);
    default:
      return launch_cluster_cfg<SkinnyCfg<MT, 1, ST, MX>>(A, B, args, M, N, K, kernel_kind, dev, stream, false, nullptr);
  }
}

// Measured choice between the few-row kernels and the 2-SM tile kernel (both
// modes behave alike): a cluster split that fits in one wave wins when each
// CTA keeps at least kClusterMinKb K-blocks with M <= 64, or the split is at
// least kClusterMinSplitWide with more rows; shallower splits lose to the
// tile kernel (64 x 8192 x 1280, 128 x 7168 x 2048).
constexpr int kClusterMinKb = 6;
constexpr int kClusterMinSplitWide = 4;

template <int MT, bool MX>
int launch_streamk(const uint8_t* A, const uint8_t* B, const FewRowArgs& args, int M, int N, int K, int kernel_kind,
                   const DeviceInfo& dev, cudaStream_t stream) {
  return launch_streamk_cfg<StreamKCfg<MT, MT <= 64 ? 8 : 6, MX>>(A, B, args, M, N, K, kernel_kind, dev, stream);
}

}  // namespace qk
