// qk_fewrow_launch.cuh -- host launch of the few-row kernels (M <= 128):
// the cluster split-K kernel (qk_skinny_kernel.cuh) and the stream-K kernel
// (qk_streamk_kernel.cuh), each in its FP8 per-token, MXFP8, MXFP4 and NVFP4
// modes (MODE 0..3), and the choice between them.
#pragma once
#include <atomic>

#include "qk_launch.cuh"
#include "qk_skinny_kernel.cuh"
#include "qk_streamk_kernel.cuh"

namespace qk {

// The operation's operands beyond A and B: per-token / per-channel fp32
// scales (FP8) or scale rows (UE8M0 for MXFP8 / MXFP4, UE4M3 for NVFP4, with
// NVFP4's per-tensor scales ga, gb), bias and output.
struct FewRowArgs {
  const float* sa = nullptr;
  const float* sb = nullptr;
  const uint8_t* sfa = nullptr;
  const uint8_t* sfw = nullptr;
  const float* ga = nullptr;
  const float* gb = nullptr;
  const uint16_t* bias = nullptr;
  uint16_t* out = nullptr;
};

// One CTA per SM, launched cooperatively so that all CTAs are resident while
// owners wait for their contributors' partials.  The partials and flags come
// from the stream-ordered workspace pool; each call gets a fresh 64-bit epoch
// (shared by both modes, since they draw on the same pool), so flags left in
// reused memory by earlier calls never read as finished.
extern std::atomic<unsigned long long> g_streamk_epoch;

// Bytes of K per operand row (packed FP4 modes: two elements per byte), and
// scale bytes per row (NVFP4: one per 16 K, else one per 32 K).
template <class C>
inline int fewrow_k_bytes(int K) { return C::FP4 ? K / 2 : K; }
template <class C>
inline int fewrow_sf_cols(int K) { return C::MODE == 3 ? K / 16 : K / 32; }

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
  const int kbytes = fewrow_k_bytes<C>(K);
  CUtensorMap tw, ta;
  int st = encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kbytes, N, kbytes, C::KB_BYTES, C::NT);
  if (st == QK_OK) st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, kbytes, M, kbytes, C::KB_BYTES, C::MT);
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
  p.sf_cols = fewrow_sf_cols<C>(K);
  p.ga = args.ga;
  p.gb = args.gb;
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
  const int kbytes = fewrow_k_bytes<C>(K);
  int st = encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kbytes, N, kbytes, C::KB_BYTES, C::NT);
  if (st == QK_OK) st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, kbytes, M, kbytes, C::KB_BYTES, C::MT);
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
  p.sf_cols = fewrow_sf_cols<C>(K);
  p.ga = args.ga;
  p.gb = args.gb;
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

// The cluster split-K kernel with the largest S (8 down to 1 for up to 64
// activation rows; 8, 4, 2, 1 for 128, whose rows then split evenly; S no
// larger than the K-blocks) whose clusters for all weight tiles fit on the
// GPU in one wave (one pass, on-chip reduction): the most SMs streaming.
// Clusters need not be powers of two: 17 tiles fit as clusters of 6 (102
// CTAs, three per GPC) where clusters of 8 do not.  Returns QK_ERR_RANGE
// without launching when no S fits (*fits_one_wave = false); with `force`
// S = 1 runs in several waves if nothing fits.
template <int MT, int MODE, int S>
int launch_cluster_s(const uint8_t* A, const uint8_t* B, const FewRowArgs& args, int M, int N, int K,
                     int kernel_kind, const DeviceInfo& dev, cudaStream_t stream, bool probe_only, int* fits) {
  constexpr int ST = MT <= 64 ? 6 : 4;
  return launch_cluster_cfg<SkinnyCfg<MT, S, ST, MODE>>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only,
                                                        fits);
}

template <int MT, int MODE>
int launch_cluster_split(int S, const uint8_t* A, const uint8_t* B, const FewRowArgs& args, int M, int N, int K,
                         int kernel_kind, const DeviceInfo& dev, cudaStream_t stream, bool probe_only, int* fits) {
  if constexpr (MT <= 64) {
    switch (S) {
      case 8: return launch_cluster_s<MT, MODE, 8>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
      case 7: return launch_cluster_s<MT, MODE, 7>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
      case 6: return launch_cluster_s<MT, MODE, 6>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
      case 5: return launch_cluster_s<MT, MODE, 5>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
      case 4: return launch_cluster_s<MT, MODE, 4>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
      case 3: return launch_cluster_s<MT, MODE, 3>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
      case 2: return launch_cluster_s<MT, MODE, 2>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
      default: return launch_cluster_s<MT, MODE, 1>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
    }
  } else {
    switch (S) {
      case 8: return launch_cluster_s<MT, MODE, 8>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
      case 4: return launch_cluster_s<MT, MODE, 4>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
      case 2: return launch_cluster_s<MT, MODE, 2>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
      default: return launch_cluster_s<MT, MODE, 1>(A, B, args, M, N, K, kernel_kind, dev, stream, probe_only, fits);
    }
  }
}

template <int MT, int MODE>
int launch_cluster(const uint8_t* A, const uint8_t* B, const FewRowArgs& args, int M, int N, int K,
                   int kernel_kind, const DeviceInfo& dev, cudaStream_t stream, bool force, bool* fits_one_wave) {
  const int n_tiles = ceil_div(N, 128);
  const int num_kb = ceil_div(MODE >= 2 ? K / 2 : K, 128);  // 128-byte K-blocks
  int chosen = 0;
  for (int S = 8; S >= 1; --S) {
    if (MT > 64 && (S & (S - 1)) != 0) continue;  // 128 rows split evenly
    if (S > num_kb && S > 1) continue;
    int fits = 0;
    launch_cluster_split<MT, MODE>(S, A, B, args, M, N, K, kernel_kind, dev, stream, true, &fits);
    if (n_tiles <= fits) {
      chosen = S;
      break;
    }
  }
  *fits_one_wave = chosen != 0;
  if (chosen == 0) {
    if (!force) return QK_ERR_RANGE;
    chosen = 1;
  }
  // launch_cluster_cfg never returns QK_ERR_RANGE
  return launch_cluster_split<MT, MODE>(chosen, A, B, args, M, N, K, kernel_kind, dev, stream, false, nullptr);
}

// Stages: 8 (MT <= 64) or 6; the FP4 modes' larger scale atoms leave room for 6 or 5.
template <int MT, int MODE>
int launch_streamk(const uint8_t* A, const uint8_t* B, const FewRowArgs& args, int M, int N, int K, int kernel_kind,
                   const DeviceInfo& dev, cudaStream_t stream) {
  constexpr int ST = MODE >= 2 ? (MT <= 64 ? 6 : 5) : (MT <= 64 ? 8 : 6);
  return launch_streamk_cfg<StreamKCfg<MT, ST, MODE>>(A, B, args, M, N, K, kernel_kind, dev, stream);
}

// The few-row choice of the block-scaled modes, measured on all three
// (event times in us, tile kernel / few-row kernel): the cluster split-K
// kernel whenever one wave of clusters covers all weight tiles, whatever the
// split and the K range per CTA (MXFP8 128x7168x2048 21.5 / 14.4, 64x8192x1280
// 19.5 / 12.3; MXFP4 64x7168x1024 17.4 / 10.2; NVFP4 96x2112x8192 29.7 /
// 22.5); otherwise stream-K for MXFP8 and MXFP4 (MXFP8 128x21504x5376 50.2 /
// 40.0, 8x28672x8192 85.0 / 50.2; MXFP4 64x28672x8192 42.0 / 40.0), and for
// NVFP4 only with at most 64 rows and 10 to 30 units of 128 weight rows x 128
// bytes of K per SM (64x21504x5376 35.8 / 31.8; its four scale words per row
// and unit make longer ranges slower than the tile kernel: 64x28672x8192
// 48.2 / 56.3); else nothing (*launched = false: the caller runs the tile
// kernel).  QK_MX_SKINNY (test-only): 1 = never, 2 = stream-K, 3 = cluster
// split-K, whenever M <= 128.
template <int MODE>
int launch_fewrow_block_scaled(const uint8_t* A, const uint8_t* B, const FewRowArgs& args, int M, int N, int K,
                               int kernel_kind, const DeviceInfo& dev, cudaStream_t stream, bool* launched) {
  *launched = false;
  const int skinny = kernel_variant("QK_MX_SKINNY");
  if (M > 128 || skinny == 1) return QK_OK;
  *launched = true;
  const long long units =
      static_cast<long long>(ceil_div(N, 128)) * ceil_div(MODE >= 2 ? K / 2 : K, 128);
  if (skinny == 2) {
    if (M <= 64) return launch_streamk<64, MODE>(A, B, args, M, N, K, kernel_kind, dev, stream);
    return launch_streamk<128, MODE>(A, B, args, M, N, K, kernel_kind, dev, stream);
  }
  bool fits = false;
  if (skinny == 3) {
    if (M <= 64) return launch_cluster<64, MODE>(A, B, args, M, N, K, kernel_kind, dev, stream, true, &fits);
    return launch_cluster<128, MODE>(A, B, args, M, N, K, kernel_kind, dev, stream, true, &fits);
  }
  const int st = M <= 64
                     ? launch_cluster<64, MODE>(A, B, args, M, N, K, kernel_kind, dev, stream, false, &fits)
                     : launch_cluster<128, MODE>(A, B, args, M, N, K, kernel_kind, dev, stream, false, &fits);
  if (st != QK_ERR_RANGE) return st;
  const long long sm = dev.sm_count;
  const bool streamk = MODE != 3 || (M <= 64 && units >= 10 * sm && units < 30 * sm);
  if (streamk) {
    if (M <= 64) return launch_streamk<64, MODE>(A, B, args, M, N, K, kernel_kind, dev, stream);
    return launch_streamk<128, MODE>(A, B, args, M, N, K, kernel_kind, dev, stream);
  }
  *launched = false;
  return QK_OK;
}

}  // namespace qk
