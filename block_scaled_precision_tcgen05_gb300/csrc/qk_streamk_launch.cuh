// qk_streamk_launch.cuh -- host launch of the stream-K few-row kernel
// (qk_streamk_kernel.cuh) for its FP8 per-token and MXFP8 modes.
#pragma once
#include <atomic>

#include "qk_launch.cuh"
#include "qk_streamk_kernel.cuh"

namespace qk {

// One CTA per SM, launched cooperatively so that all CTAs are resident while
// owners wait for their contributors' partials.  The partials and flags come
// from the stream-ordered workspace pool; each call gets a fresh 64-bit epoch
// (shared by both modes, since they draw on the same pool), so flags left in
// reused memory by earlier calls never read as finished.
extern std::atomic<unsigned long long> g_streamk_epoch;

// `p` carries the operation's scales and bias; the launcher fills in the
// sizes, the workspace, the epoch and the wait settings.
template <class C>
int launch_streamk_cfg(const uint8_t* A, const uint8_t* B, StreamKParams p, int M, int N, int K, int kernel_kind,
                       const DeviceInfo& dev, cudaStream_t stream) {
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
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_kb = num_kb;
  p.units = units;
  p.partials = static_cast<float*>(ws);
  p.flags = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + part_bytes);
  // a 64-bit value no earlier call used (odd multiplier: a bijection of the counter)
  p.epoch = (g_streamk_epoch.fetch_add(1) + 1) * 0x9E3779B97F4A7C15ull;
  p.err = dev.err_word;
  p.timeout_ns = wait_timeout_ns();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G, 1, 1);
  cfg.blockDim = dim3(C::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LaunchTimer timer(kernel_kind, stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tw, ta, p);
  timer.done();
  const cudaError_t f = cudaFreeAsync(ws, stream);
  if (e != cudaSuccess || f != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_CUDA;
  }
  count_launches(1);
  return QK_OK;
}

}  // namespace qk
