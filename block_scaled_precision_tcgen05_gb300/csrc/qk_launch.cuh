// qk_launch.cuh -- host-side launch of one GEMM kernel configuration.
#pragma once

#include <atomic>

#include "qk_gemm_kernel.cuh"
#include "qk_internal.h"

namespace qk {

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Fills the tile/k-block bookkeeping of GemmParams for configuration C.
// Row-blocks per raster group: QK_GROUP_M from the environment, else 8.
int raster_group_m();
// Test-only selector of the few-row kernels (QK_FP8_SKINNY, QK_MX_SKINNY): the
// integer value of the environment variable, 0 if unset.
int kernel_variant(const char* env_name);

template <class C>
void plan_tiles(GemmParams& p, int M, int N, int K) {
  p.group_m = raster_group_m();
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_kb = ceil_div(K, C::K_ELEMS);
  p.num_m_blocks = ceil_div(M, C::TILE_M);
  p.num_n_blocks = ceil_div(N, C::BN);
  p.num_tiles = p.num_m_blocks * p.num_n_blocks;
  if (C::INT_CHUNKS) {
    // 1024 K per chunk: |partial| <= 1024 * 2^14 = 2^24, exact in fp32.
    p.chunk_kb = 1024 / C::K_ELEMS;
  } else if (C::BLOCKSCALE) {
    p.chunk_kb = 1;  // one 128-K scale block per chunk
  } else {
    p.chunk_kb = p.num_kb;
  }
  p.num_chunks = ceil_div(p.num_kb, p.chunk_kb);
}

template <class C>
constexpr int kernel_kind() {
  return C::kind == Kind::F16    ? kKGemmInt8
         : C::kind == Kind::F8   ? kKGemmFp8
         : C::kind == Kind::MXF8 ? kKGemmMxfp8
         : C::kind == Kind::MXF4 ? kKGemmMxfp4
         : C::kind == Kind::NVF4 ? kKGemmNvfp4
                                 : kKGemmFp8Blockscale;
}

// tsa / tsb: tensor maps of the scale atoms (block-scaled kinds), else any map.
// after_prepass: launch with programmatic stream serialization, so the kernel's
// prologue overlaps the kernel before it in the stream (the scale-atom
// pre-pass, which the producer waits for before its first load).
template <class C>
int launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa, const CUtensorMap& tsb,
                const GemmParams& p, const DeviceInfo& dev, cudaStream_t stream, bool after_prepass = false) {
  auto kernel = qk_gemm_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return QK_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int slots = dev.sm_count;  // concurrently resident CTAs (one per SM) or CTA pairs
  if constexpr (C::CTAS > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // how many clusters fit at once (SMs pair up within a GPC), computed once per
    // device; threads racing on the first call store the same value
    static std::atomic<int> cached[64];
    std::atomic<int>& clusters = cached[dev.device >= 0 && dev.device < 64 ? dev.device : 0];
    int n = clusters.load(std::memory_order_relaxed);
    if (n == 0) {
      cfg.gridDim = dim3(2 * (dev.sm_count / 2), 1, 1);
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = dev.sm_count / 2;
      }
      clusters.store(n, std::memory_order_relaxed);
    }
    slots = n;
  }
  const int ctas = (p.num_tiles < slots ? p.num_tiles : slots) * C::CTAS;
  cfg.gridDim = dim3(ctas, 1, 1);
  if (after_prepass) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    ++cfg.numAttrs;
  }
  // the output as boxes of the staging blocks (32 rows x OUT_COLS), with their swizzle
  CUtensorMap tout;
  if (encode_tmap_out(&tout, p.out, static_cast<uint64_t>(p.M), static_cast<uint64_t>(p.N),
                      static_cast<int>(C::OUT), C::OUT_COLS) != QK_OK)
    return QK_ERR_CUDA;
  LaunchTimer timer(kernel_kind<C>(), stream);
  e = cudaLaunchKernelEx(&cfg, kernel, ta, tb, tsa, tsb, tout, p);
  timer.done();
  if (e != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_CUDA;
  }
  count_launches(1);
  return QK_OK;
}

}  // namespace qk
