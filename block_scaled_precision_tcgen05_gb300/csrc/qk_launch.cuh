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
  // whole tiles only; launch_gemm may split the last wave's tiles
  p.num_units = p.num_tiles;
  p.full_tiles = p.num_tiles;
  p.split = 1;
  p.split_kb = p.num_kb;
  p.split_ws = nullptr;
  p.split_cnt = nullptr;
  p.split_tag = 0;
}

// K-parts per tile of the last wave: after at least one full wave, the last
// R = tiles mod slots tiles are split when they would leave at least half of
// the slots idle, into S <= 4 parts (S * R <= slots) of at least 20 k-blocks
// each; 1 = no split.  A half-empty last wave already runs each tile faster
// than a full one (its SMs share the L2's bandwidth with fewer others), so a
// split gains only the difference between that and 1/S of a tile, less the
// partials' round trip through L2: measured +1.2 / +1.9% for MXFP4 / NVFP4
// 8192 x 8192 x 16384 and +1.5% for FP8 1024 x 21504 x 5376, while one wave of
// split tiles (MXFP4 512 x 4608 x 4096, 16 k-blocks) ran 20% slower.
inline int tail_split_parts(long long tiles, long long slots, int num_kb) {
  if (slots <= 0 || tiles < slots) return 1;
  const long long R = tiles % slots;
  if (R == 0 || 2 * R > slots) return 1;
  int S = static_cast<int>(slots / R < 4 ? slots / R : 4);
  while (S >= 2 && num_kb < 20 * S) --S;
  return S >= 2 ? S : 1;
}

// tags of the split tiles' arrival words, one per call
inline std::atomic<unsigned long long> g_split_epoch{0};

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
// pre-pass, or the int8 -> f16 widening pass, which the producer waits for
// before its first load; nothing else in the kernel reads what that pass
// writes, and every earlier kernel of the stream completed before it began).
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
  // tail split (splittable kinds): the last wave's tiles as K-parts, their
  // fp32 partials and arrival words in a stream-ordered workspace.
  // QK_TAIL_SPLIT (tests): 1 = never split; n >= 2 = split the last
  // min(tiles, slots) tiles into n parts whatever they cost.
  GemmParams q = p;
  void* ws = nullptr;
  if constexpr (C::SPLITTABLE) {
    const int force = kernel_variant("QK_TAIL_SPLIT");
    int S = 1, R = 0;
    if (force >= 2) {
      R = p.num_tiles < slots ? p.num_tiles : slots;
      S = force < p.num_kb ? force : p.num_kb;
    } else if (force != 1) {
      S = tail_split_parts(p.num_tiles, slots, p.num_kb);
      R = p.num_tiles % slots;
    }
    int skb = p.num_kb;
    if (S >= 2) {
      skb = ceil_div(p.num_kb, S);
      S = ceil_div(p.num_kb, skb);  // no empty part
    }
    if (S >= 2 && dev.pool) {
      const size_t regions = static_cast<size_t>(R) * C::CTAS * C::EPI_WARPS;
      const size_t part_bytes = regions * static_cast<size_t>(S) * 32 * C::EPI_COLS * sizeof(float);
      if (cudaMallocFromPoolAsync(&ws, part_bytes + regions * sizeof(unsigned long long), dev.pool, stream) ==
          cudaSuccess) {
        q.split = S;
        q.split_kb = skb;
        q.full_tiles = p.num_tiles - R;
        q.num_units = q.full_tiles + R * S;
        q.split_ws = static_cast<float*>(ws);
        q.split_cnt = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + part_bytes);
        // a 56-bit value no earlier call used (odd multiplier: a bijection of the counter)
        q.split_tag = ((g_split_epoch.fetch_add(1) + 1) * 0x9E3779B97F4A7C15ull) & ~0xFFull;
      } else {
        cudaGetLastError();  // no workspace: whole tiles
        ws = nullptr;
      }
    }
  }
  const int work = C::SPLITTABLE ? q.num_units : q.num_tiles;
  const int ctas = (work < slots ? work : slots) * C::CTAS;
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
                      static_cast<int>(C::OUT), C::OUT_COLS) != QK_OK) {
    if (ws) cudaFreeAsync(ws, stream);
    return QK_ERR_CUDA;
  }
  LaunchTimer timer(kernel_kind<C>(), stream);
  e = cudaLaunchKernelEx(&cfg, kernel, ta, tb, tsa, tsb, tout, q);
  timer.done();
  const cudaError_t f = ws ? cudaFreeAsync(ws, stream) : cudaSuccess;
  if (e != cudaSuccess || f != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_CUDA;
  }
  count_launches(1);
  return QK_OK;
}

}  // namespace qk
