// qk_int8_exact.cuh -- the two kernels of the exact INT8 GEMM on the f16 tensor
// pipe and the launch sequence that runs them over a given f16 workspace.
//
// sm_103a has no integer tcgen05.mma kind, so the int8 operands are widened
// to f16 (every int8 value is exact in f16) by a bandwidth-bound pass, and
// the f16 MMA accumulates in fp32 in chunks of at most 1024 K: every partial
// sum is then an integer of magnitude at most 1024 * 128 * 128 = 2^24, which
// fp32 holds exactly.  The epilogue drains each chunk to int32 and adds the
// chunks, so the accumulator is the exact integer dot product, and the
// fixed-order epilogue of comfy-kitchen PR #174 (update "Keep the cached INT8
// epilogue scale order exact") makes the bf16 result bit-identical to the
// definition.
#pragma once

#include <cuda_fp16.h>

#include "qk_launch.cuh"

namespace qk {

// 256 x 256 tiles per CTA pair, two fp32 accumulators of 256 columns per SM
// (all 512 TMEM columns); 16 epilogue warps keep the int32 running sums in
// registers, so a chunk drains while the MMAs fill the other accumulator.
using CfgInt8 = GemmCfg<Kind::F16, 256, 6, 2, true, 16, 1>;
// fp16 output: the same layout; fp32 output: 4 KB staging blocks per
// epilogue warp, so one ring stage fewer fits in shared memory.
using CfgInt8F16 = GemmCfg<Kind::F16, 256, 6, 2, true, 16, 1, OutType::F16>;
using CfgInt8F32 = GemmCfg<Kind::F16, 256, 5, 2, true, 16, 1, OutType::F32>;

// Widens 16 int8 values per thread to f16.  Byte x becomes the f16
// bit pattern 0x6400 | (x + 128), i.e. the value 1024 + x + 128, and one
// exact subtraction of 1152 leaves x.
__device__ __forceinline__ uint4 widen8(uint32_t w, uint32_t w2) {
  const __half2 bias = __float2half2_rn(1152.f);
  uint32_t o[4];
  const uint32_t in[2] = {w ^ 0x80808080u, w2 ^ 0x80808080u};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t lo = __byte_perm(in[j], 0x64646464u, 0x4140);
    uint32_t hi = __byte_perm(in[j], 0x64646464u, 0x4342);
    __half2 hlo = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
    __half2 hhi = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
    o[2 * j] = *reinterpret_cast<uint32_t*>(&hlo);
    o[2 * j + 1] = *reinterpret_cast<uint32_t*>(&hhi);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

static __global__ void __launch_bounds__(256) qk_int8_to_f16_kernel(const uint4* __restrict__ a, uint4* __restrict__ a16,
                                                              long long na, const uint4* __restrict__ b,
                                                              uint4* __restrict__ b16, long long nb) {
  // the GEMM that reads a16 / b16 may launch once every block of this pass
  // has started (it waits for the pass to complete before its first load)
  griddep_launch_dependents();
  const long long total = na + nb;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
#pragma unroll 1
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const bool in_a = i < na;
    const long long j = in_a ? i : i - na;
    const uint4 s = __ldcs(in_a ? a + j : b + j);
    uint4* d = in_a ? a16 + 2 * j : b16 + 2 * j;
    d[0] = widen8(s.x, s.y);
    d[1] = widen8(s.z, s.w);
  }
}

// Widens A and B into a16 [M, K] and b16 [N, K] (caller-provided device
// memory) and runs the GEMM over them, both on `stream`; C fixes the output
// element type.
template <class C = CfgInt8>
static inline int widen_and_gemm_int8(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                                      const uint16_t* bias, void* out, int M, int N, int K, uint16_t* a16,
                                      uint16_t* b16, const DeviceInfo& dev, cudaStream_t stream) {
  const size_t a_elems = static_cast<size_t>(M) * K;
  const size_t b_elems = static_cast<size_t>(N) * K;
  const long long na = static_cast<long long>(a_elems / 16), nb = static_cast<long long>(b_elems / 16);
  // one 16-byte element per thread and a block per 256 of them, hundreds of
  // waves of short blocks: at 30000 + 21504 rows x 5376 this moves 6.78 TB/s
  // (the measured copy rate), where a grid-stride loop over one wave of 8
  // blocks per SM moved 4.9 (2 to 8 elements in flight per thread: 4.5 to 6.1
  // TB/s, the rate rising and falling with the grid size)
  long long blocks = (na + nb + 255) / 256;
  if (blocks > 0x7fffffffLL) blocks = 0x7fffffffLL;  // the loop covers any rest
  LaunchTimer timer(kKInt8ToF16, stream);
  qk_int8_to_f16_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(A), reinterpret_cast<uint4*>(a16), na, reinterpret_cast<const uint4*>(B),
      reinterpret_cast<uint4*>(b16), nb);
  timer.done();
  int st = cudaGetLastError() == cudaSuccess ? QK_OK : QK_ERR_CUDA;
  if (st == QK_OK) count_launches(1);

  CUtensorMap ta, tb;
  if (st == QK_OK)
    st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a16, K, M, static_cast<uint64_t>(K) * 2, C::TMA_K, C::BM);
  if (st == QK_OK)
    st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, b16, K, N, static_cast<uint64_t>(K) * 2, C::TMA_K, C::B_LOAD_ROWS);
  if (st == QK_OK) {
    GemmParams p{};
    plan_tiles<C>(p, M, N, K);
    p.sa = sa;
    p.sb = sb;
    p.bias = bias;
    p.out = out;
    p.err = dev.err_word;
    p.timeout_ns = wait_timeout_ns();
    // programmatic launch: the GEMM's prologue overlaps the widening pass's
    // last wave, and its producer waits for the pass before the first load
    st = launch_gemm<C>(ta, tb, ta, tb, p, dev, stream, true);
  }
  return st;
}

}  // namespace qk
