// qk_mxfp4.cu -- MXFP4 (packed E2M1 elements, one UE8M0 scale per 32 K) GEMM
// on tcgen05.mma kind::mxf4.block_scale.scale_vec::2X, which reads the
// packed 4-bit operands directly (ROCm/FlyDSL PR #990: MXFP4 with per-1x32
// scales).  Operands are [rows, K/2] bytes, element 2i in the low nibble.
#include "qk_launch.cuh"

namespace qk {

// 256 x 256 tiles on a 2-SM CTA pair (each SM loads half of B: 32 KB of
// operands per 256-K stage instead of 48), five stages, one accumulator that
// 16 epilogue warps drain into registers (64 columns each) and release before
// the epilogue math, so the next tile's MMAs start after the drain.  Each CTA
// stages its own A scales and all of B's; the peer's relay warp forwards each
// slot to the leader, whose scale-copy thread fills both CTAs' TMEM with
// cta_group::2 copies beside the MMAs.  Measured alternatives (the same pair
// with 8 epilogue warps working from TMEM; one CTA with 128 x 256 tiles) were
// slower and are not built.
using CfgMxfp4PairDrain = GemmCfg<Kind::MXF4, 256, 5, 1, true, 16, 1>;
// The same kernel with B's scales per 32x32 block.
using CfgMxfp4PairDrainB32 = GemmCfg<Kind::MXF4, 256, 5, 1, true, 16, 1, OutType::BF16, true>;

template <class C>
static int launch_mxfp4_cfg(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                      const uint16_t* bias, uint16_t* out, int M, int N, int K, const DeviceInfo& dev,
                      cudaStream_t stream) {
  CUtensorMap ta, tb;
  const uint64_t kb = static_cast<uint64_t>(K) / 2;  // bytes per row
  int st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, kb, M, kb, C::TMA_K, C::BM);
  if (st == QK_OK) st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kb, N, kb, C::TMA_K, C::B_LOAD_ROWS);
  if (st != QK_OK) return st;
  GemmParams p{};
  plan_tiles<C>(p, M, N, K);
  p.bias = bias;
  p.out = out;
  p.sA = sA;
  p.sB = sB;
  p.sf_cols = K / 32;
  p.err = dev.err_word;
  p.timeout_ns = wait_timeout_ns();
  // Raw scale rows go through TMA when their pitch (K/32 bytes) and base
  // addresses are 16-byte multiples, through cp.async when they are 4-byte
  // multiples, else through per-stage loads.
  CUtensorMap tsa = ta, tsb = tb;
  const bool a16 = ((reinterpret_cast<uintptr_t>(sA) | reinterpret_cast<uintptr_t>(sB)) & 15u) == 0;
  p.sf_mode = (p.sf_cols % 16 == 0 && a16) ? kSfTma : (p.sf_cols % 4 == 0 ? kSfAsync : kSfLoads);
  if (p.sf_mode == kSfTma) {
    st = encode_tmap_2d_plain(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, sA, p.sf_cols, M, p.sf_cols, 16, C::BM);
    // B's scale rows: one per row of B, or one per 32 rows (C::SFB32)
    const uint64_t sb_rows = C::SFB32 ? static_cast<uint64_t>((N + 31) / 32) : static_cast<uint64_t>(N);
    if (st == QK_OK)
      st = encode_tmap_2d_plain(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, sB, p.sf_cols, sb_rows, p.sf_cols, 16,
                                C::SFB32 ? C::BN / 32 : C::BN);
    if (st != QK_OK) return st;
  }
  return launch_gemm<C>(ta, tb, tsa, tsb, p, dev, stream);
}

int launch_mxfp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const uint16_t* bias,
                 uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  return launch_mxfp4_cfg<CfgMxfp4PairDrain>(A, sA, B, sB, bias, out, M, N, K, dev, stream);
}

int launch_mxfp4_b32(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB32,
                     const uint16_t* bias, uint16_t* out, int M, int N, int K, const DeviceInfo& dev,
                     cudaStream_t stream) {
  return launch_mxfp4_cfg<CfgMxfp4PairDrainB32>(A, sA, B, sB32, bias, out, M, N, K, dev, stream);
}

}  // namespace qk
