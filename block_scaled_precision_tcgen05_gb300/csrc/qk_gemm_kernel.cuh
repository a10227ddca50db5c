// qk_gemm_kernel.cuh -- the persistent, warp-specialised tcgen05 GEMM
//
//     out[m,n] = round_out( epilogue( sum_k A[m,k] * B[n,k] ) )
//
// A [M,K] and B [N,K] are K-major; round_out is bf16 round-to-nearest-even
// unless the configuration's OutType says fp16 or fp32.  Persistent CTAs
// (one per SM, or one 2-SM pair per two SMs) walk output tiles of
// 128 x BN (a pair: 256 x BN) in a grouped-M raster.  Tail split (kinds with
// one accumulation chunk per tile): when the last wave of tiles would leave
// at least half of the CTAs idle, its tiles run as S K-parts each (work
// units after the whole tiles); every part writes its fp32 partial to a
// workspace, and per epilogue warp the part that finishes last adds the S
// partials in K order and runs the epilogue on the sum.  Roles:
//   warp 0      TMA producer: A/B tiles of 128-byte K rows into a STAGES-deep
//               shared-memory ring (128-byte swizzle); block-scaled kinds: the
//               stage's scale-factor atoms with them (see qk_sf_atoms.cuh).
//   warp 1      MMA issuer: allocates TMEM, issues tcgen05.mma into a TMEM
//               accumulator and releases ring slots / accumulators with
//               tcgen05.commit; in a pair's peer CTA it relays the peer's
//               accumulator releases to the leader.
//   warps 2, 3  block-scaled kinds, in the MMA-issuing CTA: scale-factor
//               copies (tcgen05.cp), each warp half of every ring slot's
//               atoms, committed to a per-slot barrier the MMA warp waits on,
//               so the copies run beside the MMAs instead of between them
//               (copies issued by the MMA thread run in series with its MMAs,
//               and one thread issues a copy about every 100 cycles).
//
// Scale factors (block-scaled kinds) arrive with the operands: the caller's
// raw row-major scale bytes are rearranged once per call into 512-byte atoms
// in the order tcgen05.cp reads (qk_sf_atoms.cuh), and the producer loads each
// ring stage's atoms by TMA just before its A/B tiles, counted on a barrier of
// their own (sf_full).  The copy threads move a slot's atoms into the slot's
// TMEM columns once they have landed and the MMAs of the slot's previous round
// have completed (empty), while the operands are still in flight, and commit
// to sf_ready; the MMA warp waits on full and sf_ready, so it issues nothing
// but MMAs and its ring commits.
//   warps 4..   EPI_WARPS epilogue warps (4 or 16): TMEM -> registers,
//               fixed-order scale/bias epilogue, output rounding, staged bulk
//               tensor stores; warp 4 + 4p + q owns TMEM lanes 32q..32q+31
//               (tile rows) of column part p.
//
// Kinds:
//   F16   exact INT8: int8 operands converted to f16 beforehand (exact), f16
//         MMA with fp32 accumulation.  Accumulation restarts every chunk of
//         at most 1024 K (every partial sum is then an integer below 2^24,
//         exact in fp32); the epilogue drains each chunk to int32 and adds
//         the chunks in int32, so the result is the exact integer dot
//         product.
//   F8    E4M3 x E4M3 with fp32 accumulation (per-token x per-channel FP8).
//   F8BS  E4M3 x E4M3, every 128-K block its own accumulation chunk, folded
//         into fp32 register sums with its A and B block scales (blockscale).
//   MXF8  E4M3 with one UE8M0 scale per 32 K (block_scale, scale_vec::1X).
//   MXF4  packed E2M1 with one UE8M0 scale per 32 K (kind::mxf4, 2X).
//   NVF4  packed E2M1 with one UE4M3 scale per 16 K (kind::mxf4nvf4, 4X) and
//         the product of two per-tensor fp32 scales in the epilogue.
//
// Epilogue order (comfy-kitchen PR #174, Summary and the update "Keep the
// cached INT8 epilogue scale order exact"): x = float(acc); x = x*sa[m];
// x = x*sb[n]; if bias: x = x + float(bias[n]); out = bf16_rne(x).  Without
// bias no add happens, so a -0 survives ("Preserve signed zero without INT8
// bias").  MX kinds: out = bf16_rne(acc (+ bias)).  The same page's INT8
// specialization also writes fp16 and fp32 outputs (update "rebased onto
// v0.2.38", its resources paragraph): out = fp16_rne(x) or x itself.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qk_device.cuh"

namespace qk {

enum class Kind : int { F16 = 0, F8 = 1, MXF8 = 2, MXF4 = 3, NVF4 = 4, F8BS = 5 };

// Output element type (the values of the public QK_OUT_* constants).
enum class OutType : int { BF16 = 0, F16 = 1, F32 = 2 };

struct GemmParams {
  int M, N, K;
  int num_kb;                 // k-blocks (ring stages) per tile
  int num_m_blocks, num_n_blocks, num_tiles;
  int chunk_kb;               // k-blocks per exact accumulation chunk (F16); == num_kb otherwise
  int num_chunks;             // ceil(num_kb / chunk_kb)
  const float* sa;            // [M] row scales (F16, F8)
  const float* sb;            // [N] column scales (F16, F8)
  const uint16_t* bias;       // [N] bf16 bits, nullable
  void* out;                  // [M, N] bf16 / fp16 bits or fp32 (the configuration's OutType)
  int sf_gpad;                // block-scaled kinds: atoms per 128-row block in the atom buffers (num_kb * SF_ATOMS_K)
  const float* ga;            // NVFP4 per-tensor scales (nullable: 1)
  const float* gb;
  int scale_kb;               // FP8 blockscale: K-blocks of 128 per scale row (sa [M, kb], sb [ceil(N/128), kb])
  int group_m;                // row-blocks per raster group
  // tail split: units [0, full_tiles) are whole tiles; unit full_tiles + v is
  // K-part v % split of tile full_tiles + v / split, k-blocks
  // [part * split_kb, min(num_kb, (part + 1) * split_kb))
  int num_units, full_tiles, split, split_kb;
  float* split_ws;                   // fp32 partials [tail tile][CTA][epilogue warp][part][EPI_COLS/4][32 lanes][4]
  unsigned long long* split_cnt;     // arrival words [tail tile][CTA][epilogue warp]
  unsigned long long split_tag;      // this call's tag (low 8 bits zero)
  unsigned long long* err;    // device error word
  uint64_t timeout_ns;        // bound on every barrier wait
};

// PAIR_: a cluster of two CTAs computes a (2*128) x BN tile with 2-SM MMAs
// (cta_group::2): each CTA holds 128 rows of A and BN/2 rows of B, the
// leader CTA issues the MMAs, each CTA's TMEM receives its 128 rows of D.
// EPI_WARPS_: epilogue warps (a multiple of 4; each group of four covers all
// 128 TMEM lanes for BN / (EPI_WARPS_/4) columns).  For the exact INT8 kind,
// 16 epilogue warps keep the int32 running sums in registers (64 columns per
// thread) instead of TMEM, which frees TMEM for two accumulators.
// OUT_BUFS_: shared-memory staging blocks per epilogue warp for bulk tensor
// stores of the output; 0 = the epilogue stores straight to global memory.
// OUT_COLS_: columns of a staging block (32 rows each): 32, or 16 for 16-bit
// outputs (half the staging memory, twice the bulk stores).
template <Kind KIND, int BN_, int STAGES_, int ACC_BUFS_, bool PAIR_ = false, int EPI_WARPS_ = 4,
          int OUT_BUFS_ = 2, OutType OUT_ = OutType::BF16, int OUT_COLS_ = 32>
struct GemmCfg {
  static constexpr Kind kind = KIND;
  static constexpr OutType OUT = OUT_;
  static constexpr int OUT_ELEM_BYTES = OUT_ == OutType::F32 ? 4 : 2;
  static constexpr bool PAIR = PAIR_;
  static constexpr int CTAS = PAIR ? 2 : 1;  // CTAs of a cluster
  static constexpr int BM = 128;                 // rows of A (and D) per CTA
  static constexpr int TILE_M = BM * CTAS;       // rows of a cluster's tile
  static constexpr int MMA_M = PAIR ? 256 : 128; // rows of one MMA
  static constexpr int BN = BN_;                 // columns of a tile
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;   // rows of B in a CTA's shared memory
  static constexpr int B_LOAD_ROWS = BN / CTAS;       // rows of B a CTA loads per stage
  static constexpr int STAGES = STAGES_;
  static constexpr int ACC_BUFS = ACC_BUFS_;
  static constexpr int ROW_BYTES = 128;  // bytes of K per row per ring stage (one swizzle row)
  static constexpr bool FP4 = KIND == Kind::MXF4 || KIND == Kind::NVF4;
  static constexpr int K_ELEMS = KIND == Kind::F16 ? 64 : (FP4 ? 256 : 128);
  static constexpr int TMA_K = KIND == Kind::F16 ? 64 : 128;  // tensor-map elements per stage along K
  static constexpr int UMMA_K = KIND == Kind::F16 ? 16 : (FP4 ? 64 : 32);
  static constexpr int K_STEPS = K_ELEMS / UMMA_K;  // 4 MMAs of 32 bytes of K each
  // block-scaled kinds: scales staged per ring slot and copied to TMEM
  static constexpr bool MX = KIND == Kind::MXF8 || KIND == Kind::MXF4 || KIND == Kind::NVF4;
  static constexpr int SF_BLOCK = KIND == Kind::NVF4 ? 16 : 32;  // K-elements per scale byte
  static constexpr bool ALPHA = KIND == Kind::NVF4;              // per-tensor scales in the epilogue
  static constexpr bool INT_CHUNKS = KIND == Kind::F16;
  // FP8 blockscale: every 128-K block is its own accumulation chunk, scaled
  // by sa[m, g] * sb[n / 128, g] into fp32 sums held in registers
  static constexpr bool BLOCKSCALE = KIND == Kind::F8BS;
  static constexpr bool DENSE_F8 = KIND == Kind::F8 || KIND == Kind::F8BS;
  static constexpr bool ROWWISE = KIND == Kind::F16 || KIND == Kind::F8;
  static constexpr int EPI_WARPS = EPI_WARPS_;
  static constexpr int EPI_PARTS = EPI_WARPS / 4;     // column parts of a tile
  static constexpr int EPI_COLS = BN_ / EPI_PARTS;    // columns per epilogue warp
  // 16 epilogue warps hold 64 columns per thread in registers: the exact
  // INT8 and blockscale kinds keep running sums there; the block-scaled kinds
  // drain the accumulator into them and release it before the epilogue math.
  static constexpr bool REG_SUMS = (INT_CHUNKS || BLOCKSCALE || MX || KIND == Kind::F8) && EPI_WARPS == 16;
  // kinds whose one-chunk accumulator is drained into registers and released before the epilogue math
  static constexpr bool REG_DRAIN = REG_SUMS && (MX || KIND == Kind::F8);
  // kinds whose tiles may be split along K (one accumulation chunk per tile)
  static constexpr bool SPLITTABLE = !INT_CHUNKS && !BLOCKSCALE;

  static constexpr int SF_PER_STAGE = MX ? K_ELEMS / SF_BLOCK : 0;  // scale bytes per row per stage
  static constexpr int SF_ATOMS_K = SF_PER_STAGE / 4;         // 4 scale bytes per 32-bit TMEM column
  static constexpr int NB128 = (BN + 127) / 128;              // 128-row blocks of the B tile
  static constexpr int SFA_BYTES = SF_ATOMS_K * 512;
  static constexpr int SFB_BYTES = SF_ATOMS_K * NB128 * 512;
  static constexpr int SF_STAGE_BYTES = SFA_BYTES + SFB_BYTES;

  static constexpr int A_BYTES = BM * ROW_BYTES;
  static constexpr int B_BYTES = B_ROWS * ROW_BYTES;
  // bytes a ring stage's full barrier counts (A and B tiles) and, for the
  // block-scaled kinds, its sf_full barrier (the stage's scale atoms, loaded
  // first, so their copies to TMEM overlap the operands' flight); a pair's
  // leader counts both CTAs' loads
  static constexpr uint32_t STAGE_TX = PAIR ? 2 * (A_BYTES + B_BYTES) : A_BYTES + B_BYTES;
  static constexpr uint32_t SF_TX = PAIR ? 2 * SF_STAGE_BYTES : SF_STAGE_BYTES;

  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SF_END = OFF_SF + STAGES * SF_STAGE_BYTES;
  // Output staging: each epilogue warp writes blocks of 32 rows that a bulk
  // tensor store copies to global memory: 32 columns (bf16 / fp16: 2 KB with
  // the 64-byte swizzle; fp32: 4 KB with the 128-byte swizzle) or 16 columns
  // of a 16-bit type (1 KB with the 32-byte swizzle).
  static constexpr int OUT_BUFS = OUT_BUFS_;
  static constexpr bool STORE_TMA = OUT_BUFS_ > 0;
  static constexpr int OUT_COLS = OUT_COLS_;
  static constexpr int OUT_BLOCK_BYTES = 32 * OUT_COLS * OUT_ELEM_BYTES;
  static constexpr int OFF_OUT = (OFF_SF_END + 1023) & ~1023;
  static constexpr int OFF_BAR = OFF_OUT + EPI_WARPS * OUT_BUFS * OUT_BLOCK_BYTES;
  // ring full/empty, accumulator full/empty, drain, and (block-scaled kinds)
  // a slot's scales copied to TMEM and a slot's scale atoms landed
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1 + (MX ? 2 * STAGES : 0);
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  // + slack to align the base to 1024 bytes where it fits; a layout without it
  // takes the dynamic shared-memory base as it comes (1024-aligned when the
  // kernel has no static shared memory) and checks that at entry
  static constexpr int ALIGN_SLACK = SMEM_USED + 1024 <= 232448 ? 1024 : 0;
  static constexpr int SMEM_BYTES = SMEM_USED + ALIGN_SLACK;

  static constexpr int COL_ACC = 0;
  static constexpr int COL_SUM = ACC_BUFS * BN;
  static constexpr int COL_SF = COL_SUM + (INT_CHUNKS && !REG_SUMS ? BN : 0);
  static constexpr int SF_COLS_A = SF_ATOMS_K * 4;
  static constexpr int SF_COLS_B = SF_ATOMS_K * NB128 * 4;
  static constexpr int SF_COLS_STAGE = MX ? SF_COLS_A + SF_COLS_B : 0;
  static constexpr int COLS_USED = COL_SF + STAGES * SF_COLS_STAGE;
  static constexpr int TMEM_COLS = COLS_USED <= 32    ? 32
                                   : COLS_USED <= 64  ? 64
                                   : COLS_USED <= 128 ? 128
                                   : COLS_USED <= 256 ? 256
                                                      : 512;

  static constexpr int NUM_THREADS = 32 * (4 + EPI_WARPS);

  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile N");
  static_assert(EPI_WARPS % 4 == 0 && EPI_COLS % 32 == 0, "epilogue split");
  static_assert(!REG_SUMS || EPI_COLS == 64 || (BLOCKSCALE && EPI_COLS == 32),
                "register sums hold 64 columns per thread (32 for blockscale)");
  static_assert(!BLOCKSCALE || REG_SUMS, "blockscale sums live in registers");
  static_assert(COLS_USED <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared-memory budget");
  static_assert(OUT_COLS == 32 || (OUT_COLS == 16 && OUT_ELEM_BYTES == 2), "staging block width");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms need 1024-byte alignment");
  static_assert(!MX || BN % 128 == 0, "scale atoms cover 128 rows of B");

  // Ring-slot arrivals: the producer's (a pair's leader counts both CTAs' TMA
  // bytes; each CTA of a pair loads the scale atoms of its own 128 rows of A
  // and of all BN rows of B at the same offsets).  Scale copies to TMEM: one
  // commit from each of the two copy threads.
  static constexpr uint32_t FULL_ARRIVALS = 1;
  static constexpr uint32_t SF_COPIERS = 2;

  // kind::f16: D fp32 (1), A/B f16 (0).  kind::f8f6f4: A/B E4M3 (0).
  // kind::mxf8f6f4: E4M3 (0).  kind::mxf4: E2M1 (1), UE8M0 scales.
  // kind::mxf4nvf4 (NVFP4): E2M1 (1), UE4M3 scales.
  __host__ __device__ static constexpr uint32_t idesc(uint32_t a_sf_id, uint32_t b_sf_id) {
    return KIND == Kind::F16    ? make_idesc_dense(1, 0, 0, MMA_M, BN)
           : DENSE_F8           ? make_idesc_dense(1, 0, 0, MMA_M, BN)
           : KIND == Kind::MXF8 ? make_idesc_block_scaled(0, 0, MMA_M, BN, a_sf_id, b_sf_id)
           : KIND == Kind::MXF4 ? make_idesc_block_scaled(1, 1, MMA_M, BN, a_sf_id, b_sf_id)
                                : make_idesc_block_scaled(1, 1, MMA_M, BN, a_sf_id, b_sf_id, false);
  }
};

// Work unit u: its tile t, its k-blocks [kb0, kb1) and its K-part (-1: the
// whole tile).
template <class C>
__device__ __forceinline__ void unit_of(const GemmParams& p, int u, int& t, int& kb0, int& kb1, int& kpart) {
  if (!C::SPLITTABLE || u < p.full_tiles) {
    t = u;
    kb0 = 0;
    kb1 = p.num_kb;
    kpart = -1;
    return;
  }
  const int v = u - p.full_tiles;
  t = p.full_tiles + v / p.split;
  kpart = v % p.split;
  kb0 = kpart * p.split_kb;
  kb1 = min(p.num_kb, kb0 + p.split_kb);
}

template <class C>
__device__ __forceinline__ int num_units(const GemmParams& p) {
  return C::SPLITTABLE ? p.num_units : p.num_tiles;
}

// One K-part's arrival at its region's word (the call's tag in the high 56
// bits, the arrivals so far in the low 8; a word holding another tag counts
// as none).  Returns true for the last of `parts` arrivals, which leaves the
// word at 0 for the next call (or graph replay).  Each failed exchange means
// another arrival succeeded, so the loop ends within `parts` rounds.
__device__ __forceinline__ bool split_arrive(unsigned long long* word, unsigned long long tag, int parts,
                                             unsigned long long* err) {
  unsigned long long old = atomicAdd(word, 0ull);
#pragma unroll 1
  for (int i = 0; i < 64; ++i) {
    const unsigned long long cnt = (old & ~0xFFull) == tag ? (old & 0xFFull) : 0ull;
    const bool last = cnt + 1 == static_cast<unsigned long long>(parts);
    const unsigned long long seen = atomicCAS(word, old, last ? 0ull : (tag | (cnt + 1)));
    if (seen == old) return last;
    old = seen;
  }
  report_error(err, kDevErrTimeout, kSiteSplitArrive, 0u);
  return false;
}

__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& mb, int& nb) {
  const int group_tiles = p.group_m * p.num_n_blocks;
  const int g = t / group_tiles;
  const int first_m = g * p.group_m;
  const int gm = min(p.num_m_blocks - first_m, p.group_m);
  const int local = t - g * group_tiles;
  mb = first_m + local % gm;
  nb = local / gm;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Two fp32 fused multiply-adds in one instruction (fma.rn.f32x2, sm_100 and
// later): (d0, d1) = (a0 * b + d0, a1 * b + d1), each half rounded to nearest
// even exactly as a scalar fma.rn.f32 would round it.
__device__ __forceinline__ void fma2_rn(uint32_t& d0, uint32_t& d1, uint32_t a0, uint32_t a1, float b) {
  asm("{\n .reg .b64 rd, ra, rb;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n mov.b64 rd, {%0, %1};\n"
      " fma.rn.f32x2 rd, ra, rb, rd;\n mov.b64 {%0, %1}, rd;\n}"
      : "+r"(d0), "+r"(d1)
      : "r"(a0), "r"(a1), "r"(__float_as_uint(b)));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two fp32 products in one instruction (mul.rn.f32x2): each half rounded to
// nearest even exactly as a scalar mul.rn.f32 would.  Only products use the
// paired form: a paired multiply followed by a paired add was measured to
// come out fused into one multiply-add, so additions that must round on
// their own stay scalar __fadd_rn, which is never merged.
__device__ __forceinline__ void mul2_rn(float& x0, float& x1, float b0, float b1) {
  asm("{\n .reg .b64 rx, rb;\n mov.b64 rx, {%0, %1};\n mov.b64 rb, {%2, %3};\n"
      " mul.rn.f32x2 rx, rx, rb;\n mov.b64 {%0, %1}, rx;\n}"
      : "+f"(x0), "+f"(x1)
      : "f"(b0), "f"(b1));
}

// Two fp32 values to bf16 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The same for fp16 (round to nearest even; beyond 65504 rounds to +-inf).
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <OutType OT>
__device__ __forceinline__ uint32_t pack_out16x2(float lo, float hi) {
  if constexpr (OT == OutType::F16) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

// Epilogue of COLS (32 or 16) consecutive columns [n0, n0+COLS) of one row m,
// in steps of 8 columns (8 column scales, 8 biases live at a time), written to
// row `lane` of a 32-row staging block with the swizzle the output tensor map
// uses: 32 bf16 / fp16 columns: rows of 64 bytes, 16-byte chunk c of row r at
// 64r + 16(c ^ ((r >> 1) & 3)); 16 columns: rows of 32 bytes, chunk c at
// 32r + 16(c ^ ((r >> 2) & 1)); 32 fp32 columns: rows of 128 bytes, at
// 128r + 16(c ^ (r & 7)).
// INT_ACC: v holds int32 sums; otherwise fp32 bit patterns.  Columns past N
// (N is a multiple of 8) read no scale or bias; the bulk store clips them.
// ALPHA: multiply by `sam` (the NVFP4 per-tensor scale product) before the bias.
template <bool ROWWISE, bool INT_ACC, int OFF = 0, bool ALPHA = false, OutType OT = OutType::BF16, int COLS = 32,
          int LEN = 32>
__device__ __forceinline__ void epilogue_row32(const GemmParams& p, int n0, float sam, const uint32_t (&v)[LEN],
                                               uint32_t block, int lane) {
  static_assert(COLS == 32 || (COLS == 16 && OT != OutType::F32), "staging block width");
  const bool has_bias = p.bias != nullptr;
#pragma unroll
  for (int s8 = 0; s8 < COLS / 8; ++s8) {
    const int n = n0 + 8 * s8;
    const bool in = n < p.N;
    float sbv[8];
    float bv[8];
    if constexpr (ROWWISE) {
      const float4 t0 = in ? __ldg(reinterpret_cast<const float4*>(p.sb + n)) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 t1 = in ? __ldg(reinterpret_cast<const float4*>(p.sb + n) + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
      sbv[0] = t0.x; sbv[1] = t0.y; sbv[2] = t0.z; sbv[3] = t0.w;
      sbv[4] = t1.x; sbv[5] = t1.y; sbv[6] = t1.z; sbv[7] = t1.w;
    }
    if (has_bias) {
      const uint4 t = in ? __ldg(reinterpret_cast<const uint4*>(p.bias + n)) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t wv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bv[2 * j + 0] = __uint_as_float(wv[j] << 16);
        bv[2 * j + 1] = __uint_as_float(wv[j] & 0xFFFF0000u);
      }
    }
    uint32_t packed[8];  // fp32: all 8 values; 16-bit types: 4 pairs
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const uint32_t r0 = v[OFF + 8 * s8 + i], r1 = v[OFF + 8 * s8 + i + 1];
      float x0 = INT_ACC ? __int2float_rn(static_cast<int>(r0)) : __uint_as_float(r0);
      float x1 = INT_ACC ? __int2float_rn(static_cast<int>(r1)) : __uint_as_float(r1);
      if constexpr (ROWWISE) {
        mul2_rn(x0, x1, sam, sam);
        mul2_rn(x0, x1, sbv[i], sbv[i + 1]);
      }
      if constexpr (ALPHA) mul2_rn(x0, x1, sam, sam);
      if (has_bias) {
        x0 = __fadd_rn(x0, bv[i]);
        x1 = __fadd_rn(x1, bv[i + 1]);
      }
      if constexpr (OT == OutType::F32) {
        packed[i] = __float_as_uint(x0);
        packed[i + 1] = __float_as_uint(x1);
      } else {
        packed[i / 2] = pack_out16x2<OT>(x0, x1);
      }
    }
    if constexpr (OT == OutType::F32) {
      const uint32_t row = block + 128 * lane;
      st_shared_v4(row + 16 * ((2 * s8) ^ (lane & 7)), packed[0], packed[1], packed[2], packed[3]);
      st_shared_v4(row + 16 * ((2 * s8 + 1) ^ (lane & 7)), packed[4], packed[5], packed[6], packed[7]);
    } else if constexpr (COLS == 32) {
      st_shared_v4(block + 64 * lane + 16 * (s8 ^ ((lane >> 1) & 3)), packed[0], packed[1], packed[2], packed[3]);
    } else {
      st_shared_v4(block + 32 * lane + 16 * (s8 ^ ((lane >> 2) & 1)), packed[0], packed[1], packed[2], packed[3]);
    }
  }
}

// The same epilogue with the 8-column pieces stored straight to row m of the
// output (16-byte stores; no staging).
template <bool ROWWISE, bool INT_ACC, int OFF = 0, bool ALPHA = false, OutType OT = OutType::BF16, int LEN = 32>
__device__ __forceinline__ void epilogue_row32_global(const GemmParams& p, int m, int n0, float sam,
                                                      const uint32_t (&v)[LEN]) {
  const bool has_bias = p.bias != nullptr;
  const size_t first = static_cast<size_t>(m) * static_cast<size_t>(p.N) + n0;
#pragma unroll
  for (int s8 = 0; s8 < 4; ++s8) {
    const int n = n0 + 8 * s8;
    if (n < p.N) {
      float sbv[8];
      float bv[8];
      if constexpr (ROWWISE) {
        const float4 t0 = __ldg(reinterpret_cast<const float4*>(p.sb + n));
        const float4 t1 = __ldg(reinterpret_cast<const float4*>(p.sb + n) + 1);
        sbv[0] = t0.x; sbv[1] = t0.y; sbv[2] = t0.z; sbv[3] = t0.w;
        sbv[4] = t1.x; sbv[5] = t1.y; sbv[6] = t1.z; sbv[7] = t1.w;
      }
      if (has_bias) {
        const uint4 t = __ldg(reinterpret_cast<const uint4*>(p.bias + n));
        const uint32_t wv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          bv[2 * j + 0] = __uint_as_float(wv[j] << 16);
          bv[2 * j + 1] = __uint_as_float(wv[j] & 0xFFFF0000u);
        }
      }
      uint32_t packed[8];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const uint32_t r0 = v[OFF + 8 * s8 + i], r1 = v[OFF + 8 * s8 + i + 1];
        float x0 = INT_ACC ? __int2float_rn(static_cast<int>(r0)) : __uint_as_float(r0);
        float x1 = INT_ACC ? __int2float_rn(static_cast<int>(r1)) : __uint_as_float(r1);
        if constexpr (ROWWISE) {
          mul2_rn(x0, x1, sam, sam);
          mul2_rn(x0, x1, sbv[i], sbv[i + 1]);
        }
        if constexpr (ALPHA) mul2_rn(x0, x1, sam, sam);
        if (has_bias) {
          x0 = __fadd_rn(x0, bv[i]);
          x1 = __fadd_rn(x1, bv[i + 1]);
        }
        if constexpr (OT == OutType::F32) {
          packed[i] = __float_as_uint(x0);
          packed[i + 1] = __float_as_uint(x1);
        } else {
          packed[i / 2] = pack_out16x2<OT>(x0, x1);
        }
      }
      if constexpr (OT == OutType::F32) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(p.out) + first) + 2 * s8;
        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
      } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + first);
        dst[s8] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
    }
  }
}

// One epilogue warp's output block: waits until its staging buffer is free,
// fills it (per lane one row), and issues the bulk store of the 32x32 block at
// (row m_block, column n0).  `count` numbers the warp's blocks.
template <bool INT, int OFF>
struct EmitTag {
  static constexpr bool kInt = INT;
  static constexpr int kOff = OFF;
};

struct OutStager {
  uint32_t base;    // this warp's first staging buffer (shared address)
  uint32_t count;   // blocks issued so far
};

template <class C>
__device__ __forceinline__ uint32_t out_block_acquire(OutStager& o, int lane) {
  if (lane == 0) bulk_wait_group_read<(C::OUT_BUFS > 0 ? C::OUT_BUFS - 1 : 0)>();
  __syncwarp();
  return o.base + (o.count % (C::OUT_BUFS > 0 ? C::OUT_BUFS : 1)) * C::OUT_BLOCK_BYTES;
}

template <class C>
__device__ __forceinline__ void out_block_release(OutStager& o, uint32_t block, const CUtensorMap* tmOut, int n0,
                                                  int m_block, int lane) {
  fence_proxy_async_smem();  // the block's generic writes before the bulk copy reads it
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmOut, block, n0, m_block);
    bulk_commit_group();
  }
  ++o.count;
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Scale-factor copies of the MMA-issuing CTA (block-scaled kinds), one of
// two threads: per ring slot, once the slot's scale atoms have landed
// (sf_full: both CTAs' atoms in a pair; the producer loads them before the
// operand tiles) and the MMAs of the slot's previous round have completed
// (empty), copy the atoms i with i % 2 == part into the slot's
// TMEM columns and commit to sf_ready, which counts both threads.  Atoms in
// shared memory: A's SF_ATOMS_K first, then B's 128-row blocks one after the
// other (each SF_ATOMS_K atoms); in TMEM: A's, then B's grouped by K-group
// (the NB128 row blocks of a K-group side by side, as the MMA reads them).
template <class C>
__device__ __forceinline__ void scale_copier(const GemmParams& p, uint8_t* smem, uint32_t tmem, uint64_t* sf_full,
                                             uint64_t* sf_ready, uint64_t* empty, const WaitCtl& w, int tile0,
                                             int tile_step, int part) {
  int stage = 0;
  uint32_t phase = 0;
  long long issued = 0;
  bool ok = true;
#pragma unroll 1
  for (int u = tile0; ok && u < num_units<C>(p); u += tile_step) {
    int t, ukb0, ukb1, kpart;
    unit_of<C>(p, u, t, ukb0, ukb1, kpart);
#pragma unroll 1
    for (int kb = ukb0; kb < ukb1; ++kb) {
      bool ready = mbar_wait(&sf_full[stage], phase, w, kSiteScaleCopy);
      // the slot's TMEM scales of the previous round have been read by their MMAs
      ready = ready && mbar_wait(&empty[stage], phase ^ 1u, w, kSiteScaleCopy);
      if (!ready) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t sf_tmem = tmem + static_cast<uint32_t>(C::COL_SF + stage * C::SF_COLS_STAGE);
      const uint32_t sf_smem = smem_u32(smem + C::OFF_SF + stage * C::SF_STAGE_BYTES);
#pragma unroll
      for (int i = part; i < C::SF_ATOMS_K + C::SF_ATOMS_K * C::NB128; i += 2) {
        uint32_t col, src;
        if (i < C::SF_ATOMS_K) {
          col = 4 * i;
          src = sf_smem + 512 * i;
        } else {
          const int b = i - C::SF_ATOMS_K;  // TMEM order: K-group g = b / NB128, row block rb = b % NB128
          col = C::SF_COLS_A + 4 * b;
          src = sf_smem + C::SFA_BYTES + 512 * ((b % C::NB128) * C::SF_ATOMS_K + b / C::NB128);
        }
        if constexpr (C::PAIR) {
          tmem_cp_32x128b_warpx4_pair(sf_tmem + col, make_smem_desc(src, 128, 128, 0));
        } else {
          tmem_cp_32x128b_warpx4(sf_tmem + col, make_smem_desc(src, 128, 128, 0));
        }
      }
      if constexpr (C::PAIR) {
        umma_commit_pair(&sf_ready[stage]);
      } else {
        umma_commit(&sf_ready[stage]);
      }
      ++issued;
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  // leave no copy in flight: this thread's last commit covers its earlier copies
  if (issued > 0) {
    const long long L = issued - 1;
    const uint32_t a = smem_u32(&sf_ready[static_cast<int>(L % C::STAGES)]);
    const uint32_t par = static_cast<uint32_t>((L / C::STAGES) & 1);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(a, par)) {
      if (global_timer_ns() - t0 > p.timeout_ns) {
        report_error(p.err, kDevErrTimeout, kSiteScaleCopy, static_cast<uint32_t>(L));
        break;
      }
    }
  }
}

template <class C>
__global__ void __launch_bounds__(C::NUM_THREADS, 1)
    qk_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                   const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if constexpr (C::ALIGN_SLACK == 0) {
    // no room to align the base: give up (before any barrier, TMEM or cluster
    // step, in every CTA alike) if it is not aligned
    if ((smem_u32(smem_raw) & 1023u) != 0u) {
      if (threadIdx.x == 0) report_error(p.err, kDevErrSmemBase, kSiteSmemBase, smem_u32(smem_raw));
      return;
    }
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + C::ACC_BUFS;
  uint64_t* drain = acc_empty + C::ACC_BUFS;
  uint64_t* sf_ready = drain + 1;  // block-scaled kinds: a slot's scales copied to TMEM
  uint64_t* sf_full = sf_ready + C::STAGES;  // block-scaled kinds: a slot's scale atoms landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = C::CTAS > 1 ? cluster_ctarank() : 0u;  // CTA within the cluster
  const bool leader = rank == 0u;                           // a pair's MMA issuer
  const bool issues_mma = C::PAIR ? leader : true;
  // tiles are walked per cluster (one CTA or a pair)
  const int tile0 = static_cast<int>(blockIdx.x) / C::CTAS;
  const int tile_step = static_cast<int>(gridDim.x) / C::CTAS;

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], C::FULL_ARRIVALS);
      mbar_init(&empty[s], 1u);
      if constexpr (C::MX) {
        mbar_init(&sf_ready[s], C::SF_COPIERS);
        mbar_init(&sf_full[s], 1u);
      }
    }
#pragma unroll 1
    for (int a = 0; a < C::ACC_BUFS; ++a) {
      mbar_init(&acc_full[a], 1u);
      // A pair's epilogue warps arrive on their own CTA's barrier; the peer's
      // relay thread forwards the peer's completion to the leader, whose
      // barrier therefore counts its own warps plus one relay arrival.
      mbar_init(&acc_empty[a], static_cast<uint32_t>(C::EPI_WARPS + (C::PAIR && leader ? 1 : 0)));
    }
    mbar_init(drain, 1u);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
    if (C::MX) {
      tma_prefetch_desc(&tmSA);
      tma_prefetch_desc(&tmSB);
    }
  }
  if (warp == 1) {
    if constexpr (C::PAIR) {
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (C::CTAS > 1) cluster_sync();  // peers' barriers exist before anyone signals them
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{abort_flag, p.err, p.timeout_ns};

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // the kernel this one may overlap (programmatic launch) has completed:
      // the scale-atom pre-pass (block-scaled kinds) or the int8 -> f16
      // widening pass (exact INT8), whose outputs the first loads read
      if constexpr (C::MX || C::INT_CHUNKS) griddep_wait();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      // in a pair, both CTAs' loads complete on the leader's ring barriers
      const uint32_t full_leader = C::PAIR ? mapa_shared(smem_u32(&full[0]), 0u) : 0u;
      [[maybe_unused]] const uint32_t sf_full_leader = C::MX && C::PAIR ? mapa_shared(smem_u32(&sf_full[0]), 0u) : 0u;
#pragma unroll 1
      for (int u = tile0; ok && u < num_units<C>(p); u += tile_step) {
        int t, ukb0, ukb1, kpart;
        unit_of<C>(p, u, t, ukb0, ukb1, kpart);
        int mb, nb;
        tile_coords(p, t, mb, nb);
        const int a_row = mb * C::TILE_M + static_cast<int>(rank) * C::BM;
        const int b_row = nb * C::BN + static_cast<int>(rank) * C::B_LOAD_ROWS;
#pragma unroll 1
        for (int kb = ukb0; kb < ukb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, w, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          if constexpr (C::MX) {
            // the stage's scale atoms first, on their own barrier: A's 128-row
            // block, then each 128-row block of the B tile; atom maps are
            // [blocks * gpad * 2, 256 bytes], a box being SF_ATOMS_K
            // consecutive atoms of one block
            uint8_t* sf = smem + C::OFF_SF + stage * C::SF_STAGE_BYTES;
            const int ya = ((a_row / 128) * p.sf_gpad + kb * C::SF_ATOMS_K) * 2;
            if constexpr (C::PAIR) {
              if (leader) mbar_arrive_expect_tx(&sf_full[stage], C::SF_TX);
              const uint32_t fb = sf_full_leader + 8u * static_cast<uint32_t>(stage);
              tma_load_2d_pair(sf, &tmSA, fb, 0, ya);
#pragma unroll
              for (int rb = 0; rb < C::NB128; ++rb)
                tma_load_2d_pair(sf + C::SFA_BYTES + rb * C::SF_ATOMS_K * 512, &tmSB, fb, 0,
                                 ((nb * C::NB128 + rb) * p.sf_gpad + kb * C::SF_ATOMS_K) * 2);
            } else {
              mbar_arrive_expect_tx(&sf_full[stage], C::SF_TX);
              tma_load_2d(sf, &tmSA, &sf_full[stage], 0, ya);
#pragma unroll
              for (int rb = 0; rb < C::NB128; ++rb)
                tma_load_2d(sf + C::SFA_BYTES + rb * C::SF_ATOMS_K * 512, &tmSB, &sf_full[stage], 0,
                            ((nb * C::NB128 + rb) * p.sf_gpad + kb * C::SF_ATOMS_K) * 2);
            }
          }
          if constexpr (C::PAIR) {
            if (leader) mbar_arrive_expect_tx(&full[stage], C::STAGE_TX);
            const uint32_t fb = full_leader + 8u * static_cast<uint32_t>(stage);
            tma_load_2d_pair(smem + C::OFF_A + stage * C::A_BYTES, &tmA, fb, kb * C::TMA_K, a_row);
            tma_load_2d_pair(smem + C::OFF_B + stage * C::B_BYTES, &tmB, fb, kb * C::TMA_K, b_row);
          } else {
            mbar_arrive_expect_tx(&full[stage], C::STAGE_TX);
            tma_load_2d(smem + C::OFF_A + stage * C::A_BYTES, &tmA, &full[stage], kb * C::TMA_K, a_row);
            tma_load_2d(smem + C::OFF_B + stage * C::B_BYTES, &tmB, &full[stage], kb * C::TMA_K, b_row);
          }
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Do not leave the CTA with tile loads in flight: wait (bounded) for the
      // most recent load of every ring slot.  In a pair only the leader's
      // barriers count the loads; the peer is held by the final cluster
      // barrier until the leader has seen them land.
      const WaitCtl wd{abort_flag, p.err, p.timeout_ns};
      const long long drain_n = issues_mma ? (issued < C::STAGES ? issued : C::STAGES) : 0;
#pragma unroll 1
      for (long long i = 0; i < drain_n; ++i) {
        const long long L = issued - 1 - i;
        const uint32_t par = static_cast<uint32_t>((L / C::STAGES) & 1);
#pragma unroll
        for (int which = 0; which < (C::MX ? 2 : 1); ++which) {
          uint64_t* bar = which == 0 ? &full[static_cast<int>(L % C::STAGES)] : &sf_full[static_cast<int>(L % C::STAGES)];
          const uint32_t a = smem_u32(bar);
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(a, par)) {
            if (global_timer_ns() - t0 > wd.timeout_ns) {
              report_error(p.err, kDevErrTimeout, kSiteProducerDrain, static_cast<uint32_t>(L));
              break;
            }
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (the leader CTA of a pair) ----------------
    if (lane == 0 && issues_mma) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_iter = 0;
      bool ok = true;
#pragma unroll 1
      for (int u = tile0; ok && u < num_units<C>(p); u += tile_step) {
        int t, ukb0, ukb1, kpart;
        unit_of<C>(p, u, t, ukb0, ukb1, kpart);
#pragma unroll 1
        for (int c = 0; ok && c < p.num_chunks; ++c) {
          const int a = static_cast<int>(acc_iter % C::ACC_BUFS);
          const uint32_t aph = (acc_iter / C::ACC_BUFS) & 1u;
          const bool got = C::PAIR ? mbar_wait_cluster(&acc_empty[a], aph ^ 1u, w, kSiteMmaAccEmpty)
                                   : mbar_wait(&acc_empty[a], aph ^ 1u, w, kSiteMmaAccEmpty);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem + static_cast<uint32_t>(C::COL_ACC + a * C::BN);
          // one chunk per unit for the splittable kinds (its k-blocks)
          const int kb0 = C::SPLITTABLE ? ukb0 : c * p.chunk_kb;
          const int kb1 = C::SPLITTABLE ? ukb1 : min(p.num_kb, kb0 + p.chunk_kb);
#pragma unroll 1
          for (int kb = kb0; kb < kb1; ++kb) {
            bool landed = mbar_wait(&full[stage], phase, w, kSiteMmaFull);
            // block-scaled kinds: the k-block's scale factors are in TMEM (copied by warp 3)
            if constexpr (C::MX) landed = landed && mbar_wait(&sf_ready[stage], phase, w, kSiteMmaScales);
            if (!landed) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t sf_tmem = tmem + static_cast<uint32_t>(C::COL_SF + stage * C::SF_COLS_STAGE);
            const uint64_t adesc = make_desc_kmajor_sw128(smem_u32(smem + C::OFF_A + stage * C::A_BYTES));
            const uint64_t bdesc = make_desc_kmajor_sw128(smem_u32(smem + C::OFF_B + stage * C::B_BYTES));
            int ksteps = C::K_STEPS;
            if (kb == p.num_kb - 1) {
              const int rem = p.K - kb * C::K_ELEMS;
              ksteps = min(C::K_STEPS, (rem + C::UMMA_K - 1) / C::UMMA_K);
            }
#pragma unroll
            for (int j = 0; j < C::K_STEPS; ++j) {
              if (j < ksteps) {
                const uint32_t accum = (kb > kb0 || j > 0) ? 1u : 0u;
                const uint64_t ad = adesc + static_cast<uint64_t>((j * 32) >> 4);
                const uint64_t bd = bdesc + static_cast<uint64_t>((j * 32) >> 4);
                if constexpr (C::kind == Kind::F16 && C::PAIR) {
                  umma_f16_pair(d_tmem, ad, bd, C::idesc(0, 0), accum);
                } else if constexpr (C::DENSE_F8 && C::PAIR) {
                  umma_f8f6f4_pair(d_tmem, ad, bd, C::idesc(0, 0), accum);
                } else if constexpr (C::kind == Kind::F16) {
                  umma_f16(d_tmem, ad, bd, C::idesc(0, 0), accum);
                } else if constexpr (C::DENSE_F8) {
                  umma_f8f6f4(d_tmem, ad, bd, C::idesc(0, 0), accum);
                } else if constexpr (C::kind == Kind::MXF8) {
                  // one scale byte per row per MMA: byte j of the stage's column
                  if constexpr (C::PAIR) {
                    umma_mxf8f6f4_pair(d_tmem, ad, bd, C::idesc(j, j), sf_tmem, sf_tmem + C::SF_COLS_A, accum);
                  } else {
                    umma_mxf8f6f4(d_tmem, ad, bd, C::idesc(j, j), sf_tmem, sf_tmem + C::SF_COLS_A, accum);
                  }
                } else if constexpr (C::kind == Kind::NVF4) {
                  // four UE4M3 scale bytes (one per 16 K) per row per MMA: all of column group j
                  if constexpr (C::PAIR) {
                    umma_nvf4_pair(d_tmem, ad, bd, C::idesc(0, 0), sf_tmem + 4 * j,
                                   sf_tmem + C::SF_COLS_A + 4 * C::NB128 * j, accum);
                  } else {
                    umma_nvf4(d_tmem, ad, bd, C::idesc(0, 0), sf_tmem + 4 * j,
                              sf_tmem + C::SF_COLS_A + 4 * C::NB128 * j, accum);
                  }
                } else {
                  // two scale bytes per row per MMA: bytes 2(j%2), 2(j%2)+1 of column group j/2
                  const uint32_t g = static_cast<uint32_t>(j >> 1);
                  const uint32_t id = static_cast<uint32_t>((j & 1) * 2);
                  if constexpr (C::PAIR) {
                    umma_mxf4_pair(d_tmem, ad, bd, C::idesc(id, id), sf_tmem + 4 * g,
                                   sf_tmem + C::SF_COLS_A + 4 * C::NB128 * g, accum);
                  } else {
                    umma_mxf4(d_tmem, ad, bd, C::idesc(id, id), sf_tmem + 4 * g,
                              sf_tmem + C::SF_COLS_A + 4 * C::NB128 * g, accum);
                  }
                }
              }
            }
            if constexpr (C::PAIR) {
              umma_commit_pair_multicast(&empty[stage], 0x3);  // frees the slot in both CTAs
            } else {
              umma_commit(&empty[stage]);
            }
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if constexpr (C::PAIR) {
            umma_commit_pair_multicast(&acc_full[a], 0x3);
          } else {
            umma_commit(&acc_full[a]);
          }
          ++acc_iter;
        }
      }
      // Every MMA and copy this thread issued completes before TMEM is freed.
      if constexpr (C::PAIR) {
        umma_commit_pair(drain);
      } else {
        umma_commit(drain);
      }
      const uint32_t da = smem_u32(drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(da, 0u)) {
        if (global_timer_ns() - t0 > p.timeout_ns) {
          report_error(p.err, kDevErrTimeout, kSiteDrain, 0u);
          break;
        }
      }
    } else if (C::PAIR && lane == 0) {
      // ---------------- accumulator relay (the peer CTA of a pair) ----------------
      // Once all of this CTA's epilogue warps have drained an accumulator,
      // tell the leader's MMA issuer with one remote arrive.
      const uint32_t acc_empty_leader = mapa_shared(smem_u32(&acc_empty[0]), 0u);
      uint32_t acc_iter = 0;
      bool ok = true;
#pragma unroll 1
      for (int u = tile0; ok && u < num_units<C>(p); u += tile_step) {
#pragma unroll 1
        for (int c = 0; c < p.num_chunks; ++c) {
          const int a = static_cast<int>(acc_iter % C::ACC_BUFS);
          if (!mbar_wait(&acc_empty[a], (acc_iter / C::ACC_BUFS) & 1u, w, kSiteMmaAccEmpty)) {
            ok = false;
            break;
          }
          // CTA-scope release: the drained accumulator carries no data the
          // leader reads, and tcgen05.wait::ld already completed the reads
          mbar_arrive_remote(acc_empty_leader + 8u * static_cast<uint32_t>(a));
          ++acc_iter;
        }
      }
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    // ---------------- scale-factor copies (block-scaled kinds, the MMA-issuing CTA) ----------------
    if constexpr (C::MX) {
      if (issues_mma && lane == 0) scale_copier<C>(p, smem, tmem, sf_full, sf_ready, empty, w, tile0, tile_step, warp - 2);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                          // TMEM lane quarter of this warp
    const int part = (warp - 4) >> 2;                // which EPI_COLS-wide column part
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int col_part = part * C::EPI_COLS;
    OutStager ostg{smem_u32(smem + C::OFF_OUT) +
                       static_cast<uint32_t>((warp - 4) * C::OUT_BUFS * C::OUT_BLOCK_BYTES),
                   0u};
    uint32_t acc_iter = 0;
    bool ok = true;
    float alpha = 1.f;  // NVFP4: product of the per-tensor scales, one fp32 rounding
    if constexpr (C::ALPHA) alpha = __fmul_rn(p.ga ? __ldg(p.ga) : 1.f, p.gb ? __ldg(p.gb) : 1.f);
    // accumulator releases go to the leader CTA's barrier
    // accumulator releases go to this CTA's barrier (the arrive on the
    // leader's barrier is left to the peer's single relay thread)
    auto release = [&](int a) {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);
    };
#pragma unroll 1
    for (int u = tile0; ok && u < num_units<C>(p); u += tile_step) {
      int t, ukb0, ukb1, kpart;
      unit_of<C>(p, u, t, ukb0, ukb1, kpart);
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int m_block = mb * C::TILE_M + static_cast<int>(rank) * C::BM + q * 32;  // row of lane 0
      const int m = m_block + lane;
      const bool row_ok = m < p.M;
      const bool block_ok = m_block < p.M;  // warp-uniform: any row of this block inside M
      float sam = 1.f;
      if constexpr (C::ROWWISE) sam = row_ok ? __ldg(p.sa + m) : 0.f;
      if constexpr (C::ALPHA) sam = alpha;
      const int n_tile = nb * C::BN + col_part;
      [[maybe_unused]] uint32_t sums[C::REG_SUMS ? C::EPI_COLS : 1];
      // blockscale: the first K-block's scales (later ones are loaded a chunk ahead)
      [[maybe_unused]] const bool col_in = n_tile < p.N;
      [[maybe_unused]] float sa_next = 0.f, sb_next = 0.f;
      if constexpr (C::BLOCKSCALE) {
        sa_next = row_ok ? __ldg(p.sa + static_cast<size_t>(m) * p.scale_kb) : 0.f;
        sb_next = col_in ? __ldg(p.sb + static_cast<size_t>(n_tile >> 7) * p.scale_kb) : 0.f;
#pragma unroll
        for (int i = 0; i < C::EPI_COLS; ++i) sums[i] = 0u;
      }
#pragma unroll 1
      for (int c = 0; c < p.num_chunks; ++c) {
        const int a = static_cast<int>(acc_iter % C::ACC_BUFS);
        const uint32_t aph = (acc_iter / C::ACC_BUFS) & 1u;
        if (!mbar_wait(&acc_full[a], aph, w, kSiteEpiAccFull)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const bool last = c == p.num_chunks - 1;
        const uint32_t acc_col = lane_base + static_cast<uint32_t>(C::COL_ACC + a * C::BN + col_part);
        // stages and stores one 32x32 output block from 32 values per lane
        auto emit = [&](auto tag, int n0, const auto& vals) {
          constexpr bool kInt = decltype(tag)::kInt;
          constexpr int kOff = decltype(tag)::kOff;
          if (!(block_ok && n0 < p.N)) return;
          if constexpr (C::STORE_TMA && C::OUT_COLS == 32) {
            const uint32_t block = out_block_acquire<C>(ostg, lane);
            epilogue_row32<C::ROWWISE || kInt, kInt, kOff, C::ALPHA, C::OUT>(p, n0, sam, vals, block, lane);
            out_block_release<C>(ostg, block, &tmOut, n0, m_block, lane);
          } else if constexpr (C::STORE_TMA) {
            // two 16-column blocks (the second one only where it starts inside N)
            uint32_t block = out_block_acquire<C>(ostg, lane);
            epilogue_row32<C::ROWWISE || kInt, kInt, kOff, C::ALPHA, C::OUT, 16>(p, n0, sam, vals, block, lane);
            out_block_release<C>(ostg, block, &tmOut, n0, m_block, lane);
            if (n0 + 16 < p.N) {
              block = out_block_acquire<C>(ostg, lane);
              epilogue_row32<C::ROWWISE || kInt, kInt, kOff + 16, C::ALPHA, C::OUT, 16>(p, n0 + 16, sam, vals, block,
                                                                                      lane);
              out_block_release<C>(ostg, block, &tmOut, n0 + 16, m_block, lane);
            }
          } else if (row_ok) {
            epilogue_row32_global<C::ROWWISE || kInt, kInt, kOff, C::ALPHA, C::OUT>(p, m, n0, sam, vals);
          }
        };
        if (C::SPLITTABLE && kpart >= 0) {
          // a K-part of a split tile: this warp's 32 rows x EPI_COLS columns go
          // to the workspace as fp32 (lane-contiguous 16-byte pieces), the
          // accumulator is released, and the warp whose part arrives last adds
          // the parts in K order, ((p0 + p1) + p2) ..., and emits the sum
          constexpr int PIECES = C::EPI_COLS / 4;
          const size_t region =
              (static_cast<size_t>(t - p.full_tiles) * C::CTAS + rank) * C::EPI_WARPS + static_cast<size_t>(warp - 4);
          float4* ws = reinterpret_cast<float4*>(p.split_ws) + region * static_cast<size_t>(p.split) * PIECES * 32;
          float4* mine = ws + static_cast<size_t>(kpart) * PIECES * 32;
#pragma unroll 1
          for (int g = 0; g < C::EPI_COLS / 32; ++g) {
            uint32_t v[32];
            tmem_ld_32cols(acc_col + 32 * g, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              __stcg(mine + (8 * g + i) * 32 + lane,
                     make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
          }
          release(a);
          __threadfence();  // this lane's partial before the arrival
          __syncwarp();
          int last = 0;
          if (lane == 0) last = split_arrive(p.split_cnt + region, p.split_tag, p.split, p.err) ? 1 : 0;
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) {
            __threadfence();  // the other parts' partials after their arrivals
            // BC columns at a time, all of a part's pieces in flight at once
            // (a one-piece-at-a-time loop waited for two L2 round trips per
            // piece; 64-column batches in the 8-warp configurations measured
            // no faster and took 168 registers against 110)
            constexpr int BC = 32;
            constexpr int NP = BC / 4;
#pragma unroll 1
            for (int g = 0; g < C::EPI_COLS / BC; ++g) {
              const float4* src = ws + (NP * g) * 32 + lane;
              float4 x[NP];
#pragma unroll
              for (int i = 0; i < NP; ++i) x[i] = __ldcg(src + 32 * i);
#pragma unroll 1
              for (int j = 1; j < p.split; ++j) {
                float4 y[NP];
#pragma unroll
                for (int i = 0; i < NP; ++i) y[i] = __ldcg(src + static_cast<size_t>(j) * PIECES * 32 + 32 * i);
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                  x[i].x = __fadd_rn(x[i].x, y[i].x);
                  x[i].y = __fadd_rn(x[i].y, y[i].y);
                  x[i].z = __fadd_rn(x[i].z, y[i].z);
                  x[i].w = __fadd_rn(x[i].w, y[i].w);
                }
              }
              uint32_t v[BC];
#pragma unroll
              for (int i = 0; i < NP; ++i) {
                v[4 * i] = __float_as_uint(x[i].x);
                v[4 * i + 1] = __float_as_uint(x[i].y);
                v[4 * i + 2] = __float_as_uint(x[i].z);
                v[4 * i + 3] = __float_as_uint(x[i].w);
              }
              emit(EmitTag<false, 0>{}, n_tile + BC * g, v);
              if constexpr (BC == 64) emit(EmitTag<false, 32>{}, n_tile + BC * g + 32, v);
            }
          }
        } else if constexpr (C::REG_DRAIN) {
          // one chunk per tile: four TMEM loads in flight, one wait, release the
          // accumulator, then the epilogue from registers while the MMAs go on
#pragma unroll
          for (int g = 0; g < C::EPI_COLS / 16; ++g)
            tmem_ld_16cols(acc_col + 16 * g, *reinterpret_cast<uint32_t(*)[16]>(&sums[16 * g]));
          tmem_wait_ld();
          release(a);
          emit(EmitTag<false, 0>{}, n_tile, sums);
          emit(EmitTag<false, 32>{}, n_tile + 32, sums);
        } else if constexpr (C::REG_SUMS && C::BLOCKSCALE) {
          // chunk c is K-block c: sums += partial * (sa[m, c] * sb[n / 128, c]);
          // this thread's columns lie in one 128-column block of B
          // (the sums start at +0 for each tile, so the first K-block gives
          // fma(partial, scale, +0); pairs of columns share one fma.rn.f32x2)
          const float scale = __fmul_rn(sa_next, sb_next);
          if constexpr (C::EPI_COLS == 32) {
            uint32_t v[32];
            tmem_ld_32cols(acc_col, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i += 2) fma2_rn(sums[i], sums[i + 1], v[i], v[i + 1], scale);
          } else {
#pragma unroll
            for (int g = 0; g < C::EPI_COLS / 16; ++g) {
              uint32_t v[16];
              tmem_ld_16cols(acc_col + 16 * g, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; i += 2)
                fma2_rn(sums[16 * g + i], sums[16 * g + i + 1], v[i], v[i + 1], scale);
            }
          }
          release(a);
          if (c + 1 < p.num_chunks) {  // next K-block's scales, issued after the release
            sa_next = row_ok ? __ldg(p.sa + static_cast<size_t>(m) * p.scale_kb + c + 1) : 0.f;
            sb_next = col_in ? __ldg(p.sb + static_cast<size_t>(n_tile >> 7) * p.scale_kb + c + 1) : 0.f;
          }
          if (last) {
            emit(EmitTag<false, 0>{}, n_tile, sums);
            if constexpr (C::EPI_COLS == 64) emit(EmitTag<false, 32>{}, n_tile + 32, sums);
          }
        } else if constexpr (C::REG_SUMS) {
          // drain the chunk into the register sums, free the accumulator, and
          // after the last chunk run the epilogue from the registers
#pragma unroll
          for (int g = 0; g < C::EPI_COLS / 16; ++g) {
            uint32_t v[16];
            tmem_ld_16cols(acc_col + 16 * g, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              // chunk result: an exact integer below 2^24 in magnitude
              const uint32_t x = static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[i])));
              sums[16 * g + i] = c == 0 ? x : sums[16 * g + i] + x;
            }
          }
          release(a);
          if (last) {
            emit(EmitTag<true, 0>{}, n_tile, sums);
            emit(EmitTag<true, 32>{}, n_tile + 32, sums);
          }
        } else {
          // With one accumulator the final chunk's totals go back to the TMEM
          // sum region first, so the accumulator is released before the slow
          // part (scaling, rounding, stores) and the next tile's MMAs start.
          const bool early_release = C::INT_CHUNKS && C::ACC_BUFS == 1 && last;
#pragma unroll 1
          for (int g = 0; g < C::EPI_COLS / 32; ++g) {
            const int n0 = n_tile + 32 * g;
            uint32_t v[32];
            tmem_ld_32cols(acc_col + 32 * g, v);
            tmem_wait_ld();
            if constexpr (C::INT_CHUNKS) {
              // chunk result: an exact integer below 2^24 in magnitude
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[i])));
              const uint32_t sum_col = lane_base + static_cast<uint32_t>(C::COL_SUM + col_part + 32 * g);
              if (c > 0) {
                uint32_t sv[32];
                tmem_ld_32cols(sum_col, sv);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] += sv[i];
              }
              if (!last || early_release) {
                tmem_st_32cols(sum_col, v);
              } else {
                emit(EmitTag<true, 0>{}, n0, v);
              }
            } else {
              emit(EmitTag<false, 0>{}, n0, v);
            }
          }
          if constexpr (C::INT_CHUNKS) tmem_wait_st();
          release(a);
          if (early_release) {
#pragma unroll 1
            for (int g = 0; g < C::EPI_COLS / 32; ++g) {
              const int n0 = n_tile + 32 * g;
              uint32_t v[32];
              tmem_ld_32cols(lane_base + static_cast<uint32_t>(C::COL_SUM + col_part + 32 * g), v);
              tmem_wait_ld();
              emit(EmitTag<true, 0>{}, n0, v);
            }
          }
        }
        ++acc_iter;
      }
    }
    if (C::STORE_TMA && lane == 0) bulk_wait_group_all();  // stores finished reading shared memory
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if constexpr (C::CTAS > 1) cluster_sync();  // the cluster finishes together (peers signal our barriers)
  tc_fence_after_sync();
  if (warp == 1) {
    if constexpr (C::PAIR) {
      tmem_dealloc_pair(tmem, C::TMEM_COLS);
    } else {
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
  }
}

}  // namespace qk
