// qk_fewrow_scales.cuh -- scale staging of the few-row kernels' block-scaled
// modes (qk_skinny_kernel.cuh, qk_streamk_kernel.cuh).
//
// Modes: 1 MXFP8 (E4M3, one UE8M0 byte per 32 K), 2 MXFP4 (packed E2M1, one
// UE8M0 byte per 32 K), 3 NVFP4 (packed E2M1, one UE4M3 byte per 16 K).  A
// ring stage holds 128 bytes of K per row: 128 K (MXFP8) or 256 K (FP4), so a
// row needs SW = 1, 2 or 4 four-byte scale words per stage (ROCm/mori PR #806
// "What" for the raw [rows, K/32] bytes; ROCm/aiter PR #6262 for NVFP4's
// [rows, K/16] UE4M3 bytes).
//
// The few-row kernels compute the product transposed: 128 weight rows are
// the MMA's M operand and the activation rows its N operand, so the weight's
// scales are the MMA's "A" scales and the activations' its "B" scales.  Per
// ring stage the scale warps write 2 * SW 512-byte atoms into shared memory
// -- the weight's SW atoms (128 rows each) first, then the activations' SW
// atoms (up to 128 rows) -- in the order tcgen05.cp 32x128b.warpx4 reads:
// row r's word at byte 16 (r % 32) + 4 (r / 32).  Rows and scale columns
// outside the matrices are zero.  Two warps share the work, one operand each
// (part 0 the weight, part 1 the activations): each writes its SW atoms,
// copies them into the stage's TMEM columns (weight word w at column 4w,
// activation word w at 4 SW + 4w) and commits the copies to the stage's full
// barrier, beside the TMA bytes, so the MMA thread issues nothing but MMAs
// (a copy takes about 100 cycles to issue; NVFP4's eight per stage on one
// thread set the pace of the few-row kernels).
#pragma once

#include "qk_device.cuh"
#include "qk_gemm_kernel.cuh"

namespace qk {

template <int MODE>
struct FewRowMx {
  static_assert(MODE >= 1 && MODE <= 3, "block-scaled modes");
  static constexpr int SW = MODE == 3 ? 4 : MODE == 2 ? 2 : 1;  // scale words per row per stage
  static constexpr int SF_BYTES = 2 * SW * 512;                 // shared memory per stage
  static constexpr int SF_COLS = 8 * SW;                        // TMEM columns per stage
};

// Four consecutive scale bytes of one row, little-endian; zero outside the
// matrix (the matching operand elements are zero-filled by TMA).
__device__ __forceinline__ uint32_t load_sf4(const uint8_t* s, int row, int rows, int col, int cols) {
  if (row >= rows || col >= cols) return 0u;
  const uint8_t* rp = s + static_cast<size_t>(row) * static_cast<size_t>(cols);
  if ((cols & 3) == 0) return __ldg(reinterpret_cast<const uint32_t*>(rp + col));
  uint32_t v = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (col + i < cols) v |= static_cast<uint32_t>(__ldg(rp + col + i)) << (8 * i);
  return v;
}

// Moves one operand's SW atoms of a stage (already in shared memory and
// fenced for the async proxy) into its TMEM columns and commits the copies
// to the stage's full barrier.  One thread.
template <int SW>
__device__ __forceinline__ void fewrow_scales_to_tmem(uint32_t sf_smem, uint32_t sf_tmem, uint64_t* full_bar) {
#pragma unroll
  for (int w = 0; w < SW; ++w)
    tmem_cp_32x128b_warpx4(sf_tmem + static_cast<uint32_t>(4 * w),
                           make_smem_desc(sf_smem + static_cast<uint32_t>(512 * w), 128, 128, 0));
  umma_commit(full_bar);
}

// Runs on one whole warp, for one operand: part 0 the weight (sfw, rows
// w_row0 .. w_row0+127 of N), part 1 the activations (sfa, rows 0..127 of M).
// unit(i, w_row0, col) gives the i-th unit's first weight row and its first
// scale column (4 * SW x its K-block).  sf_tmem: TMEM address of stage 0's
// scale columns (stage s at + 8 SW s).  Returns false when a bounded wait
// gave up (the error is recorded by mbar_wait).
template <int STAGES, int SW, class UnitFn>
__device__ __forceinline__ bool fewrow_stage_scales(const uint8_t* sfw, const uint8_t* sfa, int N, int M,
                                                    int sf_cols, uint8_t* sf_smem, uint32_t sf_tmem, uint64_t* full,
                                                    uint64_t* empty, long long count, UnitFn unit, int lane,
                                                    const WaitCtl& w, int part) {
  constexpr int SF_BYTES = 2 * SW * 512;
  const uint8_t* src = part == 0 ? sfw : sfa;
  const int rows = part == 0 ? N : M;
  const uint32_t atom0 = static_cast<uint32_t>(512 * SW * part);  // this operand's atoms within a stage
  bool ok = true;
  auto publish = [&](int stage) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0)
      fewrow_scales_to_tmem<SW>(smem_u32(sf_smem + stage * SF_BYTES) + atom0,
                                sf_tmem + static_cast<uint32_t>(8 * SW * stage + 4 * SW * part), &full[stage]);
    __syncwarp();
  };
  if (sf_cols % (4 * SW) == 0) {
    // every unit's words lie inside the rows: 4-byte cp.async straight into
    // the atoms, DA (up to 4) units in flight, one commit group per unit,
    // waited for before the proxy fence and the copies.
    constexpr int DA = STAGES > 4 ? 4 : STAGES - 1;
    static_assert(DA >= 1 && DA < STAGES, "a slot is reissued only after the MMA has read it");
    int is = 0, as = 0;  // slots of the next unit to issue / to publish
    uint32_t iph = 0;
    long long next = 0;
    auto issue_next = [&]() {
      if (next < count) {
        // the slot's atoms and TMEM columns have been read by its previous MMAs
        if (!mbar_wait(&empty[is], iph ^ 1u, w, kSiteScaleEmpty)) {
          ok = false;
          return;
        }
        int w_row0, col;
        unit(next, w_row0, col);
        const int row0 = part == 0 ? w_row0 : 0;
        const uint32_t sf = smem_u32(sf_smem + is * SF_BYTES) + atom0;
#pragma unroll
        for (int ww = 0; ww < SW; ++ww) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = row0 + 32 * j + lane;
            const bool in = r < rows;
            cp_async_4(sf + 512 * ww + 16 * lane + 4 * j,
                       in ? src + static_cast<size_t>(r) * static_cast<size_t>(sf_cols) + col + 4 * ww : src,
                       in ? 4u : 0u);
          }
        }
        ++next;
        if (++is == STAGES) {
          is = 0;
          iph ^= 1u;
        }
      }
      cp_async_commit();  // possibly empty: one group per unit index
    };
#pragma unroll 1
    for (int d = 0; ok && d < DA; ++d) issue_next();
#pragma unroll 1
    for (long long i = 0; ok && i < count; ++i) {
      cp_async_wait_group<DA - 1>();  // unit i's group has landed
      publish(as);
      if (++as == STAGES) as = 0;
      issue_next();
    }
    cp_async_wait_group<0>();
    __syncwarp();
  } else {
    // scale columns end inside a unit: loads into registers (zero past the
    // row's end), D units ahead of the stores.
    constexpr int D = 3;
    uint32_t vw[D][SW][4];
    auto load_unit = [&](long long i, uint32_t (&w4)[SW][4]) {
      if (i >= count) return;
      int w_row0, col;
      unit(i, w_row0, col);
      const int row0 = part == 0 ? w_row0 : 0;
#pragma unroll
      for (int ww = 0; ww < SW; ++ww) {
#pragma unroll
        for (int j = 0; j < 4; ++j) w4[ww][j] = load_sf4(src, row0 + 32 * j + lane, rows, col + 4 * ww, sf_cols);
      }
    };
#pragma unroll
    for (int d = 0; d < D; ++d) load_unit(d, vw[d]);
    int stage = 0;
    uint32_t phase = 0;
#pragma unroll 1
    for (long long i = 0; ok && i < count; i += D) {
#pragma unroll
      for (int d = 0; d < D; ++d) {
        if (!ok || i + d >= count) break;
        if (!mbar_wait(&empty[stage], phase ^ 1u, w, kSiteScaleEmpty)) {
          ok = false;
          break;
        }
        const uint32_t sf = smem_u32(sf_smem + stage * SF_BYTES) + atom0;
#pragma unroll
        for (int ww = 0; ww < SW; ++ww)
          st_shared_v4(sf + 512 * ww + 16 * lane, vw[d][ww][0], vw[d][ww][1], vw[d][ww][2], vw[d][ww][3]);
        publish(stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        load_unit(i + d + D, vw[d]);
      }
    }
  }
  // leave no copy in flight: the last unit's full barrier completes only
  // after its copies (bounded wait; the MMA thread waits for it as well)
  if (count > 0 && lane == 0) {
    const long long L = count - 1;
    const uint32_t a = smem_u32(&full[static_cast<int>(L % STAGES)]);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(a, static_cast<uint32_t>((L / STAGES) & 1))) {
      if (global_timer_ns() - t0 > w.timeout_ns) {
        report_error(w.err, kDevErrTimeout, kSiteScaleCopy, static_cast<uint32_t>(L));
        break;
      }
    }
  }
  __syncwarp();
  return ok;
}

// The MMAs of one unit, its scales already in the stage's TMEM columns
// (weight words at sf_tmem + 4w, activation words at sf_tmem + 4 SW + 4w).
//   MXFP8: four MMAs of K = 32 (kind::mxf8f6f4, scale_vec::1X), byte j of word 0.
//   MXFP4: four MMAs of K = 64 (kind::mxf4, scale_vec::2X), bytes 2(j%2) and
//          2(j%2)+1 of word j/2.
//   NVFP4: four MMAs of K = 64 (kind::mxf4nvf4, scale_vec::4X, UE4M3), word j.
template <int MODE>
__device__ __forceinline__ void fewrow_mx_mmas(uint32_t d_tmem, uint64_t wdesc, uint64_t adesc, uint32_t sf_tmem,
                                               int ksteps, bool accumulate, int nt, int mt) {
  constexpr int SW = FewRowMx<MODE>::SW;
  const uint32_t sfb = sf_tmem + static_cast<uint32_t>(4 * SW);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (j < ksteps) {
      const uint64_t wd = wdesc + static_cast<uint64_t>(2 * j);  // 32 bytes of K per MMA
      const uint64_t ad = adesc + static_cast<uint64_t>(2 * j);
      const uint32_t acc = (accumulate || j > 0) ? 1u : 0u;
      if constexpr (MODE == 1) {
        umma_mxf8f6f4(d_tmem, wd, ad,
                      make_idesc_block_scaled(0, 0, nt, mt, static_cast<uint32_t>(j), static_cast<uint32_t>(j)),
                      sf_tmem, sfb, acc);
      } else if constexpr (MODE == 2) {
        const uint32_t g = static_cast<uint32_t>(j >> 1);
        const uint32_t id = static_cast<uint32_t>((j & 1) * 2);
        umma_mxf4(d_tmem, wd, ad, make_idesc_block_scaled(1, 1, nt, mt, id, id), sf_tmem + 4 * g, sfb + 4 * g, acc);
      } else {
        umma_nvf4(d_tmem, wd, ad, make_idesc_block_scaled(1, 1, nt, mt, 0, 0, false), sf_tmem + 4 * j, sfb + 4 * j,
                  acc);
      }
    }
  }
}

}  // namespace qk
