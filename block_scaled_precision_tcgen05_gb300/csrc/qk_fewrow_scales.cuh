// qk_fewrow_scales.cuh -- UE8M0 scale staging for the few-row kernels'
// MXFP8 mode (qk_skinny_kernel.cuh, qk_streamk_kernel.cuh).
//
// The few-row kernels compute the product transposed: 128 weight rows are
// the MMA's M operand and the activation rows its N operand, so the weight's
// scales are the MMA's "A" scales and the activations' its "B" scales.  A
// unit is one 128-K step of one weight tile; it needs four scale bytes per
// row (one per MMA of K = 32).  Per ring stage the scale warp writes two
// 512-byte atoms into shared memory -- the weight's 128 rows at +0 and up to
// 128 activation rows at +512 -- in the order tcgen05.cp 32x128b.warpx4
// reads: row r's word at byte 16 (r % 32) + 4 (r / 32).  Rows outside the
// matrices are zero.  The stage's full barrier counts the warp's arrive
// beside the TMA bytes.
#pragma once

#include "qk_device.cuh"
#include "qk_gemm_kernel.cuh"

namespace qk {

constexpr int kFewRowSfBytes = 1024;  // shared memory per stage: two atoms

// Four consecutive UE8M0 bytes of one scale row, little-endian; zero outside
// the matrix (the matching operand elements are zero-filled by TMA).
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

// Runs on one whole warp.  unit(i, w_row0, col) gives the i-th unit's first
// weight row and its scale column (4 x its K-block).  Returns false when a
// bounded wait gave up (the error is recorded by mbar_wait).
template <int STAGES, class UnitFn>
__device__ __forceinline__ bool fewrow_stage_scales(const uint8_t* sfw, const uint8_t* sfa, int N, int M,
                                                    int sf_cols, uint8_t* sf_smem, uint64_t* full, uint64_t* empty,
                                                    long long count, UnitFn unit, int lane, const WaitCtl& w) {
  bool ok = true;
  if (sf_cols % 4 == 0) {
    // K % 128 == 0: 4-byte cp.async straight into the atoms, DA (up to 4)
    // units in flight, one commit group per unit, waited for before the proxy fence
    // and the arrive.
    constexpr int DA = STAGES > 4 ? 4 : STAGES - 1;
    static_assert(DA >= 1 && DA < STAGES, "a slot is reissued only after the MMA has read it");
    int is = 0, as = 0;  // slots of the next unit to issue / to publish
    uint32_t iph = 0;
    long long next = 0;
    auto issue_next = [&]() {
      if (next < count) {
        if (!mbar_wait(&empty[is], iph ^ 1u, w, kSiteScaleEmpty)) {
          ok = false;
          return;
        }
        int w_row0, col;
        unit(next, w_row0, col);
        const uint32_t sf = smem_u32(sf_smem + is * kFewRowSfBytes);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = w_row0 + 32 * j + lane;
          const bool in = r < N;
          cp_async_4(sf + 16 * lane + 4 * j,
                     in ? sfw + static_cast<size_t>(r) * static_cast<size_t>(sf_cols) + col : sfw, in ? 4u : 0u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 32 * j + lane;
          const bool in = r < M;
          cp_async_4(sf + 512 + 16 * lane + 4 * j,
                     in ? sfa + static_cast<size_t>(r) * static_cast<size_t>(sf_cols) + col : sfa, in ? 4u : 0u);
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
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[as]);
      if (++as == STAGES) as = 0;
      issue_next();
    }
    cp_async_wait_group<0>();
    __syncwarp();
    return ok;
  }
  // K / 32 not a multiple of 4: byte-wise loads into registers, D units
  // ahead of the stores.
  constexpr int D = 3;
  uint32_t vw[D][4], va[D][4];
  auto load_unit = [&](long long i, uint32_t (&w4)[4], uint32_t (&a4)[4]) {
    if (i >= count) return;
    int w_row0, col;
    unit(i, w_row0, col);
#pragma unroll
    for (int j = 0; j < 4; ++j) w4[j] = load_sf4(sfw, w_row0 + 32 * j + lane, N, col, sf_cols);
#pragma unroll
    for (int j = 0; j < 4; ++j) a4[j] = load_sf4(sfa, 32 * j + lane, M, col, sf_cols);
  };
#pragma unroll
  for (int d = 0; d < D; ++d) load_unit(d, vw[d], va[d]);
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
      const uint32_t sf = smem_u32(sf_smem + stage * kFewRowSfBytes);
      st_shared_v4(sf + 16 * lane, vw[d][0], vw[d][1], vw[d][2], vw[d][3]);
      st_shared_v4(sf + 512 + 16 * lane, va[d][0], va[d][1], va[d][2], va[d][3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[stage]);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
      load_unit(i + d + D, vw[d], va[d]);
    }
  }
  return ok;
}

// The MMA side of one unit: both atoms of the stage into its 8 TMEM columns
// (weight at +0, activations at +4), then the unit's block-scaled MMAs of
// K = 32 (kind::mxf8f6f4, scale_vec::1X), scale byte j for the j-th.
__device__ __forceinline__ void fewrow_mx_mmas(uint32_t d_tmem, uint64_t wdesc, uint64_t adesc, uint32_t sf_tmem,
                                               uint32_t sf_smem_addr, int ksteps, bool accumulate, int nt, int mt) {
  tmem_cp_32x128b_warpx4(sf_tmem, make_smem_desc(sf_smem_addr, 128, 128, 0));
  tmem_cp_32x128b_warpx4(sf_tmem + 4, make_smem_desc(sf_smem_addr + 512, 128, 128, 0));
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < ksteps)
      umma_mxf8f6f4(d_tmem, wdesc + static_cast<uint64_t>(2 * j), adesc + static_cast<uint64_t>(2 * j),
                    make_idesc_block_scaled(0, 0, nt, mt, static_cast<uint32_t>(j), static_cast<uint32_t>(j)),
                    sf_tmem, sf_tmem + 4, (accumulate || j > 0) ? 1u : 0u);
}

}  // namespace qk
