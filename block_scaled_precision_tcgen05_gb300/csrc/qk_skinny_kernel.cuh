// qk_skinny_kernel.cuh -- FP8 per-token x per-channel GEMM for few rows
// (M <= 128): the weight streams through HBM once and sets the time.
//
// The product is computed transposed, D^T[n, m] = sum_k B[n,k] A[m,k]: a
// tile of 128 weight rows is the MMA's M operand (TMEM lanes = n), the M
// activation rows, padded to MT, are its N operand (TMEM columns = m).  K is
// split over a cluster of SPLITS (1..8) CTAs; each CTA accumulates its K range in
// TMEM, stages the fp32 partial in shared memory as [m][n], and after a
// cluster barrier every CTA sums, in fixed order over the cluster, the rows
// m it owns by reading its peers' partials through distributed shared
// memory, then applies the fixed-order epilogue (x*sa[m])*sb[n] (+bias[n])
// and stages its bf16 output rows in shared memory for bulk tensor stores.
//
// Block-scaled modes (MODE_ 1 MXFP8, 2 MXFP4, 3 NVFP4): block-scaled MMAs
// with the scale staging of qk_fewrow_scales.cuh (two scale warps that also
// copy each stage's atoms into 8 SW TMEM columns after the accumulator),
// and the epilogue bf16(x (+bias)), NVFP4: bf16(x * (ga * gb) (+bias)).  A
// stage is 128 bytes of K per row in every mode (128 E4M3 or 256 packed E2M1
// elements).
// The kernel lets the next kernel of the stream launch at once (programmatic
// dependent launch) and waits for the previous one after its prologue, before
// its first global-memory access.  (An L2 prefetch of the CTA's weight slice
// before that wait measured no faster back to back and 2 us slower for one
// call: its requests competed with the loads.)
#pragma once

#include <cuda_bf16.h>

#include "qk_device.cuh"
#include "qk_fewrow_scales.cuh"
#include "qk_gemm_kernel.cuh"

namespace qk {

struct SkinnyParams {
  int M, N, K;
  int num_kb;        // k-blocks of 128 elements
  int kb_per_split;  // k-blocks per CTA of a cluster
  const float* sa;
  const float* sb;
  const uint8_t* sfa;  // MXFP8: activation UE8M0 scales [M, sf_cols]
  const uint8_t* sfw;  // MXFP8: weight UE8M0 scales [N, sf_cols]
  int sf_cols;         // K / 32
  const float* ga;     // NVFP4 per-tensor scales (nullable: 1)
  const float* gb;
  const uint16_t* bias;
  uint16_t* out;
  unsigned long long* err;
  uint64_t timeout_ns;
};

// MODE_: 0 FP8 per-token x per-channel, 1 MXFP8, 2 MXFP4, 3 NVFP4.
template <int MT_, int SPLITS_, int STAGES_, int MODE_ = 0>
struct SkinnyCfg {
  static constexpr int MODE = MODE_;
  static constexpr bool MX = MODE_ != 0;  // block-scaled MMAs
  static constexpr bool FP4 = MODE_ >= 2;
  static constexpr int MT = MT_;          // padded activation rows (MMA N)
  static constexpr int NT = 128;          // weight rows per tile (MMA M)
  static constexpr int SPLITS = SPLITS_;  // CTAs of a cluster splitting K
  static constexpr int STAGES = STAGES_;
  static constexpr int KB_BYTES = 128;          // bytes of K per row per stage (one 128-byte swizzle row)
  static constexpr int K_ELEMS = FP4 ? 256 : 128;  // elements per stage
  static constexpr int UMMA_K = FP4 ? 64 : 32;     // elements per MMA (32 bytes)
  static constexpr int W_BYTES = NT * 128;
  static constexpr int A_BYTES = MT * 128;
  static constexpr uint32_t STAGE_TX = W_BYTES + A_BYTES;
  static constexpr int OFF_W = 0;
  static constexpr int OFF_A = OFF_W + STAGES * W_BYTES;
  static constexpr int SF_BYTES = MX ? FewRowMx<MX ? MODE_ : 1>::SF_BYTES : 0;  // per stage: weight atoms, then activation atoms
  static constexpr int SF_COLS_STAGE = MX ? FewRowMx<MX ? MODE_ : 1>::SF_COLS : 0;
  static constexpr int OFF_SF = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_RED = OFF_SF + STAGES * SF_BYTES;  // fp32 partial [MT][NT]
  static constexpr int RED_BYTES = MT * NT * 4;
  static constexpr int OFF_SA = OFF_RED + RED_BYTES;           // fp32 row scales of this CTA's output rows
  // output rows each CTA reduces (the last CTA's range may run past MT: those
  // rows lie past M, read as zero and are clipped by the output store)
  static constexpr int ROWS_PER_CTA = (MT + SPLITS - 1) / SPLITS;
  // output staging: per epilogue warp [OUT_ROWS][32] bf16, written by bulk tensor stores
  static constexpr int OUT_ROWS = ROWS_PER_CTA < 32 ? ROWS_PER_CTA : 32;
  static constexpr int OFF_STG = OFF_SA + 512;
  static constexpr int STG_BYTES = 32 * 64;
  static constexpr int OFF_BAR = OFF_STG + 4 * STG_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + (2 * STAGES + 2) * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int COL_SF = MT;  // after the accumulator
  static constexpr int COLS_USED = MT + STAGES * SF_COLS_STAGE;
  static constexpr int TMEM_COLS = COLS_USED <= 32 ? 32 : COLS_USED <= 64 ? 64 : COLS_USED <= 128 ? 128 : COLS_USED <= 256 ? 256 : 512;
  static constexpr int NUM_THREADS = 256;
  static_assert(MT % 32 == 0 && MT >= 32 && MT <= 128, "activation tile");
  static_assert(SPLITS >= 1 && SPLITS <= 8, "portable cluster sizes");
  static_assert(SMEM_BYTES <= 232448, "shared-memory budget");
  static constexpr uint32_t IDESC = make_idesc_dense(1, 0, 0, NT, MT);  // fp32 D, E4M3 x E4M3
};

// A load from another CTA's shared memory.  Not volatile: the partials it
// reads are stable between the two cluster barriers, so the compiler may
// issue all of a thread's loads before the first use.
__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t cluster_addr) {
  float v;
  asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr));
  return v;
}

template <class C>
__global__ void __launch_bounds__(C::NUM_THREADS, 1)
    qk_skinny_fp8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmOut, const SkinnyParams p) {
  extern __shared__ uint8_t smem_raw[];
  griddep_launch_dependents();
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* sa_rows = reinterpret_cast<float*>(smem + C::OFF_SA);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = C::SPLITS > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int tile = static_cast<int>(blockIdx.x) / C::SPLITS;
  const int n0 = tile * C::NT;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], C::MX ? 3u : 1u);  // the TMA bytes (+ the two scale warps' copies)
      mbar_init(&empty[s], 1u);
    }
    mbar_init(acc_full, 1u);
    mbar_init(drain, 1u);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{abort_flag, p.err, p.timeout_ns};
  // the previous kernel of the stream has completed and its writes are visible
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
#pragma unroll 1
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, w, kSiteProducerEmpty)) break;
        mbar_arrive_expect_tx(&full[stage], C::STAGE_TX);
        tma_load_2d(smem + C::OFF_W + stage * C::W_BYTES, &tmW, &full[stage], kb * C::KB_BYTES, n0);
        tma_load_2d(smem + C::OFF_A + stage * C::A_BYTES, &tmA, &full[stage], kb * C::KB_BYTES, 0);
        ++issued;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // wait (bounded) for the last load of every ring slot before leaving
#pragma unroll 1
      for (int i = 0; i < (issued < C::STAGES ? issued : C::STAGES); ++i) {
        const int L = issued - 1 - i;
        const uint32_t a = smem_u32(&full[L % C::STAGES]);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(a, static_cast<uint32_t>((L / C::STAGES) & 1))) {
          if (global_timer_ns() - t0 > p.timeout_ns) {
            report_error(p.err, kDevErrTimeout, kSiteProducerDrain, static_cast<uint32_t>(L));
            break;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
#pragma unroll 1
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, w, kSiteMmaFull)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint64_t wdesc = make_desc_kmajor_sw128(smem_u32(smem + C::OFF_W + stage * C::W_BYTES));
        const uint64_t adesc = make_desc_kmajor_sw128(smem_u32(smem + C::OFF_A + stage * C::A_BYTES));
        int ksteps = 4;
        if (kb == p.num_kb - 1) ksteps = min(4, (p.K - kb * C::K_ELEMS + C::UMMA_K - 1) / C::UMMA_K);
        if constexpr (C::MX) {
          fewrow_mx_mmas<C::MODE>(tmem, wdesc, adesc, tmem + static_cast<uint32_t>(C::COL_SF + C::SF_COLS_STAGE * stage),
                                  ksteps, kb > kb0, C::NT, C::MT);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (j < ksteps)
              umma_f8f6f4(tmem, wdesc + static_cast<uint64_t>(2 * j), adesc + static_cast<uint64_t>(2 * j),
                          C::IDESC, (kb > kb0 || j > 0) ? 1u : 0u);
        }
        umma_commit(&empty[stage]);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) umma_commit(acc_full);
      umma_commit(drain);
      const uint32_t da = smem_u32(drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(da, 0u)) {
        if (global_timer_ns() - t0 > p.timeout_ns) {
          report_error(p.err, kDevErrTimeout, kSiteDrain, 0u);
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    if constexpr (C::MX) {
      constexpr int SW = FewRowMx<C::MODE>::SW;
      auto unit = [&](long long i, int& w_row0, int& col) {
        w_row0 = n0;
        col = (kb0 + static_cast<int>(i)) * 4 * SW;
      };
      fewrow_stage_scales<C::STAGES, SW>(p.sfw, p.sfa, p.N, p.M, p.sf_cols, smem + C::OFF_SF,
                                         tmem + static_cast<uint32_t>(C::COL_SF), full, empty,
                                         kb1 > kb0 ? kb1 - kb0 : 0, unit, lane, w, warp - 2);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // while the weight streams: the row scales of the output rows this CTA
    // reduces, so the reduction after the cluster barrier waits on no global load
    if constexpr (!C::MX) {
      const int t = (warp - 4) * 32 + lane;
      if (t < C::ROWS_PER_CTA) {
        const int m = split * C::ROWS_PER_CTA + t;
        sa_rows[t] = m < p.M ? __ldg(p.sa + m) : 0.f;
      }
    }
    // partial D^T (lane = weight row, column = activation row) -> red[m][n]
    const int q = warp - 4;
    const int nr = q * 32 + lane;
    const bool have = kb1 > kb0 && mbar_wait(acc_full, 0u, w, kSiteEpiAccFull);
    tc_fence_after_sync();
#pragma unroll
    for (int g = 0; g < C::MT / 32; ++g) {
      uint32_t v[32];
      if (have) {
        tmem_ld_32cols(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(32 * g), v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;  // empty K range contributes zero
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) red[(32 * g + i) * C::NT + nr] = __uint_as_float(v[i]);
    }
    tc_fence_before_sync();
  }

  // every CTA of the cluster has staged its partial
  __syncthreads();
  if constexpr (C::SPLITS > 1) cluster_sync();

  if (warp >= 4) {
    const int q = warp - 4;
    const int t = q * 32 + lane;  // weight row within the tile
    const int n = n0 + t;
    const bool col_ok = n < p.N;
    const float sbn = (col_ok && !C::MX) ? __ldg(p.sb + n) : 0.f;
    const float bn = (col_ok && p.bias) ? __uint_as_float(static_cast<uint32_t>(__ldg(p.bias + n)) << 16) : 0.f;
    const uint32_t red_base = smem_u32(red);
    const uint32_t stg = smem_u32(smem + C::OFF_STG + q * C::STG_BYTES);
    // NVFP4: the product of the per-tensor scales, one fp32 rounding
    [[maybe_unused]] float alpha = 1.f;
    if constexpr (C::MODE == 3) alpha = __fmul_rn(p.ga ? __ldg(p.ga) : 1.f, p.gb ? __ldg(p.gb) : 1.f);
    const int row0 = split * C::ROWS_PER_CTA;  // first output row of this CTA
    const bool cols_in = n0 + q * 32 < p.N;    // warp-uniform: any of this warp's columns inside N
    // RG rows at a time: all their peers' loads are issued before the first
    // sum (one row at a time, each row waited for its loads in turn; four
    // rows at a time measured 0.5 us slower than sixteen at 64x2112x7168)
    constexpr int RG = C::ROWS_PER_CTA <= 16 ? C::ROWS_PER_CTA
                       : C::ROWS_PER_CTA % 16 == 0 ? 16 : C::ROWS_PER_CTA / 2;
    static_assert(C::ROWS_PER_CTA % RG == 0 && C::OUT_ROWS % RG == 0, "row groups");
#pragma unroll 1
    for (int i0 = 0; i0 < C::ROWS_PER_CTA; i0 += RG) {
      if (row0 + i0 >= p.M) break;
      float part[RG][C::SPLITS];
#pragma unroll
      for (int g = 0; g < RG; ++g) {
        const int m = row0 + i0 + g;
        const uint32_t off = red_base + static_cast<uint32_t>((m * C::NT + t) * 4);
#pragma unroll
        for (int r = 0; r < C::SPLITS; ++r)
          part[g][r] = m >= p.M ? 0.f
                       : C::SPLITS > 1 ? ld_shared_cluster_f32(mapa_shared(off, static_cast<uint32_t>(r)))
                                       : red[m * C::NT + t];
      }
      float vals[RG];
#pragma unroll
      for (int g = 0; g < RG; ++g) {
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < C::SPLITS; ++r) sum = __fadd_rn(sum, part[g][r]);  // fixed order over the cluster
        float x = sum;
        if constexpr (!C::MX) {
          x = __fmul_rn(x, sa_rows[i0 + g]);
          x = __fmul_rn(x, sbn);
        }
        if constexpr (C::MODE == 3) x = __fmul_rn(x, alpha);
        if (p.bias) x = __fadd_rn(x, bn);
        vals[g] = x;
      }
      // stage the rows (rows past M and columns past N are clipped by the store)
      const int srow = i0 % C::OUT_ROWS;
      if (srow == 0) {
        if (lane == 0) bulk_wait_group_read<0>();  // the previous store has read the block
        __syncwarp();
      }
#pragma unroll
      for (int g = 0; g < RG; ++g)
        st_shared_u16(stg + static_cast<uint32_t>(((srow + g) * 32 + lane) * 2), __bfloat16_as_ushort(__float2bfloat16_rn(vals[g])));
      if (srow + RG == C::OUT_ROWS || i0 + RG >= C::ROWS_PER_CTA || row0 + i0 + RG >= p.M) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && cols_in) {
          tma_store_2d(&tmOut, stg, n0 + q * 32, row0 + i0 - srow);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
  }

  // peers may still read this CTA's partial until everyone is past here
  if constexpr (C::SPLITS > 1) cluster_sync();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace qk
