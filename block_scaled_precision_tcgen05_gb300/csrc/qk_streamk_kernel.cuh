// qk_streamk_kernel.cuh -- FP8 per-token x per-channel GEMM for few rows
// (M <= 128), where streaming the weight from HBM sets the time.
//
// The product is computed transposed, D^T[n, m] = sum_k B[n,k] A[m,k]: a tile
// of 128 weight rows is the MMA's M operand (TMEM lanes = n) and the M
// activation rows, padded to MT, are its N operand (TMEM columns = m).
//
// Work is balanced by stream-K: the (tile, K-block) units of the whole
// problem, tile-major, are cut into one contiguous range per CTA, one CTA per
// SM, so every SM streams the same number of weight bytes whatever the tile
// count.  A CTA's range splits into segments, one per tile it touches; each
// segment accumulates in one of two TMEM accumulators, so the epilogue of
// one segment overlaps the MMAs of the next.
//  * A segment that covers a whole tile is finished in place.
//  * A segment that does not start at K-block 0 can only be the CTA's first;
//    its fp32 partial goes to a workspace slot of that CTA.  Each epilogue
//    warp writes its 32 weight rows (bulk tensor stores from shared memory),
//    waits for those writes to complete and then releases its own flag with
//    this call's epoch, so no barrier across warps is needed.
//  * The segment holding K-block 0 owns the tile: each epilogue warp waits
//    (bounded) for the matching warp flags of the CTAs that carry the rest of
//    the tile, adds their partials in CTA order (a fixed order, so results
//    are reproducible) and runs the epilogue (x*sa[m])*sb[n] (+bias[n]) ->
//    bf16.
// Every epilogue warp stages what it writes (a partial's 32 x 32 fp32 blocks,
// the output's 32-column blocks of up to 64 rows) in 4 KB of shared memory
// and writes it with a bulk tensor store: per-thread stores of one element
// per row took microseconds at the end of the kernel.
// A contributor's segment is the first thing it computes and never waits on
// another CTA, so the waits cannot form a cycle; the launch is cooperative,
// which guarantees that all CTAs are resident at once.  Once an owner has
// added a contributor's partial it sets that flag back to 0, so a call that
// completes leaves every flag at 0: a replay of a captured graph, which reuses
// the call's epoch, cannot mistake the previous replay's flags for its own.
// The kernel lets the next kernel of the stream launch at once (programmatic
// dependent launch) and waits for the previous one after its prologue, before
// its first global-memory access.  (An L2 prefetch of the first weight tiles
// before that wait measured slower: the cooperative launch starts no CTA
// before the previous kernel's CTAs have all left, so it only lengthened the
// prologue.)
//
// Block-scaled modes (MODE_ 1 MXFP8, 2 MXFP4, 3 NVFP4): the MMAs are
// block-scaled; two scale warps stage each unit's scale atoms and copy them
// into the stage's TMEM columns (qk_fewrow_scales.cuh), and the epilogue is
// bf16(acc (+bias)), NVFP4 bf16(acc * (ga * gb) (+bias)), with no per-row
// scales.  A unit is 128 bytes of K per row in every mode.
#pragma once

#include <cuda_bf16.h>

#include "qk_device.cuh"
#include "qk_fewrow_scales.cuh"
#include "qk_gemm_kernel.cuh"

namespace qk {

struct StreamKParams {
  int M, N, K;
  int num_kb;                 // K-blocks of 128 elements
  long long units;            // n_tiles * num_kb
  const float* sa;
  const float* sb;
  const uint8_t* sfa;         // MXFP8: activation UE8M0 scales [M, sf_cols]
  const uint8_t* sfw;         // MXFP8: weight UE8M0 scales [N, sf_cols]
  int sf_cols;                // K / 32
  const float* ga;            // NVFP4 per-tensor scales (nullable: 1)
  const float* gb;
  const uint16_t* bias;
  uint16_t* out;
  float* partials;            // [gridDim.x][MT][128] fp32
  unsigned long long* flags;  // [gridDim.x][4]: one per epilogue warp
  unsigned long long epoch;   // unique per call; a flag equal to it marks a finished partial
  unsigned long long* err;
  uint64_t timeout_ns;
};

// MODE_: 0 FP8 per-token x per-channel, 1 MXFP8, 2 MXFP4, 3 NVFP4.
template <int MT_, int STAGES_, int MODE_ = 0>
struct StreamKCfg {
  static constexpr int MODE = MODE_;
  static constexpr bool MX = MODE_ != 0;  // block-scaled MMAs
  static constexpr bool FP4 = MODE_ >= 2;
  static constexpr int MT = MT_;          // padded activation rows (MMA N)
  static constexpr int NT = 128;          // weight rows per tile (MMA M)
  static constexpr int STAGES = STAGES_;
  static constexpr int KB_BYTES = 128;             // bytes of K per row per stage (one 128-byte swizzle row)
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
  // per epilogue warp 4 KB: fp32 [32 rows][32 cols] or bf16 [OUT_ROWS][32 cols]
  static constexpr int STG_BYTES = 4096;
  static constexpr int OUT_ROWS = MT < 64 ? MT : 64;  // output rows per bulk store
  static constexpr int OFF_STG = (OFF_SF + STAGES * SF_BYTES + 1023) & ~1023;
  static constexpr int OFF_BAR = OFF_STG + 4 * STG_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * 2 + 1;  // ring, accumulators, drain
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_SA = OFF_MISC + 16;  // FP8: the MT per-token scales (fp32)
  static constexpr int SMEM_BYTES = OFF_SA + MT * 4 + 1024;
  static constexpr int COL_SF = 2 * MT;        // after the two accumulators
  static constexpr int COLS_USED = COL_SF + STAGES * SF_COLS_STAGE;
  static constexpr int TMEM_COLS = COLS_USED <= 64 ? 64 : COLS_USED <= 128 ? 128 : COLS_USED <= 256 ? 256 : 512;
  static constexpr int NUM_THREADS = 256;   // warp 0 TMA, warp 1 MMA, warps 2-3 scales, 4..7 epilogue
  static_assert(MT == 32 || MT == 64 || MT == 128, "activation tile");
  static_assert(A_BYTES % 1024 == 0, "swizzle atoms need 1024-byte alignment");
  static_assert(SMEM_BYTES <= 232448, "shared-memory budget");
  static constexpr uint32_t IDESC = make_idesc_dense(1, 0, 0, NT, MT);  // fp32 D, E4M3 x E4M3
  static_assert(COLS_USED <= 512, "TMEM budget");
};

// First unit of CTA c's range (units * c / G, rounded down).
__device__ __forceinline__ long long streamk_begin(long long units, int c, int G) {
  return units * static_cast<long long>(c) / static_cast<long long>(G);
}

__device__ __forceinline__ void st_release_gpu_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

template <class C>
__global__ void __launch_bounds__(C::NUM_THREADS, 1)
    qk_streamk_fp8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmPart,
                          const StreamKParams p) {
  extern __shared__ uint8_t smem_raw[];
  griddep_launch_dependents();
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = static_cast<int>(blockIdx.x);
  const int G = static_cast<int>(gridDim.x);
  const long long u0 = streamk_begin(p.units, c, G);
  const long long u1 = streamk_begin(p.units, c + 1, G);

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], C::MX ? 3u : 1u);  // the TMA bytes (+ the two scale warps' copies)
      mbar_init(&empty[s], 1u);
    }
#pragma unroll 1
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1u);
      mbar_init(&acc_empty[a], 4u);  // the four epilogue warps
    }
    mbar_init(drain, 1u);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmOut);
    tma_prefetch_desc(&tmPart);
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
    // ---------------- TMA producer: one stage per unit of the range ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
#pragma unroll 1
      for (long long u = u0; u < u1; ++u) {
        const int t = static_cast<int>(u / p.num_kb);
        const int kb = static_cast<int>(u - static_cast<long long>(t) * p.num_kb);
        if (!mbar_wait(&empty[stage], phase ^ 1u, w, kSiteProducerEmpty)) break;
        mbar_arrive_expect_tx(&full[stage], C::STAGE_TX);
        tma_load_2d(smem + C::OFF_W + stage * C::W_BYTES, &tmW, &full[stage], kb * C::KB_BYTES, t * C::NT);
        tma_load_2d(smem + C::OFF_A + stage * C::A_BYTES, &tmA, &full[stage], kb * C::KB_BYTES, 0);
        ++issued;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // wait (bounded) for the last load of every ring slot before leaving
      const long long n = issued < C::STAGES ? issued : C::STAGES;
#pragma unroll 1
      for (long long i = 0; i < n; ++i) {
        const long long L = issued - 1 - i;
        const uint32_t a = smem_u32(&full[static_cast<int>(L % C::STAGES)]);
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
    // ---------------- MMA issuer: one accumulator per segment ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t seg = 0;
      bool ok = true;
#pragma unroll 1
      for (long long u = u0; ok && u < u1;) {
        const int t = static_cast<int>(u / p.num_kb);
        const int kb0 = static_cast<int>(u - static_cast<long long>(t) * p.num_kb);
        const int n_seg = static_cast<int>(min(static_cast<long long>(p.num_kb - kb0), u1 - u));
        const int a = static_cast<int>(seg & 1u);
        if (!mbar_wait(&acc_empty[a], ((seg >> 1) & 1u) ^ 1u, w, kSiteMmaAccEmpty)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(a * C::MT);
#pragma unroll 1
        for (int i = 0; i < n_seg; ++i) {
          const int kb = kb0 + i;
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
            fewrow_mx_mmas<C::MODE>(d_tmem, wdesc, adesc,
                                    tmem + static_cast<uint32_t>(C::COL_SF + C::SF_COLS_STAGE * stage), ksteps, i > 0,
                                    C::NT, C::MT);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (j < ksteps)
                umma_f8f6f4(d_tmem, wdesc + static_cast<uint64_t>(2 * j), adesc + static_cast<uint64_t>(2 * j),
                            C::IDESC, (i > 0 || j > 0) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&acc_full[a]);
        ++seg;
        u += n_seg;
      }
      // every MMA issued here completes before TMEM is freed
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
    // ---------------- scale warps (block-scaled modes): one operand's atoms each per unit ----------------
    if constexpr (C::MX) {
      constexpr int SW = FewRowMx<C::MODE>::SW;
      auto unit = [&](long long i, int& w_row0, int& col) {
        const long long v = u0 + i;
        const int tv = static_cast<int>(v / p.num_kb);
        w_row0 = tv * C::NT;
        col = static_cast<int>(v - static_cast<long long>(tv) * p.num_kb) * 4 * SW;
      };
      fewrow_stage_scales<C::STAGES, SW>(p.sfw, p.sfa, p.N, p.M, p.sf_cols, smem + C::OFF_SF,
                                         tmem + static_cast<uint32_t>(C::COL_SF), full, empty, u1 - u0, unit, lane, w, warp - 2);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- epilogue: thread r holds weight row r of the tile ----------------
    const int q = warp - 4;
    const int r = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t stg = smem_u32(smem + C::OFF_STG + q * C::STG_BYTES);
    // the staging block may be rewritten once the previous bulk store has read it
    auto stg_acquire = [&]() {
      if (lane == 0) bulk_wait_group_read<0>();
      __syncwarp();
    };
    auto stg_store = [&](const CUtensorMap* map, int x, int y) {
      fence_proxy_async_smem();  // the block's generic writes before the bulk copy reads it
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(map, stg, x, y);
        bulk_commit_group();
      }
    };
    // NVFP4: the product of the per-tensor scales, one fp32 rounding
    [[maybe_unused]] float alpha = 1.f;
    if constexpr (C::MODE == 3) alpha = __fmul_rn(p.ga ? __ldg(p.ga) : 1.f, p.gb ? __ldg(p.gb) : 1.f);
    // FP8: the per-token scales once, into shared memory, while the first units stream
    float* sa_s = reinterpret_cast<float*>(smem + C::OFF_SA);
    if constexpr (!C::MX) {
      if (r < C::MT) sa_s[r] = r < p.M ? __ldg(p.sa + r) : 0.f;
      named_barrier_sync(1, 128);  // the four epilogue warps
    }
    // With at most 64 rows, the head of a shared tile waits for its
    // contributors' flags and loads the first partial before its own
    // accumulator (the registers do not hold two 128-row partials).
    constexpr bool kEarlyPartial = C::MT <= 64;
    uint32_t seg = 0;
#pragma unroll 1
    for (long long u = u0; u < u1;) {
      const int t = static_cast<int>(u / p.num_kb);
      const int kb0 = static_cast<int>(u - static_cast<long long>(t) * p.num_kb);
      const int n_seg = static_cast<int>(min(static_cast<long long>(p.num_kb - kb0), u1 - u));
      const int a = static_cast<int>(seg & 1u);
      const int n = t * C::NT + r;
      // this row's column scale and bias, requested before the accumulator
      float sbn = 1.f, bn = 0.f;
      if (n < p.N) {
        if constexpr (!C::MX) sbn = __ldg(p.sb + n);
        if (p.bias) bn = __uint_as_float(static_cast<uint32_t>(__ldg(p.bias + n)) << 16);
      }
      const bool head_of_shared = kb0 == 0 && kb0 + n_seg != p.num_kb;
      int jend = c + 1;
      bool peers_ok = true;
      float pv[C::MT];
      // the contributors are CTAs c+1 .. jend-1: wait for all their flags at
      // once (one per lane); contributors publish their first segment and
      // never wait, so the wait ends
      auto wait_peers = [&]() {
        const long long tile_end = static_cast<long long>(t + 1) * p.num_kb;
        while (jend < G && streamk_begin(p.units, jend, G) < tile_end) ++jend;
#pragma unroll 1
        for (int base = c + 1; peers_ok && base < jend; base += 32) {
          const int j = base + lane;
          int seen = 1;
          if (j < jend) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_gpu_u64(p.flags + 4 * j + q) != p.epoch) {
              if (*abort_flag) {
                seen = 0;
                break;
              }
              if (global_timer_ns() - t0 > p.timeout_ns) {
                report_error(p.err, kDevErrTimeout, kSitePeerPartial, static_cast<uint32_t>(j));
                *abort_flag = 1u;
                seen = 0;
                break;
              }
            }
          }
          // each lane's acquire, then the warp barrier, orders every lane's loads after it
          peers_ok = __all_sync(0xffffffffu, seen != 0);
        }
        __syncwarp();
      };
      auto load_partial = [&](int j) {
        const float* src = p.partials + static_cast<size_t>(j) * C::MT * C::NT;
        // all the partial's loads in flight before the adds
#pragma unroll
        for (int m = 0; m < C::MT; ++m) pv[m] = m < p.M ? __ldcg(src + m * C::NT + r) : 0.f;
      };
      if (kEarlyPartial && head_of_shared) {
        wait_peers();
        if (peers_ok) load_partial(c + 1);
      }
      // warp-uniform outcome: the TMEM loads below are warp-collective
      const bool got = mbar_wait(&acc_full[a], (seg >> 1) & 1u, w, kSiteEpiAccFull);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      float acc[C::MT];
#pragma unroll
      for (int g = 0; g < C::MT / 32; ++g) {
        uint32_t v[32];
        tmem_ld_32cols(lane_base + static_cast<uint32_t>(a * C::MT + 32 * g), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[32 * g + i] = __uint_as_float(v[i]);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);

      if (kb0 != 0) {
        // the tail of a tile owned by an earlier CTA: publish the partial
        // (workspace rows c*MT .. c*MT+MT-1, this warp's 32 columns)
#pragma unroll
        for (int h = 0; h < C::MT / 32; ++h) {
          stg_acquire();
#pragma unroll
          for (int i = 0; i < 32; ++i) st_shared_f32(stg + static_cast<uint32_t>((i * 32 + lane) * 4), acc[32 * h + i]);
          stg_store(&tmPart, q * 32, c * C::MT + 32 * h);
        }
        if (lane == 0) {
          bulk_wait_group_all();       // the partial's writes are complete
          fence_proxy_async_global();  // ... and ordered before the flag
          __threadfence();
          st_release_gpu_u64(p.flags + 4 * c + q, p.epoch);
        }
        __syncwarp();
      } else {
        if (head_of_shared) {
          if (!kEarlyPartial) wait_peers();
          if (peers_ok) {
            // add the contributors' partials in CTA order
#pragma unroll 1
            for (int j = c + 1; j < jend; ++j) {
              if (!kEarlyPartial || j > c + 1) load_partial(j);
#pragma unroll
              for (int m = 0; m < C::MT; ++m)
                if (m < p.M) acc[m] = __fadd_rn(acc[m], pv[m]);
            }
            // the partials are read (their values are in the sums): clear their flags
            __syncwarp();
            for (int j = c + 1 + lane; j < jend; j += 32) p.flags[4 * j + q] = 0ull;
          }
        }
        // the output block [rows, this warp's 32 columns] in bulk stores of OUT_ROWS rows
        if (t * C::NT + q * 32 < p.N) {
          // every row's epilogue first (its scale loads batched), then the staging stores
#pragma unroll
          for (int m = 0; m < C::MT; ++m) {
            float x = acc[m];
            if constexpr (!C::MX) {
              x = __fmul_rn(x, sa_s[m]);
              x = __fmul_rn(x, sbn);
            }
            if constexpr (C::MODE == 3) x = __fmul_rn(x, alpha);
            if (p.bias) x = __fadd_rn(x, bn);
            acc[m] = x;
          }
#pragma unroll
          for (int h = 0; h < C::MT / C::OUT_ROWS; ++h) {
            if (h * C::OUT_ROWS < p.M) {
              stg_acquire();
#pragma unroll
              for (int i = 0; i < C::OUT_ROWS; ++i)
                st_shared_u16(stg + static_cast<uint32_t>((i * 32 + lane) * 2),
                              __bfloat16_as_ushort(__float2bfloat16_rn(acc[h * C::OUT_ROWS + i])));
              stg_store(&tmOut, t * C::NT + q * 32, h * C::OUT_ROWS);
            }
          }
        }
      }
      ++seg;
      u += n_seg;
    }
    // no bulk store of this warp still reads shared memory or is in flight
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace qk
