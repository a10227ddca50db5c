// qk_sf_atoms.cuh -- scale factors of the block-scaled kinds, rearranged once
// per call from the caller's raw row-major bytes (ROCm/mori PR #806, "What":
// [rows, K/32] UE8M0 bytes as the quantiser writes them; [N/32, K/32] for B
// in the 32x32-block form; NVFP4: [rows, K/16] UE4M3 bytes) into the order
// the tensor cores read them, and the launch sequence of a block-scaled GEMM.
//
// tcgen05.mma reads the scale of tile row r, for one 32-bit column of four
// consecutive scale blocks along K, from TMEM lane r at column (r / 32) of a
// 4-column group; tcgen05.cp.32x128b.warpx4 fills such a group from a
// 512-byte "atom": 32 lines of 16 bytes, line l holding the four 4-byte words
// of rows l, l + 32, l + 64 and l + 96 (replicated into the four lane
// quarters).  The pre-pass writes, per operand, one atom per (128-row block,
// K-group of four scale bytes): atom (rb, g) at byte ((rb * gpad) + g) * 512,
// K-groups padded with zero bytes to gpad = num_kb * SF_ATOMS_K so that every
// ring stage loads whole atoms, rows past the operand zero as well.  The GEMM
// kernel's producer then loads a stage's atoms by TMA beside the operand
// tiles.  The scale bytes are ~1/32 (MX) or 1/16 (NVFP4) of the operand bytes,
// so the pass costs a few microseconds next to the GEMM.
#pragma once

#include "qk_launch.cuh"

namespace qk {

// One operand's scale bytes and where its atoms go.
struct SfAtomsArgs {
  const uint8_t* src;  // [ceil(rows / rows_per), cols] raw bytes
  uint8_t* dst;        // [ceil(rows / 128), gpad, 512] atoms
  int rows, rows_per, blocks;
  int word_loads;      // 2: 16-byte loads allowed, 1: 4-byte loads, 0: bytes
};

// Both operands in one launch: blocks [0, a.blocks) of x write A's atoms, the
// rest B's.  One block per (128-row block rb, 32 K-groups starting at
// 32 * blockIdx.y): the block reads the 128 rows' 128 scale bytes of those
// K-groups -- eight threads per row, 16 bytes each when the rows allow it
// (zero past a row's `cols` bytes and for rows past `rows`) -- into shared
// memory, then writes the 32 atoms, 16 bytes per line, consecutive threads on
// consecutive lines.  Row r takes source row r / rows_per (32 for B's 32x32
// blocks).  The shared tile's row pitch of 33 words keeps both the row writes
// and the column reads free of bank conflicts.
static __global__ void __launch_bounds__(128) qk_sf_atoms_kernel(SfAtomsArgs a, SfAtomsArgs b, int cols, int gpad) {
  __shared__ uint32_t tile[128][33];
  // the GEMM that reads the atoms may start its prologue now (it waits for
  // this grid before its first load)
  griddep_launch_dependents();
  const bool is_a = static_cast<int>(blockIdx.x) < a.blocks;
  const SfAtomsArgs& o = is_a ? a : b;
  const uint8_t* __restrict__ src = o.src;
  uint8_t* __restrict__ dst = o.dst;
  const int rb = is_a ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) - a.blocks;
  const int g0 = blockIdx.y * 32;
  const int t = threadIdx.x;
  // load: piece i = t + 128 k holds 16 bytes (four words) of tile row i / 8
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = t + 128 * k;
    const int rl = i >> 3, q = i & 7;
    const int r = rb * 128 + rl;
    const int c0 = 4 * g0 + 16 * q;  // first scale byte of the piece
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    if (r < o.rows && c0 < cols) {
      const uint8_t* row = src + static_cast<size_t>(r / o.rows_per) * static_cast<size_t>(cols);
      if (o.word_loads == 2 && c0 + 16 <= cols) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(row + c0));
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
      } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int c = c0 + 4 * w;
          if (o.word_loads >= 1 && c + 4 <= cols) {
            v[w] = __ldg(reinterpret_cast<const uint32_t*>(row + c));
          } else {
#pragma unroll
            for (int bb = 0; bb < 4; ++bb)
              if (c + bb < cols) v[w] |= static_cast<uint32_t>(__ldg(row + c + bb)) << (8 * bb);
          }
        }
      }
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) tile[rl][4 * q + w] = v[w];
  }
  __syncthreads();
  // store: line j = t + 128 k of the block's 32 atoms (atom j / 32, line j % 32)
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int j = t + 128 * k;
    const int w = j >> 5, l = j & 31;
    const int g = g0 + w;
    if (g < gpad) {
      const uint4 line = make_uint4(tile[l][w], tile[l + 32][w], tile[l + 64][w], tile[l + 96][w]);
      *reinterpret_cast<uint4*>(dst + (static_cast<size_t>(rb) * gpad + g) * 512 + 16 * l) = line;
    }
  }
}

// Writes both operands' atom buffers in one launch and encodes their tensor
// maps: [blocks * gpad * 2, 256 bytes], box [256 bytes, 2 * atoms_per_stage rows].
inline int write_sf_atoms(const uint8_t* sA, uint8_t* dA, int M, const uint8_t* sB, uint8_t* dB, int N,
                          int b_rows_per, int cols, int gpad, int atoms_per_stage, CUtensorMap* mapA,
                          CUtensorMap* mapB, cudaStream_t stream) {
  auto args = [&](const uint8_t* src, uint8_t* dst, int rows, int rows_per) {
    SfAtomsArgs o;
    o.src = src;
    o.dst = dst;
    o.rows = rows;
    o.rows_per = rows_per;
    o.blocks = (rows + 127) / 128;
    const uintptr_t base = reinterpret_cast<uintptr_t>(src);
    o.word_loads = (cols % 16 == 0 && (base & 15u) == 0) ? 2 : ((cols % 4 == 0 && (base & 3u) == 0) ? 1 : 0);
    return o;
  };
  const SfAtomsArgs a = args(sA, dA, M, 1), b = args(sB, dB, N, b_rows_per);
  LaunchTimer timer(kKSfAtoms, stream);
  qk_sf_atoms_kernel<<<dim3(a.blocks + b.blocks, (gpad + 31) / 32), 128, 0, stream>>>(a, b, cols, gpad);
  timer.done();
  if (cudaGetLastError() != cudaSuccess) return QK_ERR_CUDA;
  count_launches(1);
  int st = encode_tmap_2d_plain(mapA, CU_TENSOR_MAP_DATA_TYPE_UINT8, dA, 256,
                                static_cast<uint64_t>(a.blocks) * static_cast<uint64_t>(gpad) * 2, 256, 256,
                                2 * atoms_per_stage);
  if (st == QK_OK)
    st = encode_tmap_2d_plain(mapB, CU_TENSOR_MAP_DATA_TYPE_UINT8, dB, 256,
                              static_cast<uint64_t>(b.blocks) * static_cast<uint64_t>(gpad) * 2, 256, 256,
                              2 * atoms_per_stage);
  return st;
}

// A block-scaled GEMM of configuration C: operand tensor maps, the scale-atom
// pre-pass into a workspace from the device's stream-ordered pool (returned to
// the pool on the same stream after the launch), and the GEMM.  A, B: packed
// operand rows of K * elem_bits / 8 bytes; sA [M, K / SF_BLOCK]; sB
// [ceil(N / b_rows_per), K / SF_BLOCK]; ga, gb: NVFP4 per-tensor scales.
template <class C>
int launch_block_scaled(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, int b_rows_per,
                        const float* ga, const float* gb, const uint16_t* bias, void* out, int M, int N, int K,
                        const DeviceInfo& dev, cudaStream_t stream) {
  static_assert(C::MX, "block-scaled configurations only");
  const uint64_t kbytes = C::FP4 ? static_cast<uint64_t>(K) / 2 : static_cast<uint64_t>(K);
  CUtensorMap ta, tb;
  int st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, kbytes, M, kbytes, C::TMA_K, C::BM);
  if (st == QK_OK) st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kbytes, N, kbytes, C::TMA_K, C::B_LOAD_ROWS);
  if (st != QK_OK) return st;
  GemmParams p{};
  plan_tiles<C>(p, M, N, K);
  p.bias = bias;
  p.out = out;
  p.ga = ga;
  p.gb = gb;
  p.err = dev.err_word;
  p.timeout_ns = wait_timeout_ns();
  p.sf_gpad = p.num_kb * C::SF_ATOMS_K;
  const int cols = K / C::SF_BLOCK;
  const size_t a_bytes = static_cast<size_t>((M + 127) / 128) * p.sf_gpad * 512;
  const size_t b_bytes = static_cast<size_t>((N + 127) / 128) * p.sf_gpad * 512;
  void* ws = nullptr;
  if (cudaMallocFromPoolAsync(&ws, a_bytes + b_bytes, dev.pool, stream) != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_NOMEM;
  }
  uint8_t* atoms_a = static_cast<uint8_t*>(ws);
  uint8_t* atoms_b = atoms_a + a_bytes;
  CUtensorMap tsa, tsb;
  st = write_sf_atoms(sA, atoms_a, M, sB, atoms_b, N, b_rows_per, cols, p.sf_gpad, C::SF_ATOMS_K, &tsa, &tsb, stream);
  // the GEMM overlaps its prologue with the pre-pass (programmatic dependent
  // launch); its producer waits for the pre-pass before the first load
  if (st == QK_OK) st = launch_gemm<C>(ta, tb, tsa, tsb, p, dev, stream, true);
  if (cudaFreeAsync(ws, stream) != cudaSuccess && st == QK_OK) st = QK_ERR_CUDA;
  return st;
}

}  // namespace qk
