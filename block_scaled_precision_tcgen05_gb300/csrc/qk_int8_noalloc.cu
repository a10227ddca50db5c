// qk_int8_noalloc.cu -- the INT8 GEMM for callers that cannot allocate.
//
// qk_gemm_int8_rowwise widens A and B to f16 in a workspace it takes from a
// stream-ordered memory pool.  Some callers cannot let a library allocate
// device memory: a serving process that handed all of HBM to its own
// allocator up front (a fresh allocation would fail or fragment its budget),
// code that must not pay for or block on allocator calls in its hot loop, or
// an environment whose policy forbids a library to take memory behind the
// caller's back.  qk_gemm_int8_rowwise_noalloc computes the same bit-exact
// result without any allocation: the widened operands go to a fixed scratch
// array compiled into this library, which every GPU that loads the library
// holds until the process exits.
//
// Limits and sharing:
//  - the scratch holds kScratchBytes = 32 MiB, i.e. (M + N) * K <= 16 Mi
//    elements; larger problems are rejected with QK_ERR_SCRATCH before
//    anything is launched;
//  - every call on a device uses the same array.  Calls whose kernels overlap
//    on the GPU (different streams without ordering between them) race on it
//    and give wrong results; calls on one stream, or otherwise ordered, are
//    safe.  The array keeps the last call's contents; nothing in it needs to
//    start at zero, because each call's widening pass writes every element
//    its GEMM then reads;
//  - the first call on a device looks up the array's device address on that
//    device (cudaGetSymbolAddress, with the device current), and the first
//    call of any entry point on a device also queries the device's
//    attributes.  Make that first call before any stream capture.
//  - no cudaMalloc, cudaFree, memory-pool call or other allocating routine is
//    made on this path.
#include <mutex>

#include "qk_int8_exact.cuh"

namespace qk {
namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDev];

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current.
int scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDev) return QK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return QK_ERR_CUDA;
    }
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return QK_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace qk

extern "C" int qk_gemm_int8_rowwise_noalloc(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                                            const uint16_t* bias, uint16_t* out, int64_t M, int64_t N, int64_t K,
                                            qk_stream_t stream) {
  using namespace qk;
  if (M < 0 || N < 0 || K < 1) return QK_ERR_ARG;
  if (M == 0 || N == 0) return QK_OK;
  if (!A || !B || !sa || !sb || !out) return QK_ERR_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(sa) || !aligned16(sb) || !aligned16(out) ||
      (bias && !aligned16(bias)))
    return QK_ERR_ALIGN;
  if (N % 8 != 0 || K % 16 != 0) return QK_ERR_ALIGN;
  if (M > INT32_MAX || N > INT32_MAX || K > 131056) return QK_ERR_RANGE;
  if (static_cast<uint64_t>(M + N) * static_cast<uint64_t>(K) * 2u > kScratchBytes) return QK_ERR_SCRATCH;
  int st = QK_OK;
  const DeviceInfo* dev = current_device_basics(&st);
  if (!dev) return st;
  void* scratch = nullptr;
  st = scratch_address(dev->device, &scratch);
  if (st != QK_OK) return st;
  uint16_t* a16 = static_cast<uint16_t*>(scratch);
  uint16_t* b16 = a16 + static_cast<size_t>(M) * static_cast<size_t>(K);
  return widen_and_gemm_int8(A, B, sa, sb, bias, out, static_cast<int>(M), static_cast<int>(N),
                             static_cast<int>(K), a16, b16, *dev, static_cast<cudaStream_t>(stream));
}
