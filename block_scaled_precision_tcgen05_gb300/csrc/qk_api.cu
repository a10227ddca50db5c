// qk_api.cu -- the extern "C" entry points of libqk.so: argument validation,
// per-device state (SM count, status word, workspace pool), tensor-map
// encoding and dispatch to the per-format launchers.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "qk_device.cuh"
#include "qk_internal.h"

namespace qk {

// Status word written by kernels whose bounded waits give up.
__device__ unsigned long long g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
int g_dev_state[kMaxDevices];  // 0 unknown, 1 ready, else a cached QK_ERR_* code
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_timeout_ns{0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

uint64_t default_timeout_ns() {
  const char* s = std::getenv("QK_WAIT_TIMEOUT_MS");
  if (s && *s) {
    const long long ms = std::atoll(s);
    if (ms > 0) return static_cast<uint64_t>(ms) * 1000000ull;
  }
  return 1000000000ull;  // 1 s
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

uint64_t wait_timeout_ns() {
  uint64_t t = g_timeout_ns.load(std::memory_order_relaxed);
  return t ? t : default_timeout_ns();
}

void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {

const char* const kKernelNames[kKNumKinds] = {"int8_to_f16", "gemm_int8_f16", "gemm_fp8",
                                              "gemm_mxfp8",  "gemm_mxfp4",    "wait_probe",
                                              "quantize",    "gemm_nvfp4",    "gemm_fp8_blockscale",
                                              "sf_atoms"};

struct PendingTiming {
  int kind;
  cudaEvent_t start, end;
};

std::atomic<int> g_profile_on{0};
std::mutex g_prof_mu;
std::vector<PendingTiming> g_pending;
uint64_t g_prof_launches[kKNumKinds];
double g_prof_ms[kKNumKinds];

}  // namespace

LaunchTimer::LaunchTimer(int kind, cudaStream_t stream) : kind_(kind), stream_(stream) {
  if (!g_profile_on.load(std::memory_order_relaxed)) return;
  if (cudaEventCreate(&start_) != cudaSuccess || cudaEventRecord(start_, stream_) != cudaSuccess) {
    cudaGetLastError();
    if (start_) cudaEventDestroy(start_);
    start_ = nullptr;
  }
}

void LaunchTimer::done() {
  if (!start_) return;
  cudaEvent_t end = nullptr;
  if (cudaEventCreate(&end) != cudaSuccess || cudaEventRecord(end, stream_) != cudaSuccess) {
    cudaGetLastError();
    cudaEventDestroy(start_);
    if (end) cudaEventDestroy(end);
    start_ = nullptr;
    return;
  }
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_pending.push_back({kind_, start_, end});
  start_ = nullptr;
}

const DeviceInfo* current_device_basics(int* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *status = QK_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_dev_state[dev] == 1) return &g_dev[dev];
  if (g_dev_state[dev] != 0) {
    *status = g_dev_state[dev];
    return nullptr;
  }
  DeviceInfo info;
  info.device = dev;
  if (cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    *status = QK_ERR_CUDA;
    return nullptr;
  }
  if (info.cc_major != 10 || info.cc_minor != 3) {
    g_dev_state[dev] = QK_ERR_ARCH;
    *status = QK_ERR_ARCH;
    return nullptr;
  }
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&info.err_word), g_status_word) != cudaSuccess) {
    cudaGetLastError();
    *status = QK_ERR_CUDA;
    return nullptr;
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      cudaGetLastError();
      *status = QK_ERR_CUDA;
      return nullptr;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  g_dev[dev] = info;
  g_dev_state[dev] = 1;
  return &g_dev[dev];
}

const DeviceInfo* current_device(int* status) {
  const DeviceInfo* basics = current_device_basics(status);
  if (!basics) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& info = g_dev[basics->device];
  if (info.pool) return &info;
  cudaMemPoolProps props = {};
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = info.device;
  cudaMemPool_t pool = nullptr;
  if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
    cudaGetLastError();
    *status = QK_ERR_CUDA;
    return nullptr;
  }
  uint64_t keep = UINT64_MAX;  // keep freed workspace cached in the pool
  cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
  info.pool = pool;
  return &info;
}

namespace {

int encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t rows,
              uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  if (!g_encode) return QK_ERR_CUDA;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? QK_OK : QK_ERR_CUDA;
}

}  // namespace

int encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t rows,
                   uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows) {
  return encode_2d(map, dtype, base, inner, rows, row_pitch_bytes, box_inner, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

int encode_tmap_2d_plain(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                         uint64_t rows, uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows) {
  return encode_2d(map, dtype, base, inner, rows, row_pitch_bytes, box_inner, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

int encode_tmap_out(CUtensorMap* map, void* out, uint64_t rows, uint64_t cols, int out_type, int block_cols) {
  if (out_type == QK_OUT_FP32)
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, out, cols, rows, cols * 4, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  return encode_2d(map, out_type == QK_OUT_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   out, cols, rows, cols * 2, block_cols == 16 ? 16 : 32, 32,
                   block_cols == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
}

int kernel_variant(const char* env_name) {
  const char* s = std::getenv(env_name);
  return (s && *s >= '0' && *s <= '9') ? (*s - '0') : 0;
}

int raster_group_m() {
  static const int g = [] {
    const char* s = std::getenv("QK_GROUP_M");
    const int v = (s && *s) ? std::atoi(s) : 0;
    return (v >= 1 && v <= 4096) ? v : 8;
  }();
  return g;
}

__global__ void qk_wait_probe_kernel(unsigned long long* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1u);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl w{&abort_flag, err, timeout_ns};
    mbar_wait(&bar, 0u, w, kSiteProbe);  // nothing ever arrives
  }
}

int launch_wait_probe(uint64_t timeout_ns, const DeviceInfo& dev, cudaStream_t stream) {
  LaunchTimer timer(kKWaitProbe, stream);
  qk_wait_probe_kernel<<<1, 32, 0, stream>>>(dev.err_word, timeout_ns);
  timer.done();
  if (cudaGetLastError() != cudaSuccess) return QK_ERR_CUDA;
  count_launches(1);
  return QK_OK;
}

}  // namespace qk

using namespace qk;

namespace {

// Shared checks of the row/column-scaled entry points.  Order: sizes, empty
// product, pointers, alignment, ranges.
int check_rowwise(const void* A, const void* B, const float* sa, const float* sb, const uint16_t* bias,
                  const uint16_t* out, int64_t M, int64_t N, int64_t K, int64_t k_max, bool* empty) {
  *empty = false;
  if (M < 0 || N < 0 || K < 1) return QK_ERR_ARG;
  if (M == 0 || N == 0) {
    *empty = true;
    return QK_OK;
  }
  if (!A || !B || !sa || !sb || !out) return QK_ERR_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sa, 16) || !aligned(sb, 16) || !aligned(out, 16) ||
      (bias && !aligned(bias, 16)))
    return QK_ERR_ALIGN;
  if (N % 8 != 0 || K % 16 != 0) return QK_ERR_ALIGN;
  if (M > INT32_MAX || N > INT32_MAX || K > k_max) return QK_ERR_RANGE;
  if (((M + 127) / 128) * ((N + 31) / 32) > INT32_MAX) return QK_ERR_RANGE;
  return QK_OK;
}

// Shared checks of the MX entry points (sB: the per-row or the per-32-row
// scales), in the same order.
int check_mx(int fmt, const void* A, const uint8_t* sA, const void* B, const uint8_t* sB, const uint16_t* bias,
             const void* out, int64_t M, int64_t N, int64_t K, bool* empty) {
  *empty = false;
  if (fmt != QK_FMT_MXFP8_E4M3 && fmt != QK_FMT_MXFP4_E2M1) return QK_ERR_ARG;
  if (M < 0 || N < 0 || K < 1) return QK_ERR_ARG;
  if (M == 0 || N == 0) {
    *empty = true;
    return QK_OK;
  }
  if (!A || !sA || !B || !sB || !out) return QK_ERR_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(out, 16) || (bias && !aligned(bias, 16)) ||
      !aligned(sA, 4) || !aligned(sB, 4))
    return QK_ERR_ALIGN;
  if (N % 8 != 0 || K % 32 != 0) return QK_ERR_ALIGN;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return QK_ERR_RANGE;
  if (((M + 127) / 128) * ((N + 31) / 32) > INT32_MAX) return QK_ERR_RANGE;
  return QK_OK;
}

}  // namespace

extern "C" {

int qk_gemm_int8_rowwise(const int8_t* A, const int8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                         uint16_t* out, int64_t M, int64_t N, int64_t K, qk_stream_t stream) {
  bool empty;
  int st = check_rowwise(A, B, sa, sb, bias, out, M, N, K, 131056, &empty);
  if (st != QK_OK || empty) return st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  return launch_int8_rowwise(A, B, sa, sb, bias, out, static_cast<int>(M), static_cast<int>(N),
                             static_cast<int>(K), *dev, static_cast<cudaStream_t>(stream));
}

int qk_gemm_int8_rowwise_out(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                             const uint16_t* bias, void* out, int out_type, int64_t M, int64_t N, int64_t K,
                             qk_stream_t stream) {
  if (out_type != QK_OUT_BF16 && out_type != QK_OUT_FP16 && out_type != QK_OUT_FP32) return QK_ERR_ARG;
  bool empty;
  int st = check_rowwise(A, B, sa, sb, bias, static_cast<const uint16_t*>(out), M, N, K, 131056, &empty);
  if (st != QK_OK || empty) return st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  return launch_int8_rowwise_out(A, B, sa, sb, bias, out, out_type, static_cast<int>(M), static_cast<int>(N),
                                 static_cast<int>(K), *dev, static_cast<cudaStream_t>(stream));
}

int qk_gemm_fp8_rowwise(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                        uint16_t* out, int64_t M, int64_t N, int64_t K, qk_stream_t stream) {
  bool empty;
  int st = check_rowwise(A, B, sa, sb, bias, out, M, N, K, INT32_MAX, &empty);
  if (st != QK_OK || empty) return st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  return launch_fp8_rowwise(A, B, sa, sb, bias, out, static_cast<int>(M), static_cast<int>(N),
                            static_cast<int>(K), *dev, static_cast<cudaStream_t>(stream));
}

int qk_gemm_fp8_rowwise_out(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                            const uint16_t* bias, void* out, int out_type, int64_t M, int64_t N, int64_t K,
                            qk_stream_t stream) {
  if (out_type != QK_OUT_BF16 && out_type != QK_OUT_FP16 && out_type != QK_OUT_FP32) return QK_ERR_ARG;
  bool empty;
  int st = check_rowwise(A, B, sa, sb, bias, static_cast<const uint16_t*>(out), M, N, K, INT32_MAX, &empty);
  if (st != QK_OK || empty) return st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  return launch_fp8_rowwise_out(A, B, sa, sb, bias, out, out_type, static_cast<int>(M), static_cast<int>(N),
                                static_cast<int>(K), *dev, static_cast<cudaStream_t>(stream));
}

int qk_gemm_mx(int fmt, const void* A, const uint8_t* sA, const void* B, const uint8_t* sB, const uint16_t* bias,
               uint16_t* out, int64_t M, int64_t N, int64_t K, qk_stream_t stream) {
  bool empty;
  int st = check_mx(fmt, A, sA, B, sB, bias, out, M, N, K, &empty);
  if (st != QK_OK || empty) return st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  const auto s = static_cast<cudaStream_t>(stream);
  const auto* a = static_cast<const uint8_t*>(A);
  const auto* b = static_cast<const uint8_t*>(B);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  if (fmt == QK_FMT_MXFP8_E4M3) return launch_mxfp8(a, sA, b, sB, bias, out, m, n, k, *dev, s);
  return launch_mxfp4(a, sA, b, sB, bias, out, m, n, k, *dev, s);
}

int qk_gemm_mx_out(int fmt, const void* A, const uint8_t* sA, const void* B, const uint8_t* sB, const uint16_t* bias,
                   void* out, int out_type, int64_t M, int64_t N, int64_t K, qk_stream_t stream) {
  if (out_type != QK_OUT_BF16 && out_type != QK_OUT_FP16 && out_type != QK_OUT_FP32) return QK_ERR_ARG;
  bool empty;
  int st = check_mx(fmt, A, sA, B, sB, bias, out, M, N, K, &empty);
  if (st != QK_OK || empty) return st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  const auto s = static_cast<cudaStream_t>(stream);
  const auto* a = static_cast<const uint8_t*>(A);
  const auto* b = static_cast<const uint8_t*>(B);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  if (fmt == QK_FMT_MXFP8_E4M3) return launch_mxfp8_out(a, sA, b, sB, bias, out, out_type, m, n, k, *dev, s);
  return launch_mxfp4_out(a, sA, b, sB, bias, out, out_type, m, n, k, *dev, s);
}

int qk_gemm_mx_b32(int fmt, const void* A, const uint8_t* sA, const void* B, const uint8_t* sB32,
                   const uint16_t* bias, uint16_t* out, int64_t M, int64_t N, int64_t K, qk_stream_t stream) {
  bool empty;
  int st = check_mx(fmt, A, sA, B, sB32, bias, out, M, N, K, &empty);
  if (st != QK_OK || empty) return st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  const auto s = static_cast<cudaStream_t>(stream);
  const auto* a = static_cast<const uint8_t*>(A);
  const auto* b = static_cast<const uint8_t*>(B);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  if (fmt == QK_FMT_MXFP8_E4M3) return launch_mxfp8_b32(a, sA, b, sB32, bias, out, m, n, k, *dev, s);
  return launch_mxfp4_b32(a, sA, b, sB32, bias, out, m, n, k, *dev, s);
}

const char* qk_status_string(int status) {
  switch (status) {
    case QK_OK: return "QK_OK";
    case QK_ERR_ARG: return "QK_ERR_ARG: invalid argument (null pointer, negative size, K == 0 or unknown format)";
    case QK_ERR_ALIGN: return "QK_ERR_ALIGN: pointer or size alignment requirement not met";
    case QK_ERR_RANGE: return "QK_ERR_RANGE: size out of the supported range";
    case QK_ERR_ARCH: return "QK_ERR_ARCH: the current device is not a GB300 (compute capability 10.3)";
    case QK_ERR_CUDA: return "QK_ERR_CUDA: a CUDA call or kernel launch failed";
    case QK_ERR_TIMEOUT: return "QK_ERR_TIMEOUT: a bounded wait inside a kernel gave up";
    case QK_ERR_NOMEM: return "QK_ERR_NOMEM: workspace allocation failed";
    case QK_ERR_SCRATCH:
      return "QK_ERR_SCRATCH: (M + N) * K * 2 bytes exceed the 32 MiB scratch of qk_gemm_int8_rowwise_noalloc";
    default: return "QK_ERR_UNKNOWN";
  }
}

int qk_device_status(uint64_t* word, int clear) {
  int st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_CUDA;
  }
  unsigned long long v = 0;
  if (cudaMemcpy(&v, dev->err_word, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return QK_ERR_CUDA;
  if (clear && v) {
    const unsigned long long zero = 0;
    if (cudaMemcpy(dev->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return QK_ERR_CUDA;
  }
  if (word) *word = v;
  return QK_OK;
}

void qk_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns, std::memory_order_relaxed); }

int qk_wait_timeout_probe(uint64_t timeout_ns, qk_stream_t stream) {
  int st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  uint64_t before = 0;
  st = qk_device_status(&before, 1);
  if (st != QK_OK) return st;
  st = launch_wait_probe(timeout_ns ? timeout_ns : 1000000ull, *dev, static_cast<cudaStream_t>(stream));
  if (st != QK_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QK_ERR_CUDA;
  uint64_t word = 0;
  st = qk_device_status(&word, 1);
  if (st != QK_OK) return st;
  return (word >> 56) == kDevErrTimeout ? QK_ERR_TIMEOUT : QK_OK;
}

uint64_t qk_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void qk_profile_enable(int on) { g_profile_on.store(on ? 1 : 0, std::memory_order_relaxed); }

int qk_profile_read(qk_kernel_stats* stats, int max, int* count, int reset) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  int st = QK_OK;
  for (const PendingTiming& t : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(t.end) == cudaSuccess && cudaEventElapsedTime(&ms, t.start, t.end) == cudaSuccess) {
      g_prof_launches[t.kind] += 1;
      g_prof_ms[t.kind] += ms;
    } else {
      cudaGetLastError();
      st = QK_ERR_CUDA;
    }
    cudaEventDestroy(t.start);
    cudaEventDestroy(t.end);
  }
  g_pending.clear();
  int n = 0;
  for (int k = 0; k < kKNumKinds; ++k) {
    if (g_prof_launches[k] == 0) continue;
    if (stats && n < max) {
      stats[n].name = kKernelNames[k];
      stats[n].launches = g_prof_launches[k];
      stats[n].total_ms = g_prof_ms[k];
    }
    ++n;
  }
  if (count) *count = n;
  if (reset) {
    for (int k = 0; k < kKNumKinds; ++k) {
      g_prof_launches[k] = 0;
      g_prof_ms[k] = 0.0;
    }
  }
  return st;
}

int qk_release(void) {
  int st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  if (cudaDeviceSynchronize() != cudaSuccess || cudaMemPoolTrimTo(dev->pool, 0) != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_CUDA;
  }
  return QK_OK;
}

int qk_version(void) { return 100; }

}  // extern "C"
