// qk_internal.h -- host-side plumbing shared by the libqk.so translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qk.h"

namespace qk {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0;
  int cc_minor = 0;
  unsigned long long* err_word = nullptr;  // device address of the status word
  cudaMemPool_t pool = nullptr;            // stream-ordered workspace pool
};

// Cached facts about the current device, with its workspace pool created on
// first use; nullptr and *status set on failure.
const DeviceInfo* current_device(int* status);
// The same facts without creating the workspace pool (pool may be null).
const DeviceInfo* current_device_basics(int* status);

// 2-D tiled tensor map over a row-major [rows, inner] matrix with a 128-byte
// swizzle and zero fill outside the matrix.  Returns QK_OK or QK_ERR_CUDA.
int encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t rows,
                   uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows);

// The same without swizzle (raw byte rows, e.g. scale factors).
int encode_tmap_2d_plain(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                         uint64_t rows, uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows);

// bf16 [rows, cols] output in 32x32 boxes with the 64-byte swizzle.
// The output as 32x32 boxes: bf16 / fp16 with the 64-byte swizzle, fp32 with
// the 128-byte swizzle (out_type: a QK_OUT_* value).
// the output in boxes of 32 rows x block_cols (32, or 16 for 16-bit types) columns
int encode_tmap_out(CUtensorMap* map, void* out, uint64_t rows, uint64_t cols, int out_type, int block_cols);

uint64_t wait_timeout_ns();
void count_launches(uint64_t n);

// Kernel kinds for the optional per-kernel timing (order of kKernelNames).
enum KernelKind : int {
  kKInt8ToF16 = 0,
  kKGemmInt8 = 1,
  kKGemmFp8 = 2,
  kKGemmMxfp8 = 3,
  kKGemmMxfp4 = 4,
  kKWaitProbe = 5,
  kKQuantize = 6,
  kKGemmNvfp4 = 7,
  kKGemmFp8Blockscale = 8,
  kKSfAtoms = 9,
  kKNumKinds = 10,
};

// Brackets one kernel launch with an event pair when timing is enabled.
struct LaunchTimer {
  LaunchTimer(int kind, cudaStream_t stream);
  void done();  // call right after the launch
  int kind_;
  cudaStream_t stream_;
  cudaEvent_t start_ = nullptr;
};

// Per-format launchers (arguments already validated).
int launch_int8_rowwise_out(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                            const uint16_t* bias, void* out, int out_type, int M, int N, int K, const DeviceInfo& dev,
                            cudaStream_t stream);
int launch_int8_rowwise(const int8_t* A, const int8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                        uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream);
int launch_fp8_rowwise(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                       uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream);
int launch_fp8_rowwise_out(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                           void* out, int out_type, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream);
int launch_mxfp8(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const uint16_t* bias,
                 uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream);
int launch_mxfp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const uint16_t* bias,
                 uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream);
// the same with a QK_OUT_* output type (fp16 / fp32: the tile kernel for every M)
int launch_mxfp8_out(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const uint16_t* bias,
                     void* out, int out_type, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream);
int launch_mxfp4_out(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const uint16_t* bias,
                     void* out, int out_type, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream);
// MX with B scales per 32x32 block ([ceil(N/32), K/32] bytes).
int launch_mxfp8_b32(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB32,
                     const uint16_t* bias, uint16_t* out, int M, int N, int K, const DeviceInfo& dev,
                     cudaStream_t stream);
int launch_mxfp4_b32(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB32,
                     const uint16_t* bias, uint16_t* out, int M, int N, int K, const DeviceInfo& dev,
                     cudaStream_t stream);
int launch_fp8_blockscale(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                          const uint16_t* bias, uint16_t* out, int M, int N, int K, const DeviceInfo& dev,
                          cudaStream_t stream);
int launch_wait_probe(uint64_t timeout_ns, const DeviceInfo& dev, cudaStream_t stream);

}  // namespace qk
