// qk_int8.cu -- exact INT8 row/column-scaled GEMM entry: takes the f16
// workspace from the library's stream-ordered pool, runs the widening pass
// and the f16-pipe GEMM (qk_int8_exact.cuh), and returns the workspace to the
// pool on the same stream.
#include "qk_int8_exact.cuh"

namespace qk {

int launch_int8_rowwise_out(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                            const uint16_t* bias, void* out, int out_type, int M, int N, int K, const DeviceInfo& dev,
                            cudaStream_t stream) {
  const size_t a_elems = static_cast<size_t>(M) * K;
  const size_t b_elems = static_cast<size_t>(N) * K;
  void* ws = nullptr;
  if (cudaMallocFromPoolAsync(&ws, (a_elems + b_elems) * 2, dev.pool, stream) != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_NOMEM;
  }
  uint16_t* a16 = static_cast<uint16_t*>(ws);
  uint16_t* b16 = a16 + a_elems;
  int st;
  if (out_type == QK_OUT_FP32)
    st = widen_and_gemm_int8<CfgInt8F32>(A, B, sa, sb, bias, out, M, N, K, a16, b16, dev, stream);
  else if (out_type == QK_OUT_FP16)
    st = widen_and_gemm_int8<CfgInt8F16>(A, B, sa, sb, bias, out, M, N, K, a16, b16, dev, stream);
  else
    st = widen_and_gemm_int8<CfgInt8>(A, B, sa, sb, bias, out, M, N, K, a16, b16, dev, stream);
  if (cudaFreeAsync(ws, stream) != cudaSuccess && st == QK_OK) st = QK_ERR_CUDA;
  return st;
}

int launch_int8_rowwise(const int8_t* A, const int8_t* B, const float* sa, const float* sb, const uint16_t* bias,
                        uint16_t* out, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  return launch_int8_rowwise_out(A, B, sa, sb, bias, out, QK_OUT_BF16, M, N, K, dev, stream);
}

}  // namespace qk
