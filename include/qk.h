/*
 * qk.h -- C ABI of libqk.so, block-scaled / quantized GEMM on GB300 (sm_103a).
 *
 * Every entry point computes
 *
 *     out[m, n] = bf16_rne( epilogue( sum_k A[m, k] * B[n, k] ) )
 *
 * with A [M, K] and B [N, K] both K-major (row-major, contiguous, leading
 * dimension = K elements), and out [M, N] row-major bf16 (leading dimension
 * N).  All pointers are DEVICE pointers owned by the caller; the library never
 * frees them and keeps no reference to them once the call returns.
 *
 * Calls are stream-ordered and asynchronous: they validate their arguments on
 * the host, enqueue kernels on `stream` (a cudaStream_t; NULL = the legacy
 * default stream of the current device) and return.  Faults inside the
 * kernels surface at the caller's next synchronisation; bounded waits inside
 * the kernels that give up are recorded in a device status word
 * (qk_device_status).  The device is the current CUDA device.
 *
 * bf16 values (bias, out) are passed as their 16-bit patterns (uint16_t).
 * M == 0 or N == 0 is an empty product: nothing is launched and QK_OK is
 * returned.  K must be >= 1.
 *
 * Sources (web pages, cited by title and section):
 *  - comfy-kitchen PR #174 "Optimize HIP WMMA INT8 GEMM staging, epilogue,
 *    and deep-K tiling": Summary, Validation, and the updates "Keep the cached
 *    INT8 epilogue scale order exact" and "Preserve signed zero without INT8
 *    bias".
 *  - ROCm/mori PR #806 "perf(gemm-ar): mxfp8 with row-major scales staged
 *    through LDS": section "What" (raw row-major ue8m0 scales, any M).
 *  - ROCm/FlyDSL PR #990 "[fp4_gemm_4wave] MXFP4 GEMM perf optimize":
 *    MXFP4 with per-1x32 ue8m0 scales.
 *  - ROCm/aiter PR #6262: "Technical Details" (caller-owned out=, shape and
 *    dtype checks; FP8 A8W8 GEMM with per-token and per-channel scales).
 */
#ifndef QK_H_
#define QK_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, passed as an opaque handle. */
typedef void* qk_stream_t;

/* ---- status codes ------------------------------------------------------- */
#define QK_OK 0
#define QK_ERR_ARG 1      /* null required pointer, negative size, K == 0, unknown format */
#define QK_ERR_ALIGN 2    /* a pointer not 16-byte aligned, N % 8 != 0, or K not a multiple of 16 (32 for MX) */
#define QK_ERR_RANGE 3    /* INT8: K > 131056, so the int32 accumulator could overflow; sizes beyond 2^31-1 */
#define QK_ERR_ARCH 4     /* the current device is not compute capability 10.3 (GB300) */
#define QK_ERR_CUDA 5     /* a CUDA runtime/driver call or a kernel launch failed */
#define QK_ERR_TIMEOUT 6  /* a bounded wait inside a kernel gave up (see qk_device_status) */
#define QK_ERR_NOMEM 7    /* the library's stream-ordered workspace could not be allocated */
#define QK_ERR_SCRATCH 8  /* the problem needs more than the fixed scratch of qk_gemm_int8_rowwise_noalloc */

/* ---- operand formats for qk_gemm_mx ------------------------------------ */
#define QK_FMT_MXFP8_E4M3 1 /* A, B: one E4M3 byte per element */
#define QK_FMT_MXFP4_E2M1 2 /* A, B: two E2M1 codes per byte, element 2i in the low nibble */

/* ---- output element types of the *_out entry points ----------------------- */
#define QK_OUT_BF16 0 /* 2 bytes, bf16 round to nearest even */
#define QK_OUT_FP16 1 /* 2 bytes, IEEE half round to nearest even (beyond 65504: +-inf) */
#define QK_OUT_FP32 2 /* 4 bytes, the fp32 value x itself */

/*
 * INT8 GEMM with per-row and per-column fp32 scales and an optional bias.
 * Scales and bias are read once per output tile and applied in a fixed order
 * (comfy-kitchen PR #174, Summary and the update "Keep the cached INT8
 * epilogue scale order exact"); the page validates the result as an exact
 * match of its reference (Validation).
 *
 *   acc      = sum_k A[m,k] * B[n,k]                  exact, int32
 *   x        = (float)acc                             round to nearest even
 *   x        = x * sa[m];  x = x * sb[n]              two fp32 roundings, in this order
 *   if bias:   x = x + (float)bias[n]                 one fp32 add (no FMA)
 *   out[m,n] = bf16 round-to-nearest-even(x)
 * Without bias no add is made, so a -0 produced by the products is kept.
 *
 *   A    int8  [M, K]        B    int8 [N, K]
 *   sa   fp32  [M]           sb   fp32 [N]
 *   bias bf16  [N] or NULL   out  bf16 [M, N]
 * Requirements: all pointers 16-byte aligned; N % 8 == 0; K % 16 == 0;
 * 1 <= K <= 131056.  The result is bit-identical to the definition above.
 * Internally the operands are widened to f16 in a library-owned, stream-
 * ordered workspace of (M + N) * K * 2 bytes that is released back to the
 * library's pool at the end of the call (on the stream).
 */
int qk_gemm_int8_rowwise(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                         const uint16_t* bias, uint16_t* out, int64_t M, int64_t N, int64_t K,
                         qk_stream_t stream);

/*
 * qk_gemm_int8_rowwise with a choice of output element type (comfy-kitchen
 * PR #174, update "rebased onto v0.2.38": the page's INT8 kernel
 * specialization serves bf16, fp16 and fp32 output types).  The same x as
 * above, then
 *   out_type QK_OUT_BF16: out bf16 [M, N] = bf16_rne(x)   (as qk_gemm_int8_rowwise)
 *            QK_OUT_FP16: out fp16 [M, N] = fp16_rne(x)   (+-inf beyond the fp16 range)
 *            QK_OUT_FP32: out fp32 [M, N] = x
 * `out` points to M * N elements of that type.  Arguments, requirements,
 * workspace and bit-exactness as for qk_gemm_int8_rowwise; an unknown
 * out_type returns QK_ERR_ARG.
 */
int qk_gemm_int8_rowwise_out(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                             const uint16_t* bias, void* out, int out_type, int64_t M, int64_t N, int64_t K,
                             qk_stream_t stream);

/*
 * qk_gemm_int8_rowwise without any memory allocation.  (The pages have no
 * counterpart; this entry point exists for callers that cannot let a library
 * allocate device memory: a process that gave all of HBM to its own
 * allocator, a hot loop that must not pay for or block on allocator calls, or
 * a policy that forbids a library to take memory behind the caller's back.)
 *
 * Same arguments, requirements and bit-identical result as
 * qk_gemm_int8_rowwise.  Instead of a pooled workspace it widens A and B into
 * one 32 MiB scratch array compiled into libqk.so, which every GPU that loads
 * the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree, memory-pool or other allocating routine.
 *   - (M + N) * K * 2 must not exceed 32 MiB (33554432 bytes); larger
 *     problems return QK_ERR_SCRATCH without launching anything.
 *   - All calls on a device share that array: calls whose kernels can
 *     overlap on the GPU (unordered streams) race and give wrong results.
 *     Calls ordered on one stream are safe.  The array keeps the last call's
 *     contents; no part of it needs to start at zero.
 *   - The first call on a device looks up the array's device address (and,
 *     as for every entry point, the device's attributes) with that device
 *     current; make this first call before any stream capture.
 */
int qk_gemm_int8_rowwise_noalloc(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                                 const uint16_t* bias, uint16_t* out, int64_t M, int64_t N, int64_t K,
                                 qk_stream_t stream);

/*
 * MX block-scaled GEMM (ROCm/mori PR #806, section "What": one ue8m0 scale
 * per 32 K-elements, held as raw row-major uint8 bytes [rows, K/32] for both
 * operands; ROCm/FlyDSL PR #990: MXFP4 with scales per 1x32 block).
 *
 *   out[m,n] = bf16_rne( sum_b 2^(sA[m,b]-127) * 2^(sB[n,b]-127)
 *                          * sum_{j<32} A[m,32b+j] * B[n,32b+j]   (+ bias[n]) )
 * accumulated in fp32 on the tensor cores (the summation order is free).
 *
 *   fmt  QK_FMT_MXFP8_E4M3: A [M, K] bytes, B [N, K] bytes (E4M3FN)
 *        QK_FMT_MXFP4_E2M1: A [M, K/2] bytes, B [N, K/2] bytes (packed E2M1)
 *   sA   uint8 [M, K/32]  raw row-major UE8M0 exponents (bias 127)
 *   sB   uint8 [N, K/32]
 *   bias bf16 [N] or NULL;  out bf16 [M, N]
 * Requirements: A, B, out, bias 16-byte aligned; sA, sB 4-byte aligned;
 * N % 8 == 0; K % 32 == 0.  Any M >= 1 is accepted without padding.
 * With M <= 128 both formats run the weight-streaming kernels described
 * under qk_gemm_fp8_rowwise: the cluster split-K kernel when all weight
 * tiles' clusters fit on the GPU at once, else the cooperative stream-K
 * launch, with the same pooled workspace, the same QK_ERR_NOMEM case and the
 * same reproducible fixed-order reduction.
 */
int qk_gemm_mx(int fmt, const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
               const uint16_t* bias, uint16_t* out, int64_t M, int64_t N, int64_t K, qk_stream_t stream);

/*
 * MX block-scaled GEMM with B's scales per 32x32 block (ROCm/mori PR #806,
 * section "What": the mxfp8_raw form takes B's scales as [N/32, K/32] uint8,
 * row major, read with 32 rows per scale row in the review thread's scale
 * reader).  A's scales are as in qk_gemm_mx.
 *
 *   out[m,n] = bf16_rne( sum_b 2^(sA[m,b]-127) * 2^(sB32[n/32,b]-127)
 *                          * sum_{j<32} A[m,32b+j] * B[n,32b+j]   (+ bias[n]) )
 * accumulated in fp32 on the tensor cores (the summation order is free).
 *
 *   fmt   QK_FMT_MXFP8_E4M3 or QK_FMT_MXFP4_E2M1, operands as for qk_gemm_mx
 *   sA    uint8 [M, K/32]              raw row-major UE8M0 exponents
 *   sB32  uint8 [ceil(N/32), K/32]     one row per 32 rows of B (integer division;
 *                                      the last group may hold fewer rows)
 *   bias  bf16 [N] or NULL;  out bf16 [M, N]
 * Requirements and errors as for qk_gemm_mx.  Every M runs the 2-SM tile
 * kernel (no few-row mode in this form); the per-call scale pre-pass writes
 * each 32-row group's scale bytes into the places of its 32 rows in the
 * atom buffer, so the form reads 32x fewer B scale bytes from the caller and
 * the GEMM kernel is the same as qk_gemm_mx's.
 */
int qk_gemm_mx_b32(int fmt, const void* A, const uint8_t* sA, const void* B, const uint8_t* sB32,
                   const uint16_t* bias, uint16_t* out, int64_t M, int64_t N, int64_t K, qk_stream_t stream);

/*
 * qk_gemm_mx with a choice of output element type (ROCm/aiter PR #6262: its
 * FP4 GEMM, gemm_a4w4, takes the output dtype as an argument, bf16 by
 * default).  The same fp32 value as qk_gemm_mx computes, then
 *   out_type QK_OUT_BF16: out bf16 [M, N]   (exactly qk_gemm_mx)
 *            QK_OUT_FP16: out fp16 [M, N]   round to nearest even, +-inf beyond the fp16 range
 *            QK_OUT_FP32: out fp32 [M, N]   the value itself
 * fp16 and fp32 outputs run the 2-SM tile kernel for every M (the few-row
 * kernels write bf16 only), so for a given problem the two hold the same
 * value.  Arguments, requirements and errors as for qk_gemm_mx; an unknown
 * out_type returns QK_ERR_ARG.
 */
int qk_gemm_mx_out(int fmt, const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                   const uint16_t* bias, void* out, int out_type, int64_t M, int64_t N, int64_t K,
                   qk_stream_t stream);

/*
 * FP8 E4M3 GEMM with per-token (row) and per-channel (column) fp32 scales
 * (ROCm/aiter PR #6262, gemm_a8w8_bpreshuffle with per-token/per-channel
 * scales; ROCm/mori PR #806, the "ptpc" kind).  Same epilogue as
 * qk_gemm_int8_rowwise, with acc the fp32 tensor-core sum of the decoded
 * E4M3 products.
 *   A uint8 [M, K] E4M3FN; B uint8 [N, K] E4M3FN; sa fp32 [M]; sb fp32 [N];
 *   bias bf16 [N] or NULL; out bf16 [M, N].
 * Requirements: as qk_gemm_int8_rowwise, without the K upper bound.
 * With M <= 128 a weight-streaming kernel runs: split-K over clusters when
 * all weight tiles' clusters fit on the GPU at once, else a cooperative
 * stream-K launch that takes a stream-ordered workspace from the
 * library's pool (one fp32 partial of at most 128 x 128 values and four
 * 8-byte flags per SM, returned at the end of the call); QK_ERR_NOMEM if that
 * allocation fails.  Partials of a shared tile are added in a fixed order, so
 * repeated calls give identical bits.  The few-row kernels may start while
 * the previous kernel of the stream finishes (programmatic dependent launch;
 * they touch memory only after it has completed), and a call may be captured
 * in a CUDA graph and replayed (the stream-K flags are cleared by the time a
 * call completes).
 * With more rows the 2-SM tile kernel runs; when its last wave of tiles would
 * leave at least half of the SM pairs idle after at least one full wave (and
 * K is long enough), those tiles run as 2-4 K-parts whose fp32 partials go
 * through a stream-ordered workspace from the same pool (QK_ERR_NOMEM is not
 * raised for it: without a workspace the tiles run whole) and are added in a
 * fixed order, so repeated calls and graph replays give identical bits.  The
 * same holds for qk_gemm_mx, qk_gemm_mx_b32 and qk_gemm_nvfp4.
 */
int qk_gemm_fp8_rowwise(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                        const uint16_t* bias, uint16_t* out, int64_t M, int64_t N, int64_t K,
                        qk_stream_t stream);

/*
 * qk_gemm_fp8_rowwise with a choice of output element type (ROCm/aiter PR
 * #6262: gemm_a8w8_bpreshuffle takes the output dtype as an argument, bf16 by
 * default, and checks a caller-owned out against it).  The same x as
 * qk_gemm_fp8_rowwise computes, then
 *   out_type QK_OUT_BF16: out bf16 [M, N] = bf16_rne(x)   (as qk_gemm_fp8_rowwise)
 *            QK_OUT_FP16: out fp16 [M, N] = fp16_rne(x)   (+-inf beyond the fp16 range)
 *            QK_OUT_FP32: out fp32 [M, N] = x
 * `out` points to M * N elements of that type.  fp16 and fp32 outputs run
 * the 2-SM tile kernel for every M (the few-row kernels write bf16 only), so
 * for a given problem the two hold the same x.  Arguments, requirements and
 * errors as for qk_gemm_fp8_rowwise; an unknown out_type returns QK_ERR_ARG.
 */
int qk_gemm_fp8_rowwise_out(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                            const uint16_t* bias, void* out, int out_type, int64_t M, int64_t N, int64_t K,
                            qk_stream_t stream);

/*
 * FP8 E4M3 GEMM with fp32 block scales (the "blockscale" kind of ROCm/mori PR
 * #806's measurements; the page does not give the block sizes, read here as
 * DeepSeek-V3's: 1 x 128 for A, 128 x 128 for B).
 *
 *   out[m,n] = bf16_rne( sum_g sa[m,g] * sb[n/128,g] * P_g[m,n]  (+ bias[n]) ),
 *   P_g      = sum over k in [128 g, min(128 g + 128, K)) of A[m,k] * B[n,k]
 * with each P_g an fp32 tensor-core sum and the scaled sum in fp32.
 *
 *   A uint8 [M, K] E4M3FN; B uint8 [N, K] E4M3FN
 *   sa fp32 [M, KB], sb fp32 [NB, KB], row-major, KB = ceil(K/128), NB = ceil(N/128)
 *   bias bf16 [N] or NULL;  out bf16 [M, N]
 * Requirements: A, B, out, bias 16-byte aligned; sa, sb 4-byte aligned;
 * N % 8 == 0; K % 16 == 0.  Any M >= 1.
 */
int qk_gemm_fp8_blockscale(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                           const uint16_t* bias, uint16_t* out, int64_t M, int64_t N, int64_t K,
                           qk_stream_t stream);

/*
 * NVFP4 block-scaled GEMM: E2M1 elements, one UE4M3 scale per 16 K-elements,
 * and one fp32 scale per tensor (ROCm/aiter PR #6262, the gemm_a4w4
 * signature's optional per-tensor NVFP4 scales for A and B; the format is
 * NVIDIA's published NVFP4).
 *
 *   out[m,n] = bf16_rne( acc * fl(ga * gb)  (+ bias[n]) ),
 *   acc      = sum_b ue4m3(sA[m,b]) * ue4m3(sB[n,b]) * sum_{j<16} A[m,16b+j] * B[n,16b+j]
 * with acc the fp32 tensor-core sum (summation order free), then one fp32
 * multiply by the fp32 product of the two per-tensor scales, then the bias
 * add, each rounded to nearest even.
 *
 *   A  uint8 [M, K/2] packed E2M1, element 2i in the low nibble; B uint8 [N, K/2]
 *   sA uint8 [M, K/16] raw row-major UE4M3 (E4M3FN without the sign; bit 7 must
 *      be 0); sB uint8 [N, K/16]
 *   ga, gb  device pointers to one fp32 each, or NULL for 1.0
 *   bias bf16 [N] or NULL;  out bf16 [M, N]
 * Requirements: A, B, out, bias 16-byte aligned; N % 8 == 0; K % 32 == 0.
 * Any M >= 1 is accepted without padding.  Device-side reads of ga/gb happen
 * in the kernel, so their values may be produced earlier on the same stream.
 * With M <= 128 the weight-streaming kernels run where they are faster: the
 * cluster split-K kernel when all weight tiles' clusters fit on the GPU at
 * once, the stream-K launch for M <= 64 with 10 to 30 units of 128 weight
 * rows x 256 K per SM, otherwise the tile kernel.
 */
int qk_gemm_nvfp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const float* ga,
                  const float* gb, const uint16_t* bias, uint16_t* out, int64_t M, int64_t N, int64_t K,
                  qk_stream_t stream);

/*
 * qk_gemm_nvfp4 with a choice of output element type (ROCm/aiter PR #6262:
 * gemm_a4w4 takes the output dtype beside the NVFP4 per-tensor scales), with
 * the output types, kernels and errors of qk_gemm_mx_out.
 */
int qk_gemm_nvfp4_out(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const float* ga,
                      const float* gb, const uint16_t* bias, void* out, int out_type, int64_t M, int64_t N,
                      int64_t K, qk_stream_t stream);

/*
 * Quantizers that produce the operands above from bf16 data.
 *
 * qk_quantize_mx: MX block scaling along K (OCP 1x32, raw row-major scales
 * as ROCm/mori PR #806 "What" holds them).  For each block of 32 elements of
 * a row, s = floor(log2(amax)) - emax (8 for E4M3, 2 for E2M1), clamped to
 * [-127, 127] and -127 for an all-zero block; scales[row, b] = s + 127;
 * elements x * 2^-s rounded to nearest even and saturated to +-448 (E4M3)
 * or +-6 (E2M1).  MXFP4 packs element 2i in the low nibble of byte i.
 *   x      bf16 [rows, K]      q  [rows, K] (E4M3) or [rows, K/2] (E2M1) bytes
 *   scales uint8 [rows, K/32]
 * Requirements: x and q 16-byte aligned, K % 32 == 0.  Finite inputs.
 *
 * qk_quantize_ptpc: per-row FP8 (per-token scales, ROCm/aiter PR #6262):
 * s = amax / 448 in fp32 (1 for an all-zero row), q = E4M3(x / s) with the
 * division and the conversion rounding to nearest even, saturated.
 *   x bf16 [rows, K]; q uint8 [rows, K]; scales fp32 [rows]
 * Requirements: x and q 16-byte aligned, scales 4-byte aligned, K % 16 == 0.
 * Both are bit-identical to these definitions; rows == 0 is a no-op.
 */
int qk_quantize_mx(int fmt, const uint16_t* x, uint8_t* q, uint8_t* scales, int64_t rows, int64_t K,
                   qk_stream_t stream);
int qk_quantize_ptpc(const uint16_t* x, uint8_t* q, float* scales, int64_t rows, int64_t K, qk_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* qk_status_string(int status);

/*
 * Reads (and with clear != 0, resets) the current device's status word that
 * kernels set when a bounded wait gives up.  0 means no failure was recorded.
 * Layout: bits 63..56 code (1 = timeout; 2 = a kernel whose shared-memory
 * layout needs a 1024-byte-aligned base found it unaligned and returned
 * without doing anything), 55..48 site, 47..32 CTA index, 31..0 detail.  Synchronises the device first.  Returns QK_OK or
 * QK_ERR_CUDA; *word may be NULL.
 */
int qk_device_status(uint64_t* word, int clear);

/*
 * Bound, in nanoseconds, on every barrier wait inside the kernels (default
 * 1e9, or QK_WAIT_TIMEOUT_MS from the environment).  0 restores the default.
 */
void qk_set_wait_timeout_ns(uint64_t ns);

/*
 * Launches one block whose barrier wait can never complete, with a wait
 * bound of timeout_ns, synchronises the stream and returns QK_ERR_TIMEOUT if
 * the kernel reported the give-up in the status word (the word is cleared),
 * QK_OK if it did not.  Exercises the failure path of the bounded waits
 * without faulting the GPU.
 */
int qk_wait_timeout_probe(uint64_t timeout_ns, qk_stream_t stream);

/* Number of kernels this library has launched in this process. */
uint64_t qk_launch_count(void);

/*
 * Kernel timing.  While enabled, the library records a CUDA event pair on the
 * launch stream around every kernel it launches.  qk_profile_read waits for
 * the recorded events, adds their durations to per-kernel totals, and copies
 * up to `max` entries (one per kernel kind that ran) into `stats`; *count
 * receives the number of entries.  reset != 0 clears the totals afterwards.
 * Kernel names: "int8_to_f16", "gemm_int8_f16", "gemm_fp8", "gemm_mxfp8",
 * "gemm_mxfp4", "wait_probe", "quantize", "gemm_nvfp4", "gemm_fp8_blockscale".
 */
typedef struct {
  const char* name;   /* static storage */
  uint64_t launches;
  double total_ms;
} qk_kernel_stats;

void qk_profile_enable(int on);
int qk_profile_read(qk_kernel_stats* stats, int max, int* count, int reset);

/* Frees the library's cached workspace memory on the current device. */
int qk_release(void);

/* ABI version (major * 100 + minor). */
int qk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QK_H_ */
