/*
 * q4k.h -- C ABI of libq4k, a GB300 (sm_103a) library for the packed Q4_K
 * dequant-matmul: the Op::DequantMatMul that the rlx pages emit for every
 * linear layer of a GGUF K-quant model ("rlx-qwen3" crate page, packed-GGUF
 * note under "Quick start": K-quant tensors stay packed and each matmul
 * dequantises them; "rlx-llama32" crate page, section "Packed GGUF").
 *
 * Weights stay in device memory in their 144-byte Q4_K super-blocks and are
 * dequantised inside the kernels.
 *
 * ---------------------------------------------------------------- layout ---
 * W : uint8, N rows of K/256 super-blocks, row-major. Row n's super-blocks are
 *     contiguous and in k order; super-block b of row n starts at byte
 *     (n*K/256 + b)*144. A super-block encodes weights 256b .. 256b+255:
 *       bytes 0..1   d     IEEE binary16, little-endian
 *       bytes 2..3   dmin  IEEE binary16, little-endian
 *       bytes 4..15  s[12] eight 6-bit sub-block scales and eight 6-bit mins:
 *                    sub-block j<4 : sc = s[j]&63, m = s[j+4]&63
 *                    sub-block j>=4: sc = (s[j+4]&15) | ((s[j-4]>>6)<<4),
 *                                    m  = (s[j+4]>>4) | ((s[j]>>6)<<4)
 *       bytes 16..143 qs[128]: byte 32c+l holds weight 64c+l in its low
 *                    nibble and weight 64c+32+l in its high nibble; weight i
 *                    belongs to sub-block i/32.
 *     Weight value: w = d*sc*q - dmin*m. (Both products are exact in fp32, so
 *     w is the exact value rounded once to fp32.)
 * X : [M][K] row-major activations, fp32 or bfloat16.
 * Y : fp32 [M][N] row-major, Y[m][n] = sum_k X[m][k] * w(n,k). Y is
 *     overwritten, never accumulated into.
 *
 * ---------------------------------------------------------------- calls ---
 * Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 * default stream), allocates nothing, never synchronises the host, and may be
 * captured into a CUDA graph (call q4k_init() once per device before the first
 * capture so that one-time kernel attribute set-up happens outside it).
 * All pointers are device pointers owned by the caller; the library keeps no
 * reference to them after the call returns.
 *
 * ---------------------------------------------------------------- errors ---
 * Arguments are checked on the host before anything is launched; on any
 * negative status nothing was launched, except Q4K_ERR_CUDA (the launch itself
 * failed; the CUDA error is left for the caller to query). A wait inside a
 * kernel that runs out of time (a fault, never expected) sets a device error
 * word and the kernel ends early; q4k_device_error() reports it.
 */
#ifndef Q4K_H_
#define Q4K_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum q4k_status {
    Q4K_OK = 0,
    Q4K_ERR_NULL = -1,     /* a required pointer is NULL */
    Q4K_ERR_BAD_DIM = -2,  /* a size or mode out of range: needs N, M >= 1, K >= 256 and
                              K % 256 == 0, N and M below 2^31, K <= 2^24, 1 <= count <= 8
                              (grouped calls), M <= 16 (argmax calls), mode 0..2 (PDL) */
    Q4K_ERR_CUDA = -3,     /* a CUDA runtime call or kernel launch failed */
    Q4K_ERR_ALIGN = -4,    /* W, X, Y or out not 16-byte aligned */
    Q4K_ERR_ARCH = -5,     /* current device is not compute capability 10.3 */
    Q4K_ERR_TIMEOUT = -6   /* a bounded in-kernel wait ran out (device error word) */
};

/* Human-readable name of a status code (static string, never NULL). */
const char* q4k_status_string(int status);

/*
 * One-time set-up for the current device: checks the architecture and sets the
 * kernels' shared-memory attributes. Called implicitly by the first call on a
 * device; call it explicitly before capturing a CUDA graph.
 */
int q4k_init(void);

/*
 * Standalone dequantisation (the CPU-F32 parity path of the rlx-llama32 page's
 * prefill modes, done on the GPU): out_f32[n*K + k] = w(n, k) for all n < N,
 * k < K. Bit-exact: every weight is the exact d*sc*q - dmin*m rounded once.
 *   W        device, N*K/256*144 bytes, 16-byte aligned
 *   out_f32  device, N*K floats, 16-byte aligned
 */
int q4k_dequant(const void* W, int64_t N, int64_t K, float* out_f32, void* stream);

/*
 * Y = X * W^T with fp32 activations X [M][K]: the packed-weight matmul that
 * each linear layer of a K-quant model emits ("rlx-qwen3" crate page, the
 * packed-GGUF note under "Quick start"; "rlx-llama32" crate page, section
 * "Packed GGUF"), with the weights dequantised inside the kernel.
 * M <= 16 (decode) runs one decode launch (M <= 2: the CUDA-core GEMV; 3..16:
 * the tensor-core kernel, fp32 accuracy kept by splitting X into bf16 hi +
 * lo); larger M runs it over 16-row slices of X, which reads W once per slice
 * (fp32 prefill costs ceil(M/16) weight sweeps; bf16 activations through
 * q4k_matmul_bf16 read W once). Accuracy: |Y - exact| <= 1e-4 * sum_k |X*w|
 * per output.
 *   W  device, N*K/256*144 bytes; X device, M*K floats; Y device, M*N floats;
 *   all 16-byte aligned.
 */
int q4k_matmul(const void* W, int64_t N, int64_t K, const float* X, int64_t M, float* Y,
               void* stream);

/*
 * Y = X * W^T with bfloat16 activations X_bf16 [M][K] (bit patterns): the same
 * packed-weight matmul ("rlx-llama32" crate page, section "Packed GGUF") for a
 * block of token rows, as the chunked prefill of the nx_f32_llm_run_v3 listing
 * issues it. M <= 16 runs the decode kernels (M <= 2 on the CUDA cores, 3..16
 * on the tensor cores with the 4-bit codes as the MMA operand; accuracy 1e-4 *
 * sum|X*w|); M >= 17 (chunked prefill) runs the tcgen05 tensor-core GEMM,
 * which rounds the dequantised weights to bfloat16 (accuracy 5e-3 * sum|X*w|).
 *   W  device, N*K/256*144 bytes; X_bf16 device, M*K uint16; Y device, M*N
 *   floats; all 16-byte aligned.
 */
int q4k_matmul_bf16(const void* W, int64_t N, int64_t K, const uint16_t* X_bf16, int64_t M,
                    float* Y, void* stream);

/*
 * Grouped decode call: Y_i = X * W_i^T for i < count (1 <= count <= 8), where
 * all W_i have the same K and take the same activations X -- e.g. the q, k and
 * v projections of a layer, or its gate and up projections. W, N and Y are
 * host arrays of length count holding device pointers / row counts; Y_i is
 * fp32 [M][N_i]. All matrices run in one launch (fp32 activations with
 * M > 16: one launch per 16-row slice of X), with the kernel and accuracy of
 * q4k_matmul / q4k_matmul_bf16 for the same M. The same checks as the single
 * calls apply to every matrix.
 */
int q4k_matmul_multi(int count, const void* const* W, const int64_t* N, int64_t K, const float* X,
                     int64_t M, float* const* Y, void* stream);
int q4k_matmul_multi_bf16(int count, const void* const* W, const int64_t* N, int64_t K,
                          const uint16_t* X_bf16, int64_t M, float* const* Y, void* stream);

/*
 * Fused lm_head + greedy pick (the device-side version of the host-greedy
 * decode of the "rlx-llama32" crate page, section "Env flags"; the in-graph
 * lm_head there is a DequantMatMul like every other matmul): out_idx[m] =
 * argmax_n Y[m][n] for Y = X * W^T, for 1 <= M <= 16 rows of activations,
 * without writing Y. Ties go to the lowest n; NaN outputs are never picked
 * unless every output of the row is NaN (then 0). Y itself is computed as by
 * q4k_matmul / q4k_matmul_bf16 (accuracy 1e-4 * sum|X*w|), so rows whose two
 * largest outputs differ by less than that may pick either. out_idx: device,
 * int64 [M], 8-byte aligned; it is overwritten (it holds intermediate keys
 * while the call runs). Three kernels on `stream`; allocates nothing.
 */
int q4k_matmul_argmax(const void* W, int64_t N, int64_t K, const float* X, int64_t M,
                      int64_t* out_idx, void* stream);
int q4k_matmul_argmax_bf16(const void* W, int64_t N, int64_t K, const uint16_t* X_bf16, int64_t M,
                           int64_t* out_idx, void* stream);

/*
 * Programmatic dependent launch for every later call in the process (a
 * decode step issues one call per weight matrix, so the gaps between
 * back-to-back kernels matter). Returns the previous mode, or
 * Q4K_ERR_BAD_DIM for an unknown mode.
 *   0  plain launches (default).
 *   1  each call's kernel may be scheduled while the preceding kernel on the
 *      stream is still running; it reads and writes no global memory until
 *      that kernel has completed. Always safe.
 *   2  as 1, and the kernel may also start reading its packed weights W
 *      before the preceding kernel has completed. Only valid when W is not
 *      written by the kernel that immediately precedes the call on the stream
 *      (true for model weights).
 */
int q4k_set_pdl(int mode);

/*
 * Reads the device error word of the current device (synchronous: waits for
 * all prior work on the device). Returns Q4K_OK or Q4K_ERR_TIMEOUT; with
 * clear != 0 the word is reset. Not capturable.
 */
int q4k_device_error(int clear);

/*
 * Exercises the failure path of the in-kernel waits without any fault: one
 * thread of a one-warp kernel waits on an mbarrier that nothing arrives at,
 * bounded by limit_ns nanoseconds (1 .. 10^9). The wait runs out, sets the
 * device error word as a timed-out wait in any libq4k kernel does, and the
 * kernel returns; no copy or tensor-core work is in flight, so the context
 * stays usable. Afterwards q4k_device_error() reports Q4K_ERR_TIMEOUT. For
 * tests of error handling; asynchronous on `stream`. (The pages describe no
 * such call: it checks this library's own timeout mechanism.)
 */
int q4k_selftest_timeout(int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* Q4K_H_ */
