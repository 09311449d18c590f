// q4k_api.cu -- the C ABI of libq4k (include/q4k.h): argument checks, one-time
// per-device set-up, TMA descriptor encoding and dispatch by M.
//
// Dispatch (the decode / prefill split of the rlx-llama32 page's "Decode" and
// "Packed GGUF" sections):
//   q4k_dequant              -> K1 q4k_dequant_kernel
//   q4k_matmul      M <= 2   -> K2 q4k_gemv_kernel (CUDA cores, fp32 activations)
//                   3..16    -> K4 q4k_tcgemv_kernel (tensor cores, fp32 accuracy)
//                   M >  16  -> the same over consecutive 16-row slices of X
//   q4k_matmul_bf16 M <= 16  -> K2 / K4 as above (bf16 activations)
//                   M >= 17  -> K3 q4k_gemm_kernel (tcgen05, TMEM accumulators)
//   q4k_matmul_multi[_bf16]  -> the same, for up to 8 matrices sharing K and X,
//                   all of them in one launch (per 16-row slice for fp32 M > 16)
//   q4k_matmul_argmax[_bf16] -> K2 / K4 with the fused argmax epilogue (M <= 16)
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <memory>
#include <mutex>

#include "q4k.h"
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

// Device error word: bit 0 = a bounded in-kernel wait ran out. Kernels receive
// its device address (resolved per device in init_device).
__device__ unsigned int g_device_error = 0;

// The failure path of the bounded waits, on demand: one thread waits on an
// mbarrier that nothing ever arrives at, with a short limit. The wait runs out,
// sets the error word exactly as a timed-out pipeline wait would, and the
// kernel returns. No copy or tensor-core operation is in flight.
__global__ void q4k_selftest_timeout_kernel(unsigned long long limit_ns, unsigned int* err) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x == 0) {
        const uint32_t b = smem_u32(&bar);
        mbar_init(b, 1);
        fence_barrier_init();
        (void)mbar_wait(b, 0, err, limit_ns);
    }
}

namespace {

// Decode products with at least this many activation rows (and at most 16)
// run on the tensor cores (K4), fewer on the CUDA cores (K2). K4's rate is
// bound by the SM's MMA issue rate whatever M is; K2's falls with M. Measured
// on the Qwen3-14B-shaped sweep: M = 1 K2 2.07 ms vs K4 3.3 ms; M = 4 K2 4.9
// ms vs K4 4.25 ms; M = 16 K2 19.0 ms vs K4 6.2 ms.
#ifndef Q4K_TC_MIN_M
#define Q4K_TC_MIN_M 3
#endif

cudaError_t launch_decode(const WeightGroup& grp, const void* X, bool xb, int M, int K, cudaStream_t stream,
                          const DeviceInfo& dev, int pdl, unsigned long long* amax = nullptr) {
    if (M >= Q4K_TC_MIN_M) return launch_tcgemv(grp, X, xb, M, K, stream, dev, pdl, amax);
    return launch_gemv(grp, X, xb, M, K, stream, dev, pdl, amax);
}

// bf16 activations with at most this many rows run the decode kernels; more
// rows run the tcgen05 GEMM. (A 32-row variant of the tensor-core decode
// kernel was measured at 240 us per Qwen3-8B-shaped layer of 32 rows against
// the GEMM's 87 us: with 32 columns its readout of 8 sub-blocks x 32 rows per
// super-block outweighs the MMAs, so 17.. rows stay on the GEMM.)
#ifndef Q4K_DECODE_MAX_BF16
#define Q4K_DECODE_MAX_BF16 16
#endif
constexpr int64_t kDecodeMaxBf16 = Q4K_DECODE_MAX_BF16;

constexpr int kMaxDevices = 64;

struct DeviceState {
    std::once_flag once;
    int status = Q4K_OK;
    DeviceInfo info;
};

DeviceState g_dev[kMaxDevices];
std::atomic<int> g_pdl{0};  // q4k_set_pdl mode

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

void init_device(int dev, DeviceState& st) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        st.status = Q4K_ERR_CUDA;
        return;
    }
    if (prop.major != 10 || prop.minor != 3) {
        st.status = Q4K_ERR_ARCH;
        return;
    }
    st.info.num_sms = prop.multiProcessorCount;
    st.info.max_smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess || gemv_setup(st.info) != cudaSuccess || tcgemv_setup(st.info) != cudaSuccess ||
        gemm_setup(st.info) != cudaSuccess || encoder() == nullptr) {
        st.status = Q4K_ERR_CUDA;
        return;
    }
    st.info.err = static_cast<unsigned int*>(p);
    st.status = Q4K_OK;
}

int current_device(const DeviceInfo** info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return Q4K_ERR_CUDA;
    DeviceState& st = g_dev[dev];
    std::call_once(st.once, [&] { init_device(dev, st); });
    if (st.status != Q4K_OK) return st.status;
    *info = &st.info;
    return Q4K_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Limits keep every index the kernels form in 32 bits where they use int.
int check_dims(int64_t N, int64_t K) {
    if (N < 1 || K < 256 || K % 256 != 0) return Q4K_ERR_BAD_DIM;
    if (N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 24)) return Q4K_ERR_BAD_DIM;
    return Q4K_OK;
}

// Encoded tensor maps, cached per host thread. A map is a pure function of the
// base address, the tensor's dimensions and the box (everything else is fixed
// per kind), so a cached map is valid for any later call with the same key --
// whatever the memory holds by then. Direct-mapped: a collision re-encodes.
// (A decode step issues one call per weight matrix, every token, with the same
// pointers: the cache takes cuTensorMapEncodeTiled off that host path.)
struct MapKey {
    uintptr_t ptr;
    int64_t a, b;
    int box, kind;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && a == o.a && b == o.b && box == o.box && kind == o.kind;
    }
};
struct MapEntry {
    CUtensorMap map;
    MapKey key;
    bool valid;
};
constexpr int kMapCacheSize = 1024;

MapEntry* map_slot(const MapKey& k) {
    thread_local std::unique_ptr<MapEntry[]> cache;
    if (!cache) {
        cache.reset(new MapEntry[kMapCacheSize]);
        for (int i = 0; i < kMapCacheSize; ++i) cache[i].valid = false;
    }
    uint64_t h = static_cast<uint64_t>(k.ptr >> 4) * 0x9E3779B97F4A7C15ull;
    h ^= static_cast<uint64_t>(k.a) * 0xBF58476D1CE4E5B9ull;
    h ^= static_cast<uint64_t>(k.b) * 0x94D049BB133111EBull;
    h ^= static_cast<uint64_t>(k.box * 4 + k.kind);
    return &cache[(h >> 40) % kMapCacheSize];
}

// W as a 2-D byte tensor {K/256*144, N}; box = one super-block of `rows` rows.
int encode_w_uncached(CUtensorMap* map, const void* W, int64_t N, int64_t K, int rows) {
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(K / 256) * 144;
    const cuuint64_t dims[2] = {row_bytes, static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {144, static_cast<cuuint32_t>(rows)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encoder()(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? Q4K_OK : Q4K_ERR_CUDA;
}

int encode_w(CUtensorMap* map, const void* W, int64_t N, int64_t K, int rows) {
    const MapKey key{reinterpret_cast<uintptr_t>(W), N, K, rows, 0};
    MapEntry* e = map_slot(key);
    if (e->valid && e->key == key) {
        *map = e->map;
        return Q4K_OK;
    }
    const int rc = encode_w_uncached(map, W, N, K, rows);
    if (rc == Q4K_OK) {
        e->map = *map;
        e->key = key;
        e->valid = true;
    }
    return rc;
}

// X as a 2-D bf16 tensor {K, M}; box {64, BN} with the 128-byte swizzle.
// X [M][K] bf16 as a 3-D tensor {64 k, M rows, K / 64 blocks of 64 k} (strides
// 2K bytes per row, 128 bytes per k block): a box {64, BN, s} lands as s
// consecutive k-major, 128-byte-swizzled tiles of BN rows x 64 k.
int encode_x_bf16_uncached(CUtensorMap* map, const void* X, int64_t M, int64_t K, int BN) {
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BN), static_cast<cuuint32_t>(gemm_x_steps(BN))};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encoder()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(X), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? Q4K_OK : Q4K_ERR_CUDA;
}

int encode_x_bf16(CUtensorMap* map, const void* X, int64_t M, int64_t K, int BN) {
    const MapKey key{reinterpret_cast<uintptr_t>(X), M, K, BN, 1};
    MapEntry* e = map_slot(key);
    if (e->valid && e->key == key) {
        *map = e->map;
        return Q4K_OK;
    }
    const int rc = encode_x_bf16_uncached(map, X, M, K, BN);
    if (rc == Q4K_OK) {
        e->map = *map;
        e->key = key;
        e->valid = true;
    }
    return rc;
}

// Tensor maps and the 128-row tile table of `count` matrices sharing K.
int make_group(WeightGroup* grp, int count, const void* const* W, const int64_t* N, int64_t K) {
    grp->count = count;
    grp->tile_start[0] = 0;
    for (int i = 0; i < count; ++i) {
        const int rc = encode_w(&grp->maps[i], W[i], N[i], K, 128);
        if (rc != Q4K_OK) return rc;
        grp->N[i] = static_cast<int>(N[i]);
        grp->tile_start[i + 1] = grp->tile_start[i] + static_cast<int>((N[i] + 127) / 128);
    }
    return Q4K_OK;
}

// One decode launch per 16-row slice of X over `count` matrices sharing K and X.
int run_gemv(int count, const void* const* W, const int64_t* N, int64_t K, const void* X, bool xb,
             int64_t M, float* const* Y, cudaStream_t stream, const DeviceInfo& dev) {
    WeightGroup grp;
    const int rc = make_group(&grp, count, W, N, K);
    if (rc != Q4K_OK) return rc;
    const size_t xelem = xb ? 2 : 4;
    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        const int mc = static_cast<int>(M - m0 < 16 ? M - m0 : 16);
        const void* Xc = static_cast<const uint8_t*>(X) + static_cast<size_t>(m0) * K * xelem;
        for (int i = 0; i < count; ++i) grp.Y[i] = Y[i] + m0 * N[i];
        if (launch_decode(grp, Xc, xb, mc, static_cast<int>(K), stream, dev,
                          g_pdl.load(std::memory_order_relaxed)) != cudaSuccess)
            return Q4K_ERR_CUDA;
    }
    return Q4K_OK;
}

// One GEMM launch over `count` matrices sharing K and X, per chunk of at most
// 65535 * 32 rows of X, fewer when the grid (weight tiles x token tiles of at
// least 32 rows) would pass 2^31 - 1 CTAs.
int run_gemm(int count, const void* const* W, const int64_t* N, int64_t K, const uint16_t* X,
             int64_t M, float* const* Y, cudaStream_t stream, const DeviceInfo& dev) {
    WeightGroup grp;
    int rc = make_group(&grp, count, W, N, K);
    if (rc != Q4K_OK) return rc;
    const int64_t by_grid = 32 * (((int64_t(1) << 31) - 1) / grp.tile_start[count]);
    const int64_t kChunk = by_grid < 65535LL * 32 ? by_grid : 65535LL * 32;
    for (int64_t m0 = 0; m0 < M; m0 += kChunk) {
        const int mc = static_cast<int>(M - m0 < kChunk ? M - m0 : kChunk);
        const GemmPlan plan = gemm_plan(mc, grp.tile_start[count], static_cast<int>(K), dev);
        CUtensorMap tx;
        if ((rc = encode_x_bf16(&tx, X + m0 * K, mc, K, plan.BN)) != Q4K_OK) return rc;
        for (int i = 0; i < count; ++i) grp.Y[i] = Y[i] + m0 * N[i];
        for (int p = 0; p < plan.nlaunch; ++p)
            if (launch_gemm(grp, tx, mc, static_cast<int>(K), plan.BN, plan.part[p], stream, dev,
                            g_pdl.load(std::memory_order_relaxed)) != cudaSuccess)
                return Q4K_ERR_CUDA;
    }
    return Q4K_OK;
}

// Fused GEMV + argmax (M <= 16): the keys live in `out` itself until the last
// kernel turns them into row indices.
int run_argmax(const void* W, int64_t N, int64_t K, const void* X, bool xb, int64_t M, int64_t* out,
               cudaStream_t stream, const DeviceInfo& dev) {
    WeightGroup grp;
    const int rc = make_group(&grp, 1, &W, &N, K);
    if (rc != Q4K_OK) return rc;
    grp.Y[0] = nullptr;
    auto* keys = reinterpret_cast<unsigned long long*>(out);
    const int m = static_cast<int>(M);
    if (launch_argmax_init(keys, m, stream) != cudaSuccess ||
        launch_decode(grp, X, xb, m, static_cast<int>(K), stream, dev,
                      g_pdl.load(std::memory_order_relaxed), keys) != cudaSuccess ||
        launch_argmax_finish(keys, m, stream) != cudaSuccess)
        return Q4K_ERR_CUDA;
    return Q4K_OK;
}

int check_argmax(const void* W, int64_t N, int64_t K, const void* X, int64_t M, const int64_t* out) {
    if (!W || !X || !out) return Q4K_ERR_NULL;
    const int rc = check_dims(N, K);
    if (rc != Q4K_OK) return rc;
    if (M < 1 || M > 16) return Q4K_ERR_BAD_DIM;
    if (!aligned16(W) || !aligned16(X) || (reinterpret_cast<uintptr_t>(out) & 7u) != 0) return Q4K_ERR_ALIGN;
    return Q4K_OK;
}

// Checks shared by the single and grouped matmul calls.
int check_matmul(int count, const void* const* W, const int64_t* N, int64_t K, const void* X,
                 int64_t M, float* const* Y) {
    if (!W || !N || !X || !Y) return Q4K_ERR_NULL;
    if (count < 1 || count > kMaxGroup) return Q4K_ERR_BAD_DIM;
    if (M < 1 || M > (int64_t(1) << 31) - 1) return Q4K_ERR_BAD_DIM;
    for (int i = 0; i < count; ++i) {
        if (!W[i] || !Y[i]) return Q4K_ERR_NULL;
        const int rc = check_dims(N[i], K);
        if (rc != Q4K_OK) return rc;
    }
    if (!aligned16(X)) return Q4K_ERR_ALIGN;
    for (int i = 0; i < count; ++i)
        if (!aligned16(W[i]) || !aligned16(Y[i])) return Q4K_ERR_ALIGN;
    return Q4K_OK;
}

}  // namespace
}  // namespace q4k

using namespace q4k;

extern "C" {

const char* q4k_status_string(int status) {
    switch (status) {
        case Q4K_OK: return "Q4K_OK";
        case Q4K_ERR_NULL: return "Q4K_ERR_NULL: a required pointer is NULL";
        case Q4K_ERR_BAD_DIM:
            return "Q4K_ERR_BAD_DIM: a size or mode is out of range (N, M >= 1; K >= 256, K % 256 == 0; "
                   "N, M < 2^31; K <= 2^24; group count 1..8; argmax M <= 16; PDL mode 0..2)";
        case Q4K_ERR_CUDA: return "Q4K_ERR_CUDA: a CUDA call or kernel launch failed";
        case Q4K_ERR_ALIGN: return "Q4K_ERR_ALIGN: W, X, Y and out must be 16-byte aligned";
        case Q4K_ERR_ARCH: return "Q4K_ERR_ARCH: the current device is not compute capability 10.3";
        case Q4K_ERR_TIMEOUT: return "Q4K_ERR_TIMEOUT: an in-kernel wait ran out of time";
    }
    return "unknown q4k status";
}

int q4k_init(void) {
    const DeviceInfo* info = nullptr;
    return current_device(&info);
}

int q4k_dequant(const void* W, int64_t N, int64_t K, float* out_f32, void* stream) {
    if (!W || !out_f32) return Q4K_ERR_NULL;
    int rc = check_dims(N, K);
    if (rc != Q4K_OK) return rc;
    if (!aligned16(W) || !aligned16(out_f32)) return Q4K_ERR_ALIGN;
    const DeviceInfo* dev = nullptr;
    if ((rc = current_device(&dev)) != Q4K_OK) return rc;
    if (launch_dequant(static_cast<const uint8_t*>(W), N, K, out_f32,
                       static_cast<cudaStream_t>(stream), dev->num_sms) != cudaSuccess)
        return Q4K_ERR_CUDA;
    return Q4K_OK;
}

int q4k_matmul(const void* W, int64_t N, int64_t K, const float* X, int64_t M, float* Y,
               void* stream) {
    if (!W || !X || !Y) return Q4K_ERR_NULL;
    int rc = check_matmul(1, &W, &N, K, X, M, &Y);
    if (rc != Q4K_OK) return rc;
    const DeviceInfo* dev = nullptr;
    if ((rc = current_device(&dev)) != Q4K_OK) return rc;
    return run_gemv(1, &W, &N, K, X, false, M, &Y, static_cast<cudaStream_t>(stream), *dev);
}

int q4k_matmul_bf16(const void* W, int64_t N, int64_t K, const uint16_t* X_bf16, int64_t M,
                    float* Y, void* stream) {
    if (!W || !X_bf16 || !Y) return Q4K_ERR_NULL;
    int rc = check_matmul(1, &W, &N, K, X_bf16, M, &Y);
    if (rc != Q4K_OK) return rc;
    const DeviceInfo* dev = nullptr;
    if ((rc = current_device(&dev)) != Q4K_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M <= kDecodeMaxBf16) return run_gemv(1, &W, &N, K, X_bf16, true, M, &Y, st, *dev);
    return run_gemm(1, &W, &N, K, X_bf16, M, &Y, st, *dev);
}

int q4k_matmul_multi(int count, const void* const* W, const int64_t* N, int64_t K, const float* X,
                     int64_t M, float* const* Y, void* stream) {
    int rc = check_matmul(count, W, N, K, X, M, Y);
    if (rc != Q4K_OK) return rc;
    const DeviceInfo* dev = nullptr;
    if ((rc = current_device(&dev)) != Q4K_OK) return rc;
    return run_gemv(count, W, N, K, X, false, M, Y, static_cast<cudaStream_t>(stream), *dev);
}

int q4k_matmul_multi_bf16(int count, const void* const* W, const int64_t* N, int64_t K,
                          const uint16_t* X_bf16, int64_t M, float* const* Y, void* stream) {
    int rc = check_matmul(count, W, N, K, X_bf16, M, Y);
    if (rc != Q4K_OK) return rc;
    const DeviceInfo* dev = nullptr;
    if ((rc = current_device(&dev)) != Q4K_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M <= kDecodeMaxBf16) return run_gemv(count, W, N, K, X_bf16, true, M, Y, st, *dev);
    return run_gemm(count, W, N, K, X_bf16, M, Y, st, *dev);
}

int q4k_matmul_argmax(const void* W, int64_t N, int64_t K, const float* X, int64_t M,
                      int64_t* out_idx, void* stream) {
    int rc = check_argmax(W, N, K, X, M, out_idx);
    if (rc != Q4K_OK) return rc;
    const DeviceInfo* dev = nullptr;
    if ((rc = current_device(&dev)) != Q4K_OK) return rc;
    return run_argmax(W, N, K, X, false, M, out_idx, static_cast<cudaStream_t>(stream), *dev);
}

int q4k_matmul_argmax_bf16(const void* W, int64_t N, int64_t K, const uint16_t* X_bf16, int64_t M,
                           int64_t* out_idx, void* stream) {
    int rc = check_argmax(W, N, K, X_bf16, M, out_idx);
    if (rc != Q4K_OK) return rc;
    const DeviceInfo* dev = nullptr;
    if ((rc = current_device(&dev)) != Q4K_OK) return rc;
    return run_argmax(W, N, K, X_bf16, true, M, out_idx, static_cast<cudaStream_t>(stream), *dev);
}

int q4k_set_pdl(int mode) {
    if (mode < 0 || mode > 2) return Q4K_ERR_BAD_DIM;
    return g_pdl.exchange(mode);
}

int q4k_selftest_timeout(int64_t limit_ns, void* stream) {
    if (limit_ns < 1 || limit_ns > 1000000000LL) return Q4K_ERR_BAD_DIM;
    const DeviceInfo* dev = nullptr;
    const int rc = current_device(&dev);
    if (rc != Q4K_OK) return rc;
    q4k_selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned long long>(limit_ns), dev->err);
    return cudaGetLastError() == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}

int q4k_device_error(int clear) {
    const DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != Q4K_OK) return rc;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return Q4K_ERR_CUDA;
    if (clear && v) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return Q4K_ERR_CUDA;
    }
    return v ? Q4K_ERR_TIMEOUT : Q4K_OK;
}

}  // extern "C"
