// q4k_gemv.cu -- K2: split-K GEMV for the packed Q4_K decode step (M = 1..16).
//
// Decode reads every packed weight matrix once per token (the per-token weight
// sweep of the rlx-llama32 page, section "Decode"), so this kernel is bound by
// HBM bandwidth at M = 1 and by fp32 issue rate as M grows.
//
// Work decomposition
//   grid.x  = 32-row groups of W (one warp lane per weight row)
//   grid.y  = K splits (a thread-block cluster along y; partial sums are
//             reduced through distributed shared memory, in rank order)
//   CTA     = 4 consumer warps that split the CTA's super-blocks between them,
//             plus one producer warp that streams the packed tiles with TMA.
// A TMA box is {144 bytes, 32 rows}: one super-block of 32 consecutive rows,
// landing in shared memory as [row][144] so that the 32 lanes' 16-byte loads
// of one super-block hit distinct banks.
//
// Per-weight arithmetic (the unpack happens in registers):
//   A 4-bit quant q left in place inside its 32-bit word at bit 4p (p = 0..3)
//   is, read as an fp32 bit pattern, the subnormal q * 2^(4p-149); the fp32
//   FMA handles subnormal operands at full rate without flushing. Each
//   activation is pre-scaled once per (block, row of X) by 2^(E+149-4p), so
//   one mask and one FMA give q*x*2^E exactly rounded, with no int->float
//   conversion. E is chosen from the block's largest |x| so that neither the
//   scaled activations overflow nor the products leave the normal range.
//   Sub-block sums are then combined as d*sc*S - dmin*m*sum(x) and rescaled.
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

constexpr int kGemvConsumers = 4;
constexpr int kGemvThreads = 32 * (kGemvConsumers + 1);
constexpr int kGemvRows = 32;
constexpr int kGemvSubBytes = kGemvRows * kBlockBytes;               // 4608
constexpr int kGemvStageBytes = kGemvConsumers * kGemvSubBytes;      // 18432

template <int MT>
struct GemvCfg {
    static constexpr int kStages = MT >= 8 ? 2 : 3;
    static constexpr int kOffW = 0;
    static constexpr int kOffX = kOffW + kStages * kGemvStageBytes;              // x' [warp][m][256]
    static constexpr int kOffXs = kOffX + kGemvConsumers * MT * 256 * 4;          // sums [warp][m][8]
    static constexpr int kOffRed = kOffXs + kGemvConsumers * MT * 8 * 4;          // [warp][m][32]
    static constexpr int kOffPart = kOffRed + kGemvConsumers * MT * 32 * 4;       // [m][32]
    static constexpr int kOffBar = kOffPart + MT * 32 * 4;                        // full, empty
    static constexpr int kSmem = kOffBar + 2 * kStages * 8 + 128;  // + alignment slack
};

// Loads 8 consecutive activations of row m as fp32 (zeros past M).
template <bool XB>
__device__ __forceinline__ void load_x8(const void* X, int m, int M, int64_t K, int64_t k,
                                        float (&v)[8]) {
    if (m >= M) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
        return;
    }
    if constexpr (XB) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(
            static_cast<const uint16_t*>(X) + static_cast<int64_t>(m) * K + k));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(X) +
                                                          static_cast<int64_t>(m) * K + k);
        const float4 a = __ldg(p), b = __ldg(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// Unbiased exponent of the largest |x| of the block, clamped to [-20, 127].
__device__ __forceinline__ int block_exponent(float amax) {
    int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
    return e < -20 ? -20 : (e > 127 ? 127 : e);
}

template <int MT, bool XB>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const __grid_constant__ CUtensorMap tmapW,
                                                            const void* __restrict__ X, int M, int N,
                                                            int K, float* __restrict__ Y,
                                                            int kb_per_split, unsigned int* err) {
    using Cfg = GemvCfg<MT>;
    constexpr int NS = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = K / kBlockWeights;
    const int row0 = blockIdx.x * kGemvRows;
    const int kb0 = blockIdx.y * kb_per_split;
    const int kb1 = min(KB, kb0 + kb_per_split);
    const int nst = (kb1 - kb0 + kGemvConsumers - 1) / kGemvConsumers;  // stages for this CTA

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + Cfg::kOffBar;
    const uint32_t bar_empty = bar_full + NS * 8;
    float* xs_all = reinterpret_cast<float*>(smem + Cfg::kOffX);
    float* xsum_all = reinterpret_cast<float*>(smem + Cfg::kOffXs);
    float* red = reinterpret_cast<float*>(smem + Cfg::kOffRed);
    float* part = reinterpret_cast<float*>(smem + Cfg::kOffPart);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kGemvConsumers);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kGemvConsumers) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            tma_prefetch_desc(&tmapW);
            const uint64_t pol = policy_evict_first();
            for (int st = 0; st < nst; ++st) {
                const int s = st % NS;
                const uint32_t ph = (st / NS) & 1;
                if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, err)) break;
                const int b0 = kb0 + st * kGemvConsumers;
                const int nb = min(kGemvConsumers, kb1 - b0);
                mbar_arrive_expect_tx(bar_full + 8 * s, nb * kGemvSubBytes);
                for (int i = 0; i < nb; ++i)
                    tma_load_2d_hint(sbase + Cfg::kOffW + s * kGemvStageBytes + i * kGemvSubBytes,
                                     &tmapW, (b0 + i) * kBlockBytes, row0, bar_full + 8 * s, pol);
            }
        }
        __syncwarp();
    } else {
        // --------------------------------------------------- consumers ---
        float y[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) y[m] = 0.f;
        float* xs = xs_all + warp * MT * 256;
        float* xsum = xsum_all + warp * MT * 8;
        bool ok = true;

        for (int st = 0; st < nst && ok; ++st) {
            const int s = st % NS;
            const uint32_t ph = (st / NS) & 1;
            const int b = kb0 + st * kGemvConsumers + warp;
            const bool has = b < kb1;
            float inv_a[MT], inv_b[MT];  // 2^-E as two factors
            if (has) {
                // stage this block's activations: lane owns k = 8*lane .. 8*lane+7
                const int64_t kx = static_cast<int64_t>(b) * kBlockWeights + 8 * lane;
                const int hsel = (lane >> 2) & 1;  // weight is a high-nibble one (k % 64 >= 32)
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float v[8];
                    load_x8<XB>(X, m, M, K, kx, v);
                    float amax = 0.f, sum = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        amax = fmaxf(amax, fabsf(v[i]));
                        sum += v[i];
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, o));
                    sum += __shfl_xor_sync(~0u, sum, 1);
                    sum += __shfl_xor_sync(~0u, sum, 2);
                    const int e = block_exponent(amax);
                    // E = -23 - e; x' = x * 2^(E + 149 - 4p) = x * 2^(126 - e - 4p)
                    const int t0 = 126 - e - 4 * hsel;  // p = 2*(k&1) + hsel; even k: p = hsel
                    const int t1 = t0 - 8;              // odd k: p = 2 + hsel
                    const float f0a = exp2i(t0 >> 1), f0b = exp2i(t0 - (t0 >> 1));
                    const float f1a = exp2i(t1 >> 1), f1b = exp2i(t1 - (t1 >> 1));
                    float4 o0, o1;
                    o0.x = (v[0] * f0a) * f0b; o0.y = (v[1] * f1a) * f1b;
                    o0.z = (v[2] * f0a) * f0b; o0.w = (v[3] * f1a) * f1b;
                    o1.x = (v[4] * f0a) * f0b; o1.y = (v[5] * f1a) * f1b;
                    o1.z = (v[6] * f0a) * f0b; o1.w = (v[7] * f1a) * f1b;
                    float4* dst = reinterpret_cast<float4*>(xs + m * 256 + 8 * lane);
                    dst[0] = o0;
                    dst[1] = o1;
                    // sub-block sum scaled by 2^E, E = -23 - e (two factors)
                    const int E = -23 - e;
                    if ((lane & 3) == 0)
                        xsum[m * 8 + (lane >> 2)] = (sum * exp2i(E >> 1)) * exp2i(E - (E >> 1));
                    const int ie = 23 + e;  // 2^-E
                    inv_a[m] = exp2i(ie >> 1);
                    inv_b[m] = exp2i(ie - (ie >> 1));
                }
                __syncwarp();
            }
            if (!mbar_wait(bar_full + 8 * s, ph, err)) ok = false;
            if (has && ok) {
                const uint8_t* P = smem + Cfg::kOffW + s * kGemvStageBytes + warp * kGemvSubBytes +
                                   lane * kBlockBytes;
                const uint4 h = *reinterpret_cast<const uint4*>(P);
                const ScaleBytes sb = decode_scales(h.y, h.z, h.w);
                const float d = half_lo(h.x), dmin = half_hi(h.x);
                float d1[8], mm[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    d1[j] = d * static_cast<float>(byte_of(sb.sc_lo, j));
                    mm[j] = dmin * static_cast<float>(byte_of(sb.m_lo, j));
                    d1[j + 4] = d * static_cast<float>(byte_of(sb.sc_hi, j));
                    mm[j + 4] = dmin * static_cast<float>(byte_of(sb.m_hi, j));
                }
                float acc[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 qa = *reinterpret_cast<const uint4*>(P + 16 + 32 * c);
                    const uint4 qb = *reinterpret_cast<const uint4*>(P + 32 + 32 * c);
                    const uint32_t wq[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                    float slo[MT], shi[MT], slo2[MT], shi2[MT];
#pragma unroll
                    for (int m = 0; m < MT; ++m) slo[m] = shi[m] = slo2[m] = shi2[m] = 0.f;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t wd = wq[u], wh = wd >> 16;
                        // low nibbles: weights 64c+4u+{0,1,2,3}; high: +32
                        const float qA = __uint_as_float(wd & 0x000Fu);
                        const float qC = __uint_as_float(wd & 0x0F00u);
                        const float qE = __uint_as_float(wh & 0x000Fu);
                        const float qG = __uint_as_float(wh & 0x0F00u);
                        const float qB = __uint_as_float(wd & 0x00F0u);
                        const float qD = __uint_as_float(wd & 0xF000u);
                        const float qF = __uint_as_float(wh & 0x00F0u);
                        const float qH = __uint_as_float(wh & 0xF000u);
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            const float4 xl = *reinterpret_cast<const float4*>(xs + m * 256 + 64 * c + 4 * u);
                            const float4 xh =
                                *reinterpret_cast<const float4*>(xs + m * 256 + 64 * c + 32 + 4 * u);
                            slo[m] = fmaf(qA, xl.x, slo[m]);
                            slo2[m] = fmaf(qC, xl.y, slo2[m]);
                            slo[m] = fmaf(qE, xl.z, slo[m]);
                            slo2[m] = fmaf(qG, xl.w, slo2[m]);
                            shi[m] = fmaf(qB, xh.x, shi[m]);
                            shi2[m] = fmaf(qD, xh.y, shi2[m]);
                            shi[m] = fmaf(qF, xh.z, shi[m]);
                            shi2[m] = fmaf(qH, xh.w, shi2[m]);
                        }
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const float* xsm = xsum + m * 8;
                        float a = acc[m];
                        a = fmaf(d1[2 * c], slo[m] + slo2[m], a);
                        a = fmaf(-mm[2 * c], xsm[2 * c], a);
                        a = fmaf(d1[2 * c + 1], shi[m] + shi2[m], a);
                        a = fmaf(-mm[2 * c + 1], xsm[2 * c + 1], a);
                        acc[m] = a;
                    }
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) y[m] += (acc[m] * inv_a[m]) * inv_b[m];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) red[(warp * MT + m) * 32 + lane] = y[m];
    }
    __syncthreads();

    // fixed-order reduction over the consumer warps
    for (int idx = threadIdx.x; idx < MT * 32; idx += kGemvThreads) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kGemvConsumers; ++w) s += red[w * MT * 32 + idx];
        part[idx] = s;
    }
    if (gridDim.y == 1) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < MT * 32; idx += kGemvThreads) {
            const int m = idx >> 5, r = row0 + (idx & 31);
            if (m < M && r < N) Y[static_cast<int64_t>(m) * N + r] = part[idx];
        }
    } else {
        // cluster along y: rank 0 sums the partials of all ranks in rank order
        cluster_sync_all();
        if (cluster_ctarank() == 0) {
            const uint32_t paddr = smem_u32(part);
            for (int idx = threadIdx.x; idx < MT * 32; idx += kGemvThreads) {
                const int m = idx >> 5, r = row0 + (idx & 31);
                float s = 0.f;
                for (uint32_t rk = 0; rk < gridDim.y; ++rk)
                    s += ld_shared_cluster_f32(map_shared_rank(paddr + 4 * idx, rk));
                if (m < M && r < N) Y[static_cast<int64_t>(m) * N + r] = s;
            }
        }
        cluster_sync_all();
    }
}

// ------------------------------------------------------------------ host ---

template <int MT, bool XB>
static cudaError_t set_attr() {
    return cudaFuncSetAttribute(gemv_kernel<MT, XB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemvCfg<MT>::kSmem);
}

cudaError_t gemv_setup() {
    cudaError_t e = cudaSuccess;
    cudaError_t r;
#define Q4K_SET(MT)                                          \
    if ((r = set_attr<MT, false>()) != cudaSuccess) e = r;   \
    if ((r = set_attr<MT, true>()) != cudaSuccess) e = r;
    Q4K_SET(1) Q4K_SET(2) Q4K_SET(4) Q4K_SET(8) Q4K_SET(16)
#undef Q4K_SET
    return e;
}

template <int MT, bool XB>
static cudaError_t launch_mt(const CUtensorMap& tmapW, const void* X, int M, int N, int K, float* Y,
                             cudaStream_t stream, const DeviceInfo& dev) {
    const int KB = K / kBlockWeights;
    const int rg = (N + kGemvRows - 1) / kGemvRows;
    const int target = 2 * dev.num_sms;
    int ks = (target + rg - 1) / rg;
    ks = ks < 1 ? 1 : ks;
    ks = ks > 8 ? 8 : ks;
    ks = ks > KB ? KB : ks;
    const int kb_per = (KB + ks - 1) / ks;
    ks = (KB + kb_per - 1) / kb_per;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rg, ks, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = GemvCfg<MT>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = ks;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<MT, XB>, tmapW, X, M, N, K, Y, kb_per, dev.err);
}

cudaError_t launch_gemv(const CUtensorMap& tmapW, const void* X, bool x_bf16, int M, int N, int K,
                        float* Y, cudaStream_t stream, const DeviceInfo& dev) {
    const int mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16;
#define Q4K_CASE(MT)                                                                     \
    case MT:                                                                             \
        return x_bf16 ? launch_mt<MT, true>(tmapW, X, M, N, K, Y, stream, dev)           \
                      : launch_mt<MT, false>(tmapW, X, M, N, K, Y, stream, dev);
    switch (mt) {
        Q4K_CASE(1) Q4K_CASE(2) Q4K_CASE(4) Q4K_CASE(8) Q4K_CASE(16)
    }
#undef Q4K_CASE
    return cudaErrorInvalidValue;
}

}  // namespace q4k
