// q4k_gemm.cu -- K3: packed Q4_K x bf16 GEMM on the 5th-generation tensor
// cores, for chunked prefill (M = 17 .. thousands of token rows).
//
// The rlx prefill path builds one Op::DequantMatMul per linear layer over a
// block of tokens ("rlx-llama32" page, section "Packed GGUF"; blocks of up to
// 32 tokens in the nx_f32_llm_run_v3 listing's bounded-chunk prefill), so the
// packed weights are read once per block rather than once per token. Here the
// product is computed as Y^T = W * X^T:
//   MMA A operand = 128 dequantised weight rows (MMA M = 128), K-major bf16
//   MMA B operand = BN token rows of X (MMA N = BN <= 256), K-major bf16
//   accumulator    = 128 TMEM lanes x BN fp32 columns
// so each dequantised weight tile is reused across all BN tokens of the tile.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: packed W super-block tiles {144 B, 128 rows}
//               and X tiles {64 k, BN rows} (128-byte swizzle)
//   warp 1      TMEM allocator and MMA issuer (one elected thread)
//   warps 2..5  dequantisers (thread t <-> weight row t of the tile): read the
//               packed block from shared memory, write 64 bf16 weights per
//               k-step into the swizzled A tile; then the epilogue (TMEM ->
//               registers -> Y, 128-byte coalesced stores per token column).
// All pipeline waits are bounded (see mbar_wait).
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

constexpr int kGemmBM = 128;
constexpr int kGemmKStep = 64;                       // bf16 k per A/B stage (one 128-byte row)
constexpr int kGemmThreads = 192;
constexpr int kGemmWStages = 2;
constexpr int kGemmWStageBytes = kGemmBM * kBlockBytes;   // 18432
constexpr int kGemmAStageBytes = kGemmBM * 128;           // 16384

template <int BN>
struct GemmCfg {
    static constexpr int kABStages = BN == 256 ? 3 : 4;
    static constexpr int kBStageBytes = BN * 128;
    static constexpr int kOffA = 0;                                            // 1024-aligned
    static constexpr int kOffB = kOffA + kABStages * kGemmAStageBytes;         // 1024-aligned
    static constexpr int kOffW = kOffB + kABStages * kBStageBytes;
    static constexpr int kOffBar = kOffW + kGemmWStages * kGemmWStageBytes;
    // barriers: w_full[2], w_empty[2], a_full[S], b_full[S], ab_empty[S], acc_full, tmem slot
    static constexpr int kNumBars = 2 * kGemmWStages + 3 * kABStages + 1;
    static constexpr int kOffTmem = kOffBar + kNumBars * 8;
    static constexpr int kSmem = kOffTmem + 16 + 1024;   // + alignment slack
    static constexpr uint32_t kTmemCols = BN < 32 ? 32 : BN;
};

// Converts 8 low (or high) nibbles of two qs words into 8 bf16 weights
// w = d1*q - m1 (fp32 FMA, then round-to-nearest-even to bf16).
__device__ __forceinline__ uint4 dequant8(uint32_t w0, uint32_t w1, int shift, float d1, float nm1) {
    const uint32_t a = (w0 >> shift) & 0x0F0F0F0Fu;
    const uint32_t b = (w1 >> shift) & 0x0F0F0F0Fu;
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // 0x4B0000qq is 2^23 + q exactly; subtracting 2^23 leaves q
        f[i] = __uint_as_float(__byte_perm(a, 0x4B000000u, 0x7440u | i)) - 8388608.f;
        f[4 + i] = __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7440u | i)) - 8388608.f;
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 p =
            __floats2bfloat162_rn(fmaf(f[2 * i], d1, nm1), fmaf(f[2 * i + 1], d1, nm1));
        o[i] = *reinterpret_cast<const uint32_t*>(&p);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmapW, const __grid_constant__ CUtensorMap tmapX,
                int M, int N, int K, float* __restrict__ Y, int pdl_flags, unsigned int* err) {
    using Cfg = GemmCfg<BN>;
    constexpr int S = Cfg::kABStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kGemmBM;
    const int m0 = blockIdx.y * BN;
    const int KB = K / kBlockWeights;
    const int nks = K / kGemmKStep;

    const uint32_t bw_full = sbase + Cfg::kOffBar;
    const uint32_t bw_empty = bw_full + 8 * kGemmWStages;
    const uint32_t ba_full = bw_empty + 8 * kGemmWStages;
    const uint32_t bb_full = ba_full + 8 * S;
    const uint32_t bab_empty = bb_full + 8 * S;
    const uint32_t bacc = bab_empty + 8 * S;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffTmem);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kGemmWStages; ++i) {
            mbar_init(bw_full + 8 * i, 1);
            mbar_init(bw_empty + 8 * i, 128);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(ba_full + 8 * i, 128);
            mbar_init(bb_full + 8 * i, 1);
            mbar_init(bab_empty + 8 * i, 1);
        }
        mbar_init(bacc, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) pdl_launch_dependents();
    // Every warp except the producer waits for the preceding grid here; the
    // producer waits before its first activation load (and, unless weight
    // prefetch is allowed, before its first weight load).
    if (warp != 0) pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            tma_prefetch_desc(&tmapW);
            tma_prefetch_desc(&tmapX);
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            if (pdl_flags & 1) pdl_wait();
            for (int ks = 0; ks < nks; ++ks) {
                if ((ks & 3) == 0) {
                    const int sb = ks >> 2;
                    const int ws = sb % kGemmWStages;
                    if (!mbar_wait(bw_empty + 8 * ws, ((sb / kGemmWStages) & 1) ^ 1, err)) break;
                    mbar_arrive_expect_tx(bw_full + 8 * ws, kGemmWStageBytes);
                    tma_load_2d_hint(sbase + Cfg::kOffW + ws * kGemmWStageBytes, &tmapW,
                                     sb * kBlockBytes, n0, bw_full + 8 * ws, pol_w);
                }
                const int s = ks % S;
                if (!mbar_wait(bab_empty + 8 * s, ((ks / S) & 1) ^ 1, err)) break;
                if (ks == 0 && !(pdl_flags & 1)) pdl_wait();
                mbar_arrive_expect_tx(bb_full + 8 * s, Cfg::kBStageBytes);
                tma_load_2d_hint(sbase + Cfg::kOffB + s * Cfg::kBStageBytes, &tmapX, ks * kGemmKStep,
                                 m0, bb_full + 8 * s, pol_x);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer ---
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kGemmBM, BN);
            bool ok = true;
            for (int ks = 0; ks < nks && ok; ++ks) {
                const int s = ks % S;
                const uint32_t ph = (ks / S) & 1;
                ok = mbar_wait(ba_full + 8 * s, ph, err) && mbar_wait(bb_full + 8 * s, ph, err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a0 = sbase + Cfg::kOffA + s * kGemmAStageBytes;
                const uint32_t b0 = sbase + Cfg::kOffB + s * Cfg::kBStageBytes;
#pragma unroll
                for (int kk = 0; kk < kGemmKStep / 16; ++kk)
                    tc_mma_bf16(tmem, sw128_desc(a0 + 32 * kk), sw128_desc(b0 + 32 * kk), idesc,
                                (ks | kk) != 0);
                tc_commit(bab_empty + 8 * s);
            }
            tc_commit(bacc);
        }
        __syncwarp();
    } else {
        // ------------------------------------------ dequantisers (A) ---
        const int t = threadIdx.x - 64;  // weight row within the tile
        bool ok = true;
        for (int sb = 0; sb < KB && ok; ++sb) {
            const int ws = sb % kGemmWStages;
            if (!mbar_wait(bw_full + 8 * ws, (sb / kGemmWStages) & 1, err)) { ok = false; break; }
            const uint8_t* P = smem + Cfg::kOffW + ws * kGemmWStageBytes + t * kBlockBytes;
            const uint4 h = *reinterpret_cast<const uint4*>(P);
            const ScaleBytes scb = decode_scales(h.y, h.z, h.w);
            const float d = half_lo(h.x), dmin = half_hi(h.x);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int ks = sb * 4 + c;
                const int s = ks % S;
                if (!mbar_wait(bab_empty + 8 * s, ((ks / S) & 1) ^ 1, err)) { ok = false; break; }
                const uint32_t scw = c < 2 ? scb.sc_lo : scb.sc_hi;
                const uint32_t mw = c < 2 ? scb.m_lo : scb.m_hi;
                const int jb = (2 * c) & 3;
                const float d1l = d * static_cast<float>(byte_of(scw, jb));
                const float m1l = -(dmin * static_cast<float>(byte_of(mw, jb)));
                const float d1h = d * static_cast<float>(byte_of(scw, jb + 1));
                const float m1h = -(dmin * static_cast<float>(byte_of(mw, jb + 1)));
                const uint4 qa = *reinterpret_cast<const uint4*>(P + 16 + 32 * c);
                const uint4 qb = *reinterpret_cast<const uint4*>(P + 32 + 32 * c);
                // 16-byte chunk j of the row holds k = 8j .. 8j+7 of this 64-k step:
                //   j < 4: low nibbles of qs bytes 8j..8j+7 (sub-block 2c)
                //   j >= 4: high nibbles of qs bytes 8(j-4)..  (sub-block 2c+1)
                uint8_t* arow = smem + Cfg::kOffA + s * kGemmAStageBytes + t * 128;
                const int sw = t & 7;
                const uint32_t wq[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    *reinterpret_cast<uint4*>(arow + ((j ^ sw) << 4)) =
                        dequant8(wq[2 * j], wq[2 * j + 1], 0, d1l, m1l);
                    *reinterpret_cast<uint4*>(arow + (((j + 4) ^ sw) << 4)) =
                        dequant8(wq[2 * j], wq[2 * j + 1], 4, d1h, m1h);
                }
                fence_proxy_async_smem();
                mbar_arrive(ba_full + 8 * s);
            }
            mbar_arrive(bw_empty + 8 * ws);
        }

        // ------------------------------------------------- epilogue ---
        if (ok && mbar_wait(bacc, 0, err)) {
            tc_fence_after();
            const int q = warp & 3;  // TMEM lane quadrant this warp may access
            const int n = n0 + 32 * q + lane;
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + 32 * cc, v);
                tmem_ld_wait();
                if (n < N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int m = m0 + 32 * cc + j;
                        if (m < M) Y[static_cast<int64_t>(m) * N + n] = __uint_as_float(v[j]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

// ------------------------------------------------------------------ host ---

int gemm_pick_bn(int M) { return M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256; }

template <int BN>
static cudaError_t set_attr() {
    return cudaFuncSetAttribute(gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemmCfg<BN>::kSmem);
}

cudaError_t gemm_setup() {
    cudaError_t e = cudaSuccess, r;
    if ((r = set_attr<32>()) != cudaSuccess) e = r;
    if ((r = set_attr<64>()) != cudaSuccess) e = r;
    if ((r = set_attr<128>()) != cudaSuccess) e = r;
    if ((r = set_attr<256>()) != cudaSuccess) e = r;
    return e;
}

template <int BN>
static cudaError_t launch_bn(const CUtensorMap& tmapW, const CUtensorMap& tmapX, int M, int N, int K,
                             float* Y, cudaStream_t stream, unsigned int* err, int pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + kGemmBM - 1) / kGemmBM, (M + BN - 1) / BN, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = GemmCfg<BN>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const int pdl_flags = (pdl == 2) ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<BN>, tmapW, tmapX, M, N, K, Y, pdl_flags, err);
}

cudaError_t launch_gemm(const CUtensorMap& tmapW, const CUtensorMap& tmapX, int M, int N, int K,
                        float* Y, int BN, cudaStream_t stream, const DeviceInfo& dev, int pdl) {
    switch (BN) {
        case 32: return launch_bn<32>(tmapW, tmapX, M, N, K, Y, stream, dev.err, pdl);
        case 64: return launch_bn<64>(tmapW, tmapX, M, N, K, Y, stream, dev.err, pdl);
        case 128: return launch_bn<128>(tmapW, tmapX, M, N, K, Y, stream, dev.err, pdl);
        case 256: return launch_bn<256>(tmapW, tmapX, M, N, K, Y, stream, dev.err, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace q4k
