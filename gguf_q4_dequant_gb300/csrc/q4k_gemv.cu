// q4k_gemv.cu -- K2: split-K GEMV for the packed Q4_K decode step (M = 1..16).
//
// Decode reads every packed weight matrix once per token (the per-token weight
// sweep of the rlx-llama32 page, section "Decode"), so this kernel is bound by
// HBM bandwidth at M = 1 and by fp32 issue rate as M grows.
//
// Work decomposition
//   tile      = 128 consecutive rows of W; one TMA box {144 bytes, 128 rows}
//               brings one super-block of every row of the tile into shared
//               memory as [row][144] (a stage, 18 KB).
//   K-slice   = a contiguous range of super-blocks. When there are fewer tiles
//               than CTA slots, the K range is split across a thread-block
//               cluster (one K-slice per CTA); ranks 1..C-1 send their partial
//               sums into rank 0's shared memory with st.async, which counts the
//               bytes on rank 0's mbarrier, and rank 0 adds them in rank order
//               (deterministic).
//   group     = up to 8 weight matrices that share K and the activations (q, k
//               and v of a layer; gate and up) are one launch: their tiles are
//               numbered consecutively and each has its own TMA map and output.
//   CTA       = 4 consumer warps (warp w owns rows 32w..32w+31 of the tile,
//               one lane per row and the whole super-block of that row per
//               stage, so the per-stage and per-super-block set-up -- barrier
//               waits, scale unpacking -- is paid once per 256 weights; for
//               M >= 8 two such groups, each taking half of the activation
//               rows), 1 TMA producer warp and 1 activation warp. CTAs are
//               persistent over tiles, so the stage ring streams continuously.
//
// Per-weight arithmetic (the unpack happens in registers):
//   A 4-bit quant q left in place inside its 32-bit word at bit 4p (p = 0..4)
//   is, read as an fp32 bit pattern, the subnormal q * 2^(4p-149); the fp32
//   FMA handles subnormal operands at full rate without flushing. Two
//   neighbouring qs words form one 64-bit register pair, so a 64-bit mask
//   yields the same nibble of both words as an fp32 pair for the paired FMA
//   (fma.rn.f32x2); the top three nibbles of each word are first brought down
//   by one 64-bit shift by 12. The one-row fp32 kernel of launches that do not
//   split K instead moves bits 20..31 of each word down (the subnormal u*2^-149 of
//   the 12-bit field u) and splits u into its three codes with products by
//   2^-8 and 2^-4 rounded toward zero -- floor on the subnormal grid -- and
//   exact FMAs: work moved from the integer pipe (logic and shifts issue at
//   half the FMA rate) to the FMA pipe. Each activation is pre-scaled once per
//   (super-block, row of X) by 2^(E+149-4p) by the activation warp and stored
//   in the order the pairs consume them, so a mask and half a paired FMA per
//   weight give q*x*2^E with a single rounding and no int->float conversion.
//   E is chosen from the block's largest |x| so that neither the scaled
//   activations overflow nor the products leave the normal range. Sub-block
//   sums are then combined per super-block as d*sum(sc*S) - dmin*sum(m*sum(x))
//   and scaled back by 2^-E.
//
// Epilogue: one store per lane and activation row, or, for the fused greedy
// pick (q4k_matmul_argmax), a warp-wide maximum of 64-bit (logit, row) keys
// combined into the caller's output with atomicMax -- no Y is written.
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

constexpr int kGemvTileRows = 128;
constexpr int kGemvConsumers = 4;  // consumer warps: one lane per row of the tile
constexpr int kGemvStageBytes = kGemvTileRows * kBlockBytes;  // 18432

template <int MT>
struct GemvCfg {
    // M >= 8: two groups of consumer warps on the same rows and stages, each
    // taking half of the activation rows (kML of them), so that a lane's
    // accumulators fit and twice as many warps share the FMA work
    static constexpr int kMGroups = MT >= 8 ? 2 : 1;
    static constexpr int kML = MT / kMGroups;
    // M <= 2: kSGroups groups of consumer warps take alternate stages of the
    // same tile (more warps to hide latency); their partial sums are added at
    // the end of the tile, group 0 + group 1 (deterministic)
    static constexpr int kSGroups = MT <= 2 ? 2 : 1;
    static constexpr int kStageConsumers = kGemvConsumers * kMGroups;  // warps reading a stage
    static constexpr int kConsumers = kStageConsumers * kSGroups;
    static constexpr int kProducerWarp = kConsumers;
    static constexpr int kStagerWarp = kConsumers + 1;
    static constexpr int kThreads = 32 * (kConsumers + 2);
    // registers: two resident CTAs per SM for small M (measured: more registers
    // per thread buy more overlap than a third CTA would); M >= 8 takes ~145-165
    // registers a thread at 320 threads, one CTA per SM
    static constexpr int kMinBlocks = MT >= 8 ? 1 : 2;
    static constexpr int kStages = 4;
    static constexpr int kOffW = 0;
    static constexpr int kOffX = kOffW + kStages * kGemvStageBytes;     // x' [stage][m][256]
    static constexpr int kOffXs = kOffX + kStages * MT * 256 * 4;        // sums [stage][m][8]
    static constexpr int kOffInv = kOffXs + kStages * MT * 8 * 4;        // 2^-E [stage][m][2]
    // K-split across a cluster of at most kMaxSplit CTAs (16 is a non-portable
    // cluster size, used only where its reduction slots stay small)
    static constexpr int kMaxSplit = MT <= 2 ? 16 : 8;
    static constexpr int kOffRed = kOffInv + kStages * MT * 2 * 4;       // ranks 1..: [kMaxSplit-1][m][128]
    // stage groups 1..: their partial sums of a tile, [kSGroups-1][m][128]
    static constexpr int kOffComb = kOffRed + (kMaxSplit - 1) * MT * kGemvTileRows * 4;
    // wfull[S] (the stage's weight bytes), xfull[S] (its activations), empty[S],
    // red, comb_full, comb_empty
    static constexpr int kOffBar = kOffComb + (kSGroups - 1) * MT * kGemvTileRows * 4;
    static constexpr int kSmem = kOffBar + (3 * kStages + 3) * 8 + 128;  // + alignment slack
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

// Pre-scales one row of activations for the subnormal-quant products and
// stores it in consumption order. Lane l holds x for k = 8l .. 8l+7 of the
// super-block: chunk c = l/8, high-nibble half h = (l/4)%2, word pair v = l%4,
// element i = 4*up + j (up: which word of the pair, j: byte in the word).
// The consumer reads, per word pair, 16 floats ordered
//   [A A C C E E G G | B B D D F F H H]   (each letter: word u, word u+1)
// where A,C,E,G are the low nibbles of bytes 0..3 and B,D,F,H the high ones,
// so this lane's 8 values go to the 8 floats at c*64 + v*16 + 8h, slot 2j+up.
// The consumer reads the codes as q*2^(4p-149): p is the nibble's position in
// its word for the five codes in bits 0..19 (A0 B1 C2 D3 E4); F, G and H are
// brought down by 12 bits first (F2 G3 H4), or, with SPLIT, split out of bits
// 20..31 on the FMA pipe (F0 G0 H0).
// Also stores the sub-block sums scaled by 2^E and 2^-E (as two factors).
template <bool SPLIT>
__device__ __forceinline__ void scale_activations(const float (&v)[8], int lane, float* xs,
                                                  float* xsum, float* inv) {
    const int h = (lane >> 2) & 1;
    uint32_t amax = 0;  // |x| bit patterns order like the values
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        amax = max(amax, __float_as_uint(v[i]) & 0x7FFFFFFFu);
        sum += v[i];
    }
    amax = __reduce_max_sync(~0u, amax);
    sum += __shfl_xor_sync(~0u, sum, 1);
    sum += __shfl_xor_sync(~0u, sum, 2);
    const int e = block_exponent(__uint_as_float(amax));
    // E = -23 - e; x' = x * 2^(E + 149 - 4p) = x * 2^(126 - e - 4p)
    const int base = 126 - e;
    float o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // nibble position of byte j's low (h = 0) or high (h = 1) nibble
        const int p = SPLIT ? (h ? ((0x0031 >> (4 * j)) & 0xF) : ((0x0420 >> (4 * j)) & 0xF))
                            : (h ? ((0x4231 >> (4 * j)) & 0xF) : ((0x3420 >> (4 * j)) & 0xF));
        const int t = base - 4 * p;
        const float fa = exp2i(t >> 1), fb = exp2i(t - (t >> 1));
        o[2 * j] = (v[j] * fa) * fb;          // up = 0: word u
        o[2 * j + 1] = (v[4 + j] * fa) * fb;  // up = 1: word u+1
    }
    float4* dst = reinterpret_cast<float4*>(xs + (lane >> 3) * 64 + (lane & 3) * 16 + 8 * h);
    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    const int E = -23 - e;
    if ((lane & 3) == 0) xsum[lane >> 2] = (sum * exp2i(E >> 1)) * exp2i(E - (E >> 1));
    if (lane == 0) {
        const int ie = 23 + e;
        inv[0] = exp2i(ie >> 1);
        inv[1] = exp2i(ie - (ie >> 1));
    }
}

// Rows kept in registers across one stage by the activation warp (the next
// stage's loads are in flight while the current stage is written): all of
// them for small M; for M >= 8 the rows of a stage are loaded in batches of 8
// whose loads are in flight together.
template <int MT>
struct XPrefetch {
    static constexpr int kRows = MT <= 4 ? MT : 0;
};
// fp32 pairs (both halves equal) for splitting a 12-bit field of codes:
// 2^-8, 2^-4 and -256, -16.
constexpr uint64_t kPairP2m8 = 0x3B8000003B800000ull;
constexpr uint64_t kPairP2m4 = 0x3D8000003D800000ull;
constexpr uint64_t kPairM256 = 0xC3800000C3800000ull;
constexpr uint64_t kPairM16 = 0xC1800000C1800000ull;

// a * b elementwise on fp32 pairs, rounded toward zero (subnormals kept).
__device__ __forceinline__ uint64_t mul2_rz(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Bits 20..31 of each 32-bit half of p, moved down (zero-filled).
__device__ __forceinline__ uint64_t top12_pair(uint64_t p) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r)
        : "r"(static_cast<uint32_t>(p) >> 20), "r"(static_cast<uint32_t>(p >> 32) >> 20));
    return r;
}

// One consumer lane: the contribution of one super-block of its row, scaled by
// 2^E (acc[m] for each activation row m). SPLIT selects how the codes in bits
// 20..31 of each word are unpacked (scale_activations<SPLIT> matches it).
template <int MT, bool SPLIT>
__device__ __forceinline__ void block_dot(const uint8_t* P, const float* xs, const float* xsum,
                                          float (&acc)[MT]) {
    const uint4 h = *reinterpret_cast<const uint4*>(P);
    const ScaleBytes sb = decode_scales(h.y, h.z, h.w);
    const float d = half_lo(h.x), dmin = half_hi(h.x);
    // d and dmin are applied once per super-block, after the sums over its
    // sub-blocks: d * sum_j sc_j*S_j - dmin * sum_j m_j*sum(x)_j
    uint64_t scp[8];  // (sc_j, sc_j) pairs
    float mf[8];      // m_j
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t scw = j < 4 ? sb.sc_lo : sb.sc_hi;
        const uint32_t mw = j < 4 ? sb.m_lo : sb.m_hi;
        const float a = byte_to_float(scw, j & 3);
        scp[j] = pack2(a, a);
        mf[j] = byte_to_float(mw, j & 3);
    }
    uint64_t tot[MT];  // sum over sub-blocks of sc_j*S_j, as a pair
#pragma unroll
    for (int m = 0; m < MT; ++m) tot[m] = 0ull;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        // the 32 qs bytes of chunk c as four word pairs (u, u+1)
        const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(P + 16 + 32 * c);
        const ulonglong2 qb = *reinterpret_cast<const ulonglong2*>(P + 32 + 32 * c);
        const uint64_t wp[4] = {qa.x, qa.y, qb.x, qb.y};
        // fp32 pair accumulators: two independent chains per nibble half for
        // small M; one for M >= 8, where the rows already give enough
        // independent FMAs and the registers are needed
        constexpr int NA = MT < 8 ? 2 : 1;
        uint64_t lo[MT][NA], hi[MT][NA];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int a = 0; a < NA; ++a) lo[m][a] = hi[m][a] = 0ull;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint64_t Pw = wp[v];
            // the five codes in bits 0..19 of each word, masked in place: the
            // fp32 bit pattern is the subnormal q*2^(4p-149)
            const uint64_t qA = Pw & 0x0000000F0000000Full;  // byte 0 low   p0
            const uint64_t qB = Pw & 0x000000F0000000F0ull;  // byte 0 high  p1
            const uint64_t qC = Pw & 0x00000F0000000F00ull;  // byte 1 low   p2
            const uint64_t qD = Pw & 0x0000F0000000F000ull;  // byte 1 high  p3
            const uint64_t qE = Pw & 0x000F0000000F0000ull;  // byte 2 low   p4
            uint64_t qF, qG, qH;
            if constexpr (SPLIT) {
                // bits 20..31 of each word moved down, u = F + 16*G + 256*H:
                // the subnormal u*2^-149. A product with 2^-8 rounded toward zero
                // lands on floor(u/256)*2^-149 (the subnormal grid is 2^-149) and
                // the FMA that takes it back off is exact, so two such steps give
                // F, G and H as q*2^-149: four FMA-pipe operations where the
                // masks below take five integer ones
                const uint64_t T = top12_pair(Pw);
                qH = mul2_rz(T, kPairP2m8);               // byte 3 high
                const uint64_t t = fma2(qH, kPairM256, T);  // F + 16*G
                qG = mul2_rz(t, kPairP2m4);               // byte 3 low
                qF = fma2(qG, kPairM16, t);               // byte 2 high
            } else {
                const uint64_t Sw = Pw >> 12;  // bits 20..31 of each word brought down to 8..19
                qF = Sw & 0x00000F0000000F00ull;  // byte 2 high  p2
                qG = Sw & 0x0000F0000000F000ull;  // byte 3 low   p3
                qH = Sw & 0x000F0000000F0000ull;  // byte 3 high  p4
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const ulonglong2* xp = reinterpret_cast<const ulonglong2*>(xs + m * 256 + 64 * c + 16 * v);
                const ulonglong2 x0 = xp[0], x1 = xp[1], x2 = xp[2], x3 = xp[3];
                lo[m][0] = fma2(qA, x0.x, lo[m][0]);
                lo[m][NA - 1] = fma2(qC, x0.y, lo[m][NA - 1]);
                lo[m][0] = fma2(qE, x1.x, lo[m][0]);
                lo[m][NA - 1] = fma2(qG, x1.y, lo[m][NA - 1]);
                hi[m][0] = fma2(qB, x2.x, hi[m][0]);
                hi[m][NA - 1] = fma2(qD, x2.y, hi[m][NA - 1]);
                hi[m][0] = fma2(qF, x3.x, hi[m][0]);
                hi[m][NA - 1] = fma2(qH, x3.y, hi[m][NA - 1]);
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const uint64_t L = NA == 2 ? add2(lo[m][0], lo[m][NA - 1]) : lo[m][0];
            const uint64_t H = NA == 2 ? add2(hi[m][0], hi[m][NA - 1]) : hi[m][0];
            tot[m] = fma2(L, scp[2 * c], tot[m]);
            tot[m] = fma2(H, scp[2 * c + 1], tot[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float* xsm = xsum + m * 8;
        float mins = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) mins = fmaf(mf[j], xsm[j], mins);
        const float2 t = unpack2(tot[m]);
        acc[m] = d * (t.x + t.y) - dmin * mins;
    }
}

// Grid: gridDim.x = (number of clusters) * C; a cluster of C CTAs along x
// shares tiles and splits K into C slices of kb_per super-blocks. With C > 1
// every cluster owns exactly one tile. amax == nullptr: Y_i is written; else
// (one matrix) no Y is written and each row's argmax key goes to amax[m].
template <int MT, bool XB, bool SPLIT>
__global__ void __launch_bounds__(GemvCfg<MT>::kThreads, GemvCfg<MT>::kMinBlocks)
    q4k_gemv_kernel(const __grid_constant__ WeightGroup grp, const void* __restrict__ X, int M, int K,
                int C, int kb_per, int pdl_flags, unsigned long long* amax, unsigned int* err) {
    using Cfg = GemvCfg<MT>;
    constexpr int S = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = K / kBlockWeights;
    const int rank = blockIdx.x % C;
    const int cid = blockIdx.x / C;
    const int ncl = gridDim.x / C;
    const int kb0 = rank * kb_per;
    const int nb = min(KB, kb0 + kb_per) - kb0;
    const int tiles = grp.tile_start[grp.count];
    const int nt_local = (tiles - cid + ncl - 1) / ncl;  // tiles cid, cid + ncl, ...
    const int total = nt_local * nb;                     // stages this CTA streams

    // a stage is ready when its weight bytes have landed (wfull: the producer's
    // arrival and the TMA byte count) and its activations are staged (xfull);
    // the producer can then drain its own copies without depending on others
    const uint32_t bar_wfull = sbase + Cfg::kOffBar;
    const uint32_t bar_xfull = bar_wfull + 8 * S;
    const uint32_t bar_empty = bar_xfull + 8 * S;
    float* xs_ring = reinterpret_cast<float*>(smem + Cfg::kOffX);
    float* xsum_ring = reinterpret_cast<float*>(smem + Cfg::kOffXs);
    float* inv_ring = reinterpret_cast<float*>(smem + Cfg::kOffInv);
    float* red = reinterpret_cast<float*>(smem + Cfg::kOffRed);
    const uint32_t bar_red = bar_empty + 8 * S;
    const uint32_t bar_cfull = bar_red + 8, bar_cempty = bar_red + 16;
    float* comb = reinterpret_cast<float*>(smem + Cfg::kOffComb);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_wfull + 8 * s, 1);   // producer, with the stage's bytes
            mbar_init(bar_xfull + 8 * s, 32);  // the 32 activation lanes
            mbar_init(bar_empty + 8 * s, Cfg::kStageConsumers);  // the warps of one stage group
        }
        mbar_init(bar_cfull, 32 * Cfg::kStageConsumers);   // every lane of stage group 1
        mbar_init(bar_cempty, 32 * Cfg::kStageConsumers);  // every lane of stage group 0
        // rank 0 of a cluster: the other ranks' partial sums land with
        // st.async and count their bytes; rank 0's own arrival carries the total
        mbar_init(bar_red, 1);
        fence_barrier_init();
        if (C > 1 && rank == 0)
            mbar_arrive_expect_tx(bar_red, (C - 1) * MT * kGemvTileRows * 4);
    }
    __syncthreads();
    if (C > 1) cluster_arrive_relaxed();  // the barriers above are ready for remote arrivals
    if (threadIdx.x == 0) pdl_launch_dependents();

    if (warp == Cfg::kProducerWarp) {
        // ---------------------------------------------------- TMA producer ---
        if (lane == 0) {
            for (int i = 0; i < grp.count; ++i) tma_prefetch_desc(&grp.maps[i]);
            if (pdl_flags & 1) pdl_wait();
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (; issued < total; ++issued) {
                const int st = issued;
                const int s = st % S;
                if (!mbar_wait(bar_empty + 8 * s, ((st / S) & 1) ^ 1, err)) break;
                const int t = cid + (st / nb) * ncl;
                const int mi = group_matrix(grp, t);
                const int b = kb0 + st % nb;
                mbar_arrive_expect_tx(bar_wfull + 8 * s, kGemvStageBytes);
                tma_load_2d_hint(sbase + Cfg::kOffW + s * kGemvStageBytes, &grp.maps[mi],
                                 b * kBlockBytes, (t - grp.tile_start[mi]) * kGemvTileRows,
                                 bar_wfull + 8 * s, pol);
            }
            // The CTA must not exit while a copy into its shared memory is in
            // flight. Stage st is issued only after the consumers released stage
            // st - S, which they do only after its bytes landed, so at most the
            // last S issued stages can still be in flight: wait for exactly those.
            for (int st = issued - S < 0 ? 0 : issued - S; st < issued; ++st)
                mbar_wait(bar_wfull + 8 * (st % S), (st / S) & 1, err, kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == Cfg::kStagerWarp) {
        // ------------------------------------------------ activation warp ---
        pdl_wait();
        constexpr int PF = XPrefetch<MT>::kRows;
        float nxt[PF > 0 ? PF : 1][8];
        if constexpr (PF > 0) {
            if (total > 0) {
#pragma unroll
                for (int m = 0; m < PF; ++m)
                    load_x8<XB>(X, m, M, K, static_cast<int64_t>(kb0) * kBlockWeights + 8 * lane, nxt[m]);
            }
        }
        for (int st = 0; st < total; ++st) {
            const int s = st % S;
            float* xs = xs_ring + s * MT * 256;
            float* xsum = xsum_ring + s * MT * 8;
            float* inv = inv_ring + s * MT * 2;
            if constexpr (PF > 0) {
                float cur[PF][8];
#pragma unroll
                for (int m = 0; m < PF; ++m)
#pragma unroll
                    for (int i = 0; i < 8; ++i) cur[m][i] = nxt[m][i];
                if (st + 1 < total) {
                    const int64_t kn = static_cast<int64_t>(kb0 + (st + 1) % nb) * kBlockWeights + 8 * lane;
#pragma unroll
                    for (int m = 0; m < PF; ++m) load_x8<XB>(X, m, M, K, kn, nxt[m]);
                }
                if (!mbar_wait(bar_empty + 8 * s, ((st / S) & 1) ^ 1, err)) break;
#pragma unroll
                for (int m = 0; m < PF; ++m)
                    scale_activations<SPLIT>(cur[m], lane, xs + m * 256, xsum + m * 8, inv + 2 * m);
            } else {
                // rows in batches of 8 whose loads are all in flight together
                // (the first batch before the wait for the slot)
                constexpr int B = MT < 8 ? MT : 8;
                const int64_t kx = static_cast<int64_t>(kb0 + st % nb) * kBlockWeights + 8 * lane;
                float v[B][8];
#pragma unroll
                for (int j = 0; j < B; ++j) load_x8<XB>(X, j, M, K, kx, v[j]);
                if (!mbar_wait(bar_empty + 8 * s, ((st / S) & 1) ^ 1, err)) break;
#pragma unroll
                for (int m0 = 0; m0 < MT; m0 += B) {
                    if (m0 > 0) {
#pragma unroll
                        for (int j = 0; j < B; ++j) load_x8<XB>(X, m0 + j, M, K, kx, v[j]);
                    }
#pragma unroll
                    for (int j = 0; j < B; ++j)
                        scale_activations<SPLIT>(v[j], lane, xs + (m0 + j) * 256, xsum + (m0 + j) * 8, inv + 2 * (m0 + j));
                }
            }
            __syncwarp();
            mbar_arrive(bar_xfull + 8 * s);
        }
    } else {
        // ------------------------------------------------------- consumers ---
        pdl_wait();  // before any global write
        // every CTA of the cluster has initialised its barriers (waited for here,
        // while the stage ring fills, rather than after the compute)
        if (C > 1) cluster_wait();
        constexpr int ML = Cfg::kML;
        constexpr int SG = Cfg::kSGroups;
        const int sg = warp / Cfg::kStageConsumers;                   // stage group
        const int r = 32 * (warp % kGemvConsumers) + lane;            // row within the tile
        const int m0 = ((warp / kGemvConsumers) % Cfg::kMGroups) * ML;  // first activation row
        float y[ML];
#pragma unroll
        for (int m = 0; m < ML; ++m) y[m] = 0.f;
        // After a timed-out wait the warp stops: it releases no further stage,
        // so the producer and the activation warp run out of time as well and
        // nothing more is copied into this CTA. Waits are voted warp-uniform.
        bool ok = true;
        // Stage groups 1.. hand their partial sums of tile i to group 0 through
        // `comb` (bounded waits on both sides); group 0 adds them in order.
        auto combine = [&](int i) -> bool {
            if constexpr (SG > 1) {
                if (sg != 0) {
                    if (!__all_sync(0xffffffffu, mbar_wait(bar_cempty, (i & 1) ^ 1, err))) return false;
#pragma unroll
                    for (int m = 0; m < ML; ++m) {
                        comb[(m0 + m) * kGemvTileRows + r] = y[m];
                        y[m] = 0.f;
                    }
                    mbar_arrive(bar_cfull);
                } else {
                    if (!__all_sync(0xffffffffu, mbar_wait(bar_cfull, i & 1, err))) return false;
#pragma unroll
                    for (int m = 0; m < ML; ++m) y[m] += comb[(m0 + m) * kGemvTileRows + r];
                    mbar_arrive(bar_cempty);
                }
            }
            return true;
        };
        for (int i = 0; i < nt_local && ok; ++i) {
            for (int bl = 0; bl < nb; ++bl) {
                const int st = i * nb + bl;
                if (SG > 1 && st % SG != sg) continue;
                const int s = st % S;
                const uint32_t par = (st / S) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(bar_wfull + 8 * s, par, err) &&
                                                 mbar_wait(bar_xfull + 8 * s, par, err))) {
                    ok = false;
                    break;
                }
                float acc[ML];
                const uint8_t* P = smem + Cfg::kOffW + s * kGemvStageBytes + r * kBlockBytes;
                const float* xs = xs_ring + (s * MT + m0) * 256;
                const float* xsm = xsum_ring + (s * MT + m0) * 8;
                block_dot<ML, SPLIT>(P, xs, xsm, acc);
                const float* inv = inv_ring + (s * MT + m0) * 2;
#pragma unroll
                for (int m = 0; m < ML; ++m) y[m] += (acc[m] * inv[2 * m]) * inv[2 * m + 1];
                fence_proxy_async_smem();  // generic reads of the W stage before its next TMA write
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * s);
            }
            ok = ok && combine(i);
            if (ok && C == 1 && sg == 0) {  // C > 1: one tile per CTA, reduced across the cluster below
                const int t = cid + i * ncl;
                const int mi = group_matrix(grp, t);
                const int row = (t - grp.tile_start[mi]) * kGemvTileRows + r;
                const int Nm = grp.N[mi];
                float* Ym = grp.Y[mi];
#pragma unroll
                for (int m = 0; m < ML; ++m) {
                    if (amax != nullptr)
                        argmax_combine(row < Nm ? argmax_key(y[m], row) : 0ull, lane, m0 + m < M,
                                       amax + m0 + m);
                    else if (m0 + m < M && row < Nm)
                        Ym[static_cast<int64_t>(m0 + m) * Nm + row] = y[m];
                    y[m] = 0.f;
                }
            }
        }
        if (C > 1) {
            // K-slices of this cluster's tile: ranks 1.. push into rank 0, which adds
            // in rank order. A rank that timed out pushes nothing; rank 0 always
            // waits (bounded) for the pushes before it exits, so none lands in the
            // shared memory of a CTA that has gone.
            if (sg != 0) return;
            if (rank != 0) {
                if (!ok) return;
                const uint32_t dst = map_shared_rank(smem_u32(red + (rank - 1) * MT * kGemvTileRows), 0);
                const uint32_t rbar = map_shared_rank(bar_red, 0);
#pragma unroll
                for (int m = 0; m < ML; ++m) st_async_f32(dst + 4 * ((m0 + m) * kGemvTileRows + r), y[m], rbar);
            } else if (__all_sync(0xffffffffu, mbar_wait(bar_red, 0, err)) && ok) {  // warp-uniform (argmax shuffles)
                const int mi = group_matrix(grp, cid);
                const int row = (cid - grp.tile_start[mi]) * kGemvTileRows + r;
                const int Nm = grp.N[mi];
                float* Ym = grp.Y[mi];
#pragma unroll
                for (int m = 0; m < ML; ++m) {
                    float v = y[m];
                    for (int q = 1; q < C; ++q) v += red[(q - 1) * MT * kGemvTileRows + (m0 + m) * kGemvTileRows + r];
                    if (amax != nullptr)
                        argmax_combine(row < Nm ? argmax_key(v, row) : 0ull, lane, m0 + m < M,
                                       amax + m0 + m);
                    else if (m0 + m < M && row < Nm)
                        Ym[static_cast<int64_t>(m0 + m) * Nm + row] = v;
                }
            }
            return;
        }
    }
    if (C > 1) cluster_wait();  // every thread that arrived also waits

}

// ------------------------------------------------------------------ host ---

template <int MT, bool XB>
static cudaError_t set_attr(DeviceInfo& dev, int slot) {
    const auto kern = q4k_gemv_kernel<MT, XB, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GemvCfg<MT>::kSmem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, GemvCfg<MT>::kThreads, GemvCfg<MT>::kSmem);
    if (e != cudaSuccess) return e;
    if constexpr (MT == 1 && !XB) {
        // the variant that unpacks part of the codes on the FMA pipe, for
        // launches that do not split K (it runs without clusters); the CTA
        // slots of the plan are the fewer of the two kernels'
        const auto ks = q4k_gemv_kernel<MT, XB, true>;
        e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, GemvCfg<MT>::kSmem);
        if (e != cudaSuccess) return e;
        int occ_s = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_s, ks, GemvCfg<MT>::kThreads, GemvCfg<MT>::kSmem);
        if (e != cudaSuccess) return e;
        occ = occ_s < occ ? occ_s : occ;
    }
    dev.gemv_occ[XB ? 1 : 0][slot] = occ < 1 ? 1 : occ;
    if (GemvCfg<MT>::kMaxSplit > 8 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess)
        (void)cudaGetLastError();  // then the occupancy query below reports 0 for C > 8
    for (int c = 2; c <= GemvCfg<MT>::kMaxSplit; ++c) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c, 1, 1);
        cfg.blockDim = dim3(GemvCfg<MT>::kThreads, 1, 1);
        cfg.dynamicSmemBytes = GemvCfg<MT>::kSmem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = c;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        dev.gemv_clusters[XB ? 1 : 0][slot][c] = n;
    }
    return cudaSuccess;
}

cudaError_t gemv_setup(DeviceInfo& dev) {
    cudaError_t e = cudaSuccess;
    cudaError_t r;
#define Q4K_SET(MT, SLOT)                                                \
    if ((r = set_attr<MT, false>(dev, SLOT)) != cudaSuccess) e = r;      \
    if ((r = set_attr<MT, true>(dev, SLOT)) != cudaSuccess) e = r;
    Q4K_SET(1, 0) Q4K_SET(2, 1) Q4K_SET(4, 2) Q4K_SET(8, 3) Q4K_SET(16, 4)
#undef Q4K_SET
    return e;
}

template <int MT, bool XB>
static cudaError_t launch_mt(const WeightGroup& grp, const void* X, int M, int K, cudaStream_t stream,
                             const DeviceInfo& dev, int slot, int pdl, unsigned long long* amax) {
    const int KB = K / kBlockWeights;
    const int tiles = grp.tile_start[grp.count];
    const int slots = dev.num_sms * dev.gemv_occ[XB ? 1 : 0][slot];
    int C = 1, kb_per = KB, grid;
    if (tiles >= slots) {
        // persistent, one CTA per resident slot (CTA c streams tiles c, c + grid,
        // ...): the busiest SM then holds ceil(tiles / SMs) tiles, where sizing the
        // grid to equalise tiles per CTA would leave some SMs with one CTA and
        // others with two full ones
        grid = slots;
    } else {
        // split K across a cluster (at least one super-block per CTA), as wide
        // as 85 % of the CTA slots allow while every cluster is resident at
        // once. The free slots let the next launch's clusters start (and
        // stream their weights) before this launch ends. Measured per launch
        // (304 slots): 7168 x 5120 q/k/v 280 CTAs 10.2 us, 224 CTAs 6.9 us;
        // 5120 x 17408 down 280 CTAs 16.9 us, 240 CTAs 14.1 us; 16384 x 2048
        // gate/up 256 CTAs 6.35 us, 128 CTAs 9.5 us.
        int c = (17 * slots / 20) / tiles;
        c = c > GemvCfg<MT>::kMaxSplit ? GemvCfg<MT>::kMaxSplit : c;
        c = c > KB ? KB : c;
        C = 1;
        for (; c >= 2; --c) {
            const int kp = (KB + c - 1) / c;
            const int ce = (KB + kp - 1) / kp;
            if (dev.gemv_clusters[XB ? 1 : 0][slot][ce] >= tiles) {
                C = ce;
                kb_per = kp;
                break;
            }
        }
        grid = tiles * C;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(GemvCfg<MT>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = GemvCfg<MT>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (C > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = C;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    // pdl_flags bit 0: the producer also waits for the preceding grid before
    // streaming W (cleared only when the caller allows weight prefetch).
    const int pdl_flags = (pdl == 2) ? 0 : 1;
    // M = 1, fp32 X, without a K split (long, persistent launches, bound by
    // the issue rate of the SMs that hold two CTAs): the variant that moves
    // part of the unpacking to the FMA pipe. Split launches, whose few stages
    // per CTA are latency-bound after the release, keep the shorter dependency
    // chains. Measured (M = 1): 34816 x 5120 gate/up 23.1 -> 21.9 us; 7168 x
    // 5120 q/k/v (split 4 ways) 6.9 -> 7.2 us with the variant; with bf16 X
    // the Qwen3-14B-shaped sweep 1.93 -> 1.98 ms, so bf16 X keeps the masks.
    auto kern = q4k_gemv_kernel<MT, XB, false>;
    if constexpr (MT == 1 && !XB) {
        if (C == 1) kern = q4k_gemv_kernel<MT, XB, true>;
    }
    return cudaLaunchKernelEx(&cfg, kern, grp, X, M, K, C, kb_per, pdl_flags, amax,
                              dev.err);
}

cudaError_t launch_gemv(const WeightGroup& grp, const void* X, bool x_bf16, int M, int K,
                        cudaStream_t stream, const DeviceInfo& dev, int pdl, unsigned long long* amax) {
    const int mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16;
#define Q4K_CASE(MT, SLOT)                                                            \
    case MT:                                                                          \
        return x_bf16 ? launch_mt<MT, true>(grp, X, M, K, stream, dev, SLOT, pdl, amax)   \
                      : launch_mt<MT, false>(grp, X, M, K, stream, dev, SLOT, pdl, amax);
    switch (mt) {
        Q4K_CASE(1, 0) Q4K_CASE(2, 1) Q4K_CASE(4, 2) Q4K_CASE(8, 3) Q4K_CASE(16, 4)
    }
#undef Q4K_CASE
    return cudaErrorInvalidValue;
}

// Keys of the fused argmax: cleared before the GEMV, turned into row indices after it.
__global__ void q4k_argmax_init_kernel(unsigned long long* keys, int M) {
    if (static_cast<int>(threadIdx.x) < M) keys[threadIdx.x] = 0ull;
}
__global__ void q4k_argmax_finish_kernel(unsigned long long* keys, int M) {
    if (static_cast<int>(threadIdx.x) < M) keys[threadIdx.x] = 0xFFFFFFFFull - (keys[threadIdx.x] & 0xFFFFFFFFull);
}

cudaError_t launch_argmax_init(unsigned long long* keys, int M, cudaStream_t stream) {
    q4k_argmax_init_kernel<<<1, 32, 0, stream>>>(keys, M);
    return cudaGetLastError();
}
cudaError_t launch_argmax_finish(unsigned long long* keys, int M, cudaStream_t stream) {
    q4k_argmax_finish_kernel<<<1, 32, 0, stream>>>(keys, M);
    return cudaGetLastError();
}

}  // namespace q4k
