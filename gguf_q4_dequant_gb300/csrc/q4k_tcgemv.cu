// q4k_tcgemv.cu -- K4: the decode product (M = 1..16 token rows) on the
// tensor cores, at the fp32 accuracy of the GEMV.
//
// Decode reads every packed weight matrix once per token (the per-token weight
// sweep of the rlx-llama32 page, section "Decode"). On CUDA cores each weight
// costs a nibble isolation, a multiply-add per activation row and a shared
// activation load per row; here the tensor core does the multiply-adds and a
// weight costs about half a logic operation:
//
//   For row n, super-block b and sub-block j (32 weights) the product is
//     sum_k w x = d*sc_j * sum_k q_k x_k  -  dmin*m_j * sum_k x_k,
//   so only S_j = sum_k q_k x_k needs the weights themselves. The MMA computes
//   S_j for 128 rows at once with A = the 4-bit codes q and B = the
//   activations, each sub-block into its own TMEM columns (accumulate is reset
//   at the sub-block's first MMA); a readout applies d*sc_j and subtracts the
//   min term per super-block.
//
//   A operand: a code q masked in place inside a 16-bit half, with nothing
//   else set, is, read as a bfloat16 bit pattern, exactly q * 2^-133 (low
//   nibble, bits 0..3) or 16q * 2^-133 (high nibble, bits 4..7: bit 7 is the
//   exponent's low bit, and a pattern below 2^8 reads as pattern * 2^-133
//   whether or not bit 7 is set). One AND of a 32-bit word of codes with
//   0x000F000F (or 0x00F000F0) gives a pair of such operands -- the codes of
//   bytes 0 and 2 -- and a shift by 8 first gives bytes 1 and 3. So the k
//   order within each group of four weights is (0, 2, 1, 3); the B tiles are
//   written in that order too, which leaves the products unchanged.
//   B operand: x of each activation row, scaled per super-block by a power of
//   two S (largest |x| of the block to about 2^120, so the products q * x *
//   2^(S-133) are normal fp32 numbers), split into bfloat16 hi = rn(x') and
//   lo = rn(x' - hi): column 2m holds hi, column 2m+1 lo. The split
//   keeps 16 significant bits (|x' - hi - lo| <= 2^-16 |x'|); the products of
//   bf16 operands are exact in the fp32 accumulator.
//   Readout, per row and activation row m: y += d * 2^(133-S) * sum_j sc_j' *
//   (D_j[2m] + D_j[2m+1]) - dmin * sum_j m_j * sum_k x_k, with sc_j' = sc_j for
//   low-nibble sub-blocks and sc_j / 16 for high-nibble ones (both exact).
//
// Work decomposition (as in K2): tile = 128 rows (MMA M = TMEM lanes); CTAs
// are persistent over tiles, or split K across a thread-block cluster whose
// ranks 1.. push their partial sums into rank 0 (st.async), added in rank order.
//
// Warp roles (one CTA per SM):
//   warp 0        TMA producer: one super-block of 128 rows per W stage
//   warps 1..     MMA issuers (4, or 2 at M = 16; the first allocates TMEM):
//                 per 64-k chunk 4 MMAs (128 x N x 16) into the chunk's two
//                 sub-blocks' columns; issuer i takes the chunks c = i mod n,
//                 so the waits and issue latencies of several chunks overlap
//   8 warps       expansion: thread = (64-k chunk, rows r and r + 64): reads its
//                 code bytes into registers, releases the W stage, writes 128
//                 bf16 operands into the swizzled K-major A tile of the chunk
//                 (chunk-0 threads also copy the rows' headers for the readout);
//                 the four chunks of a super-block are expanded in parallel
//   4 warps       readout (TMEM lane quadrant = warp % 4, lane = row): per
//                 super-block, TMEM -> registers, scales, mins, and the
//                 epilogue (Y stores, or the fused argmax keys)
//   last warps    activations: per super-block, scale, split and write the
//                 B tiles, and the sub-block sums of x
// Two or four TMEM accumulator buffers (all 512 columns) let the MMAs of the
// next super-blocks run while the readout drains one; the readout issues the
// loads of several sub-blocks before one wait. All waits are bounded (see
// mbar_wait).
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

constexpr int kTcRows = 128;
constexpr int kTcWStageBytes = kTcRows * kBlockBytes;  // 18432
constexpr int kTcAStepBytes = kTcRows * 128;           // 128 rows x 64 k bf16 (one 64-k chunk)
constexpr int kTcExpThreads = 256;                     // 8 expansion warps
constexpr int kTcReadThreads = 128;                    // 4 readout warps

template <int MT, bool XB>
struct TcCfg {
    // fp32 activations: columns 2m (hi) and 2m+1 (lo); bf16 activations are
    // exact in bf16 (and stay so scaled by 2^S), so column m holds x' alone
    static constexpr bool kLo = !XB;
    static constexpr int kCPM = kLo ? 2 : 1;                 // B columns per activation row
    static constexpr int kCols = kCPM * MT;
    static constexpr int kMH = MT < 8 ? MT : 8;              // activation rows per readout pass
    static constexpr int kN = kCols <= 16 ? 16 : 32;         // MMA N
    static constexpr int kXWarps = MT >= 8 ? MT / 4 : 1;    // activation warps
    static constexpr int kXRows = MT / kXWarps;              // activation rows per warp
    static constexpr int kWS = 4;                            // W ring (super-blocks)
    static constexpr int kBS = kN == 16 ? 12 : 8;            // B tile ring (chunks): the activation
                                                             // warps run up to 2-3 super-blocks ahead
    static constexpr int kHR = 4;                            // per-super-block side data ring
    static constexpr int kMaxSplit = MT >= 16 ? 4 : 8;
    static constexpr int kAS = 4;                            // A tile ring (chunks: one super-block)
    // MMA-issuing warps: warp i of them takes chunk c of every super-block with
    // c % kMmaWarps == i, so their barrier waits and issue latencies overlap
    // (measured: one warp 122 us, two 82 us, four 83 us on a 128256 x 3072
    // matrix at M = 1 -- beyond two, the SM's MMA issue rate is the limit)
    static constexpr int kMmaWarps = 2;
    static constexpr int kWarpMma = 1;
    static constexpr int kWarpExp = kWarpMma + kMmaWarps;
    static constexpr int kWarpRead = kWarpExp + 8;
    static constexpr int kWarpX = kWarpRead + 4;
    static constexpr int kThreads = 32 * (kWarpX + kXWarps);
    static constexpr int kNAcc = 512 / (8 * kN);             // accumulator buffers (4 or 2)
    static constexpr uint32_t kTmemCols = kNAcc * 8 * kN;    // all 512 columns
    static constexpr int kCPJ = kCPM * kMH;                  // TMEM columns per sub-block and pass
    static constexpr int kJB = kCPJ <= 4 ? 8 : (kCPJ <= 8 ? 4 : (MT >= 16 ? 1 : 2));  // sub-blocks per TMEM wait
    static constexpr int kBStepBytes = kN * 128;
    static constexpr int kOffA = 0;                                            // 1024-aligned
    static constexpr int kOffB = kOffA + kAS * kTcAStepBytes;                  // 1024-aligned
    static constexpr int kOffW = kOffB + kBS * kBStepBytes;
    static constexpr int kOffHdr = kOffW + kWS * kTcWStageBytes;               // [HR][128] x 16 B
    static constexpr int kOffXs = kOffHdr + kHR * kTcRows * 16;                // [HR][MT][8] sum_k x
    static constexpr int kOffG = kOffXs + kHR * MT * 8 * 4;                    // [HR][MT][2] 2^(133-S)
    static constexpr int kOffRed = kOffG + kHR * MT * 2 * 4;                   // [kMaxSplit-1][MT][128]
    static constexpr int kOffBar = kOffRed + (kMaxSplit - 1) * MT * kTcRows * 4;
    // wfull[WS] wempty[WS] afull[AS] aempty[AS] bfull[BS] bempty[BS] hfull[HR] hempty[HR]
    // accfull[4] accempty[4] red fin
    static constexpr int kNumBars = 2 * kWS + 2 * kAS + 2 * kBS + 2 * kHR + 8 + 2;
    static constexpr int kOffTmem = kOffBar + kNumBars * 8;  // TMEM address; +8: a word holding 0
    static constexpr int kSmem = kOffTmem + 16 + 1024;  // + alignment slack
    static_assert(kSmem <= 232448, "shared memory");
};

// 2^n as the product of two floats, for n in [-252, 254].
__device__ __forceinline__ void exp2_pair(int n, float& a, float& b) {
    a = exp2i(n >> 1);
    b = exp2i(n - (n >> 1));
}

// Byte offset of bf16 element (row n, position p < 64) in a K-major tile with
// the 128-byte swizzle: rows of 128 bytes, 16-byte chunks XOR (n % 8).
__device__ __forceinline__ uint32_t sw128_offset(int n, int chunk) {
    return static_cast<uint32_t>((n >> 3) * 1024 + (n & 7) * 128 + ((chunk ^ (n & 7)) << 4));
}

template <int MT, bool XB>
__global__ void __launch_bounds__(TcCfg<MT, XB>::kThreads, 1)
    q4k_tcgemv_kernel(const __grid_constant__ WeightGroup grp, const void* __restrict__ X, int M, int K,
                      int C, int kb_per, int pdl_flags, unsigned long long* amax, unsigned int* err) {
    using Cfg = TcCfg<MT, XB>;
    constexpr int WS = Cfg::kWS, AS = Cfg::kAS, BS = Cfg::kBS, HR = Cfg::kHR, N = Cfg::kN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int KB = K / kBlockWeights;
    const int rank = blockIdx.x % C;
    const int cid = blockIdx.x / C;
    const int ncl = gridDim.x / C;
    const int kb0 = rank * kb_per;
    const int nb = min(KB, kb0 + kb_per) - kb0;
    const int tiles = grp.tile_start[grp.count];
    const int nt_local = (tiles - cid + ncl - 1) / ncl;  // tiles cid, cid + ncl, ...
    const int total = nt_local * nb;                     // super-blocks this CTA processes

    const uint32_t b_wfull = sbase + Cfg::kOffBar;
    const uint32_t b_wempty = b_wfull + 8 * WS;
    const uint32_t b_afull = b_wempty + 8 * WS;
    const uint32_t b_aempty = b_afull + 8 * AS;
    const uint32_t b_bfull = b_aempty + 8 * AS;
    const uint32_t b_bempty = b_bfull + 8 * BS;
    const uint32_t b_hfull = b_bempty + 8 * BS;
    const uint32_t b_hempty = b_hfull + 8 * HR;
    const uint32_t b_accfull = b_hempty + 8 * HR;
    const uint32_t b_accempty = b_accfull + 32;
    const uint32_t b_red = b_accempty + 32;
    const uint32_t b_fin = b_red + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffTmem);
    uint32_t* zero_slot = tmem_slot + 2;
    float* red = reinterpret_cast<float*>(smem + Cfg::kOffRed);

    if (threadIdx.x == 0) {
        *zero_slot = 0u;
        for (int i = 0; i < WS; ++i) {
            mbar_init(b_wfull + 8 * i, 1);                 // producer, with the stage's bytes
            mbar_init(b_wempty + 8 * i, kTcExpThreads);    // every expansion thread
        }
        for (int i = 0; i < AS; ++i) {
            mbar_init(b_afull + 8 * i, kTcExpThreads / 4);  // the expansion threads of one chunk
            mbar_init(b_aempty + 8 * i, 1);                // the MMA commit
        }
        for (int i = 0; i < BS; ++i) {
            mbar_init(b_bfull + 8 * i, 32 * Cfg::kXWarps);  // the activation lanes
            mbar_init(b_bempty + 8 * i, 1);                 // the MMA commit
        }
        for (int i = 0; i < HR; ++i) {
            mbar_init(b_hfull + 8 * i, kTcExpThreads / 4 + 32 * Cfg::kXWarps);  // headers + activation sums
            mbar_init(b_hempty + 8 * i, kTcReadThreads);
        }
        for (int i = 0; i < Cfg::kNAcc; ++i) {
            mbar_init(b_accfull + 8 * i, Cfg::kMmaWarps);  // one commit per MMA warp
            mbar_init(b_accempty + 8 * i, kTcReadThreads);
        }
        mbar_init(b_red, 1);
        mbar_init(b_fin, Cfg::kMmaWarps);
        fence_barrier_init();
        if (C > 1 && rank == 0) mbar_arrive_expect_tx(b_red, (C - 1) * MT * kTcRows * 4);
    }
    if (warp == Cfg::kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (C > 1) cluster_arrive_relaxed();  // the barriers above are ready for remote arrivals
    if (threadIdx.x == 0) pdl_launch_dependents();

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer ---
        if (lane == 0) {
            for (int i = 0; i < grp.count; ++i) tma_prefetch_desc(&grp.maps[i]);
            if (pdl_flags & 1) pdl_wait();
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (; issued < total; ++issued) {
                const int sb = issued, ws = sb % WS;
                if (!mbar_wait(b_wempty + 8 * ws, ((sb / WS) & 1) ^ 1, err)) break;
                const int t = cid + (sb / nb) * ncl;
                const int mi = group_matrix(grp, t);
                mbar_arrive_expect_tx(b_wfull + 8 * ws, kTcWStageBytes);
                tma_load_2d_hint(sbase + Cfg::kOffW + ws * kTcWStageBytes, &grp.maps[mi],
                                 (kb0 + sb % nb) * kBlockBytes, (t - grp.tile_start[mi]) * kTcRows,
                                 b_wfull + 8 * ws, pol);
            }
            // at most the last WS issued stages can still be landing (a stage is
            // reissued only after the expansion threads read its previous use)
            for (int sb = issued - WS < 0 ? 0 : issued - WS; sb < issued; ++sb)
                mbar_wait(b_wfull + 8 * (sb % WS), (sb / WS) & 1, err, kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp < Cfg::kWarpExp) {
        // ----------------------------------------------------- MMA issuers ---
        constexpr uint32_t idesc = idesc_bf16_f32(kTcRows, N);
        constexpr int NA = Cfg::kNAcc, MW = Cfg::kMmaWarps;
        const int mw = warp - Cfg::kWarpMma;
        for (int sb = 0; sb < total; ++sb) {
            const int u = sb % NA;
            if (!__all_sync(0xffffffffu, mbar_wait(b_accempty + 8 * u, ((sb / NA) & 1) ^ 1, err))) break;
            tc_fence_after();
            bool ok = true;
            for (int c = mw; c < 4; c += MW) {
                const int st = 4 * sb + c, as = st % AS, bs = st % BS;
                if (!__all_sync(0xffffffffu, mbar_wait(b_bfull + 8 * bs, (st / BS) & 1, err) &&
                                                 mbar_wait(b_afull + 8 * as, (st / AS) & 1, err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    const uint64_t a0 = sw128_desc(sbase + Cfg::kOffA + as * kTcAStepBytes);
                    const uint64_t b0 = sw128_desc(sbase + Cfg::kOffB + bs * Cfg::kBStepBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // chunk c holds sub-blocks 2c (k 0..31) and 2c+1 (k 32..63); the
                        // first MMA of each sub-block resets its accumulator
                        const uint32_t d = tmem + static_cast<uint32_t>((u * 8 + 2 * c + (kk >> 1)) * N);
                        tc_mma_bf16(d, a0 + 2 * kk, b0 + 2 * kk, idesc, kk & 1);
                    }
                    tc_commit(b_aempty + 8 * as);
                    tc_commit(b_bempty + 8 * bs);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) tc_commit(b_accfull + 8 * u);
            __syncwarp();
        }
        if (elect_one()) tc_commit(b_fin);  // every MMA of this thread has completed
        __syncwarp();
    } else if (warp < Cfg::kWarpRead) {
        // ------------------------------------------------------- expansion ---
        // thread = (chunk c of the super-block, rows r0 and r0 + 64): one step
        // per super-block, the four chunks in parallel
        const int t = threadIdx.x - 32 * Cfg::kWarpExp;
        const int c = t >> 6;              // warp-uniform (two warps per chunk)
        const int r0 = t & 63;
        // 0, read from shared memory so that the compiler cannot fold the
        // data dependence built from it below
        const uint32_t zero = *reinterpret_cast<volatile uint32_t*>(zero_slot);
        for (int sb = 0; sb < total; ++sb) {
            const int ws = sb % WS;
            if (!mbar_wait(b_wfull + 8 * ws, (sb / WS) & 1, err)) break;
            uint4 q[2][2], hd[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const uint8_t* P = smem + Cfg::kOffW + ws * kTcWStageBytes + (r0 + 64 * rr) * kBlockBytes;
                q[rr][0] = *reinterpret_cast<const uint4*>(P + 16 + 32 * c);
                q[rr][1] = *reinterpret_cast<const uint4*>(P + 32 + 32 * c);
                hd[rr] = c == 0 ? *reinterpret_cast<const uint4*>(P) : make_uint4(0u, 0u, 0u, 0u);
            }
            // the stage goes back to the producer only after these reads have
            // returned (its next TMA write must not overtake them): the
            // release's barrier address depends on the loaded values
            const uint32_t dep = (q[0][0].x ^ q[0][1].x ^ q[1][0].x ^ q[1][1].x ^ hd[0].x ^ hd[1].x) & zero;
            mbar_arrive(b_wempty + 8 * ws + dep);
            if (c == 0) {  // the rows' headers, for the readout
                const int hs = sb % HR;
                if (!mbar_wait(b_hempty + 8 * hs, ((sb / HR) & 1) ^ 1, err)) break;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
                    *reinterpret_cast<uint4*>(smem + Cfg::kOffHdr + (hs * kTcRows + r0 + 64 * rr) * 16) = hd[rr];
                mbar_arrive(b_hfull + 8 * hs);
            }
            // word i of the chunk row (bytes 4i..4i+3): low nibbles are k = 4i..4i+3
            // (positions 4i.. in the order 0, 2, 1, 3), high nibbles k = 32 + 4i..
            uint32_t lo[2][16], hi[2][16];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const uint32_t w[8] = {q[rr][0].x, q[rr][0].y, q[rr][0].z, q[rr][0].w,
                                       q[rr][1].x, q[rr][1].y, q[rr][1].z, q[rr][1].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t v8 = w[i] >> 8;
                    lo[rr][2 * i] = w[i] & 0x000F000Fu;      // k 4i+0, 4i+2 (low nibbles of bytes 0, 2)
                    lo[rr][2 * i + 1] = v8 & 0x000F000Fu;    // k 4i+1, 4i+3 (bytes 1, 3)
                    hi[rr][2 * i] = w[i] & 0x00F000F0u;      // high nibbles, 16q
                    hi[rr][2 * i + 1] = v8 & 0x00F000F0u;
                }
            }
            const int st = 4 * sb + c, as = st % AS;
            if (!mbar_wait(b_aempty + 8 * as, ((st / AS) & 1) ^ 1, err)) break;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = r0 + 64 * rr, sw = r & 7;
                uint8_t* arow = smem + Cfg::kOffA + as * kTcAStepBytes + r * 128;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {  // 16-byte chunks q4 (low) and 4 + q4 (high)
                    *reinterpret_cast<uint4*>(arow + ((q4 ^ sw) << 4)) =
                        make_uint4(lo[rr][4 * q4], lo[rr][4 * q4 + 1], lo[rr][4 * q4 + 2], lo[rr][4 * q4 + 3]);
                    *reinterpret_cast<uint4*>(arow + (((4 + q4) ^ sw) << 4)) =
                        make_uint4(hi[rr][4 * q4], hi[rr][4 * q4 + 1], hi[rr][4 * q4 + 2], hi[rr][4 * q4 + 3]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(b_afull + 8 * as);
        }
    } else if (warp < Cfg::kWarpX) {
        // --------------------------------------------------------- readout ---
        pdl_wait();  // before any global write
        if (C > 1) cluster_wait();
        const int qd = warp & 3;                 // TMEM lane quadrant
        const int r = 32 * qd + lane;            // weight row within the tile
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        float y[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) y[m] = 0.f;
        bool ok = true;
        for (int i = 0; i < nt_local && ok; ++i) {
            for (int bl = 0; bl < nb; ++bl) {
                const int sb = i * nb + bl, u = sb % Cfg::kNAcc, hs = sb % HR;
                if (!__all_sync(0xffffffffu, mbar_wait(b_hfull + 8 * hs, (sb / HR) & 1, err) &&
                                                 mbar_wait(b_accfull + 8 * u, (sb / Cfg::kNAcc) & 1, err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint4 hd = *reinterpret_cast<const uint4*>(smem + Cfg::kOffHdr + (hs * kTcRows + r) * 16);
                const ScaleBytes scb = decode_scales(hd.y, hd.z, hd.w);
                const float* xsum = reinterpret_cast<const float*>(smem + Cfg::kOffXs) + hs * MT * 8;
                const float* gf = reinterpret_cast<const float*>(smem + Cfg::kOffG) + hs * MT * 2;
                const float d = half_lo(hd.x), dmin = half_hi(hd.x);
                constexpr int MH = Cfg::kMH, CPM = Cfg::kCPM;
#pragma unroll
                for (int p0 = 0; p0 < MT; p0 += MH) {
                    float qa[MH], ma[MH];
#pragma unroll
                    for (int m = 0; m < MH; ++m) qa[m] = ma[m] = 0.f;
                    constexpr int JB = Cfg::kJB;
#pragma unroll
                    for (int j0 = 0; j0 < 8; j0 += JB) {
                    // JB sub-blocks' loads in flight together, one wait
                    uint32_t vb[JB][CPM * MH];
#pragma unroll
                    for (int jj = 0; jj < JB; ++jj)
                        tmem_ld_32x32b(tl + static_cast<uint32_t>((u * 8 + j0 + jj) * N + CPM * p0), vb[jj]);
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < JB; ++jj) {
                        const int j = j0 + jj;
                        const uint32_t (&v)[CPM * MH] = vb[jj];
                        const uint32_t scw = j < 4 ? scb.sc_lo : scb.sc_hi;
                        const uint32_t mw = j < 4 ? scb.m_lo : scb.m_hi;
                        const float mj = byte_to_float(mw, j & 3);
                        // high-nibble sub-blocks (odd j) carry 16q: sc/16 is exact
                        const float scj = byte_to_float(scw, j & 3) * ((j & 1) ? 0.0625f : 1.f);
#pragma unroll
                        for (int m = 0; m < MH; ++m) {
                            const float sj = CPM == 2 ? __uint_as_float(v[2 * m]) + __uint_as_float(v[CPM * m + 1])
                                                      : __uint_as_float(v[m]);
                            qa[m] = fmaf(scj, sj, qa[m]);
                            ma[m] = fmaf(mj, xsum[(p0 + m) * 8 + j], ma[m]);
                        }
                    }
                    }
#pragma unroll
                    for (int m = 0; m < MH; ++m) {
                        const float g1 = gf[2 * (p0 + m)], g2 = gf[2 * (p0 + m) + 1];
                        y[p0 + m] += d * ((qa[m] * g1) * g2) - dmin * ma[m];
                    }
                }
                tc_fence_before();
                mbar_arrive(b_accempty + 8 * u);
                mbar_arrive(b_hempty + 8 * hs);
            }
            if (ok && C == 1) {
                const int t = cid + i * ncl;
                const int mi = group_matrix(grp, t);
                const int row = (t - grp.tile_start[mi]) * kTcRows + r;
                const int Nm = grp.N[mi];
                float* Ym = grp.Y[mi];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (amax != nullptr)
                        argmax_combine(row < Nm ? argmax_key(y[m], row) : 0ull, lane, m < M, amax + m);
                    else if (m < M && row < Nm)
                        Ym[static_cast<int64_t>(m) * Nm + row] = y[m];
                    y[m] = 0.f;
                }
            }
        }
        if (C > 1) {
            // ranks 1.. push their partial sums into rank 0, which adds them in
            // rank order; a rank that timed out pushes nothing, and rank 0 waits
            // (bounded) for the pushes before it exits
            if (rank != 0) {
                if (ok) {
                    const uint32_t dst = map_shared_rank(smem_u32(red + (rank - 1) * MT * kTcRows), 0);
                    const uint32_t rbar = map_shared_rank(b_red, 0);
#pragma unroll
                    for (int m = 0; m < MT; ++m) st_async_f32(dst + 4 * (m * kTcRows + r), y[m], rbar);
                }
            } else if (__all_sync(0xffffffffu, mbar_wait(b_red, 0, err)) && ok) {
                const int mi = group_matrix(grp, cid);
                const int row = (cid - grp.tile_start[mi]) * kTcRows + r;
                const int Nm = grp.N[mi];
                float* Ym = grp.Y[mi];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float v = y[m];
                    for (int qq = 1; qq < C; ++qq) v += red[((qq - 1) * MT + m) * kTcRows + r];
                    if (amax != nullptr)
                        argmax_combine(row < Nm ? argmax_key(v, row) : 0ull, lane, m < M, amax + m);
                    else if (m < M && row < Nm)
                        Ym[static_cast<int64_t>(m) * Nm + row] = v;
                }
            }
        }
    } else {
        // ----------------------------------------------------- activations ---
        // Lane l holds k = 8l .. 8l+7 of the super-block: chunk c = l / 8,
        // 16-byte chunk l % 8 of the B row, sub-block j = l / 4.
        pdl_wait();
        constexpr int XR = Cfg::kXRows;
        const int mx0 = (warp - Cfg::kWarpX) * XR;  // first activation row of this warp
        const int c = lane >> 3;
        // a row's 8 activations as loaded: one uint4 (8 bf16) or two (8 fp32),
        // kept packed while the next super-block's loads are in flight
        constexpr int RW = XB ? 1 : 2;
        uint4 nxt[XR][RW];
        auto load = [&](int sb, uint4 (&v)[XR][RW]) {
            const int64_t k = static_cast<int64_t>(kb0 + sb % nb) * kBlockWeights + 8 * lane;
#pragma unroll
            for (int m = 0; m < XR; ++m) {
                const int mm = mx0 + m;
#pragma unroll
                for (int h = 0; h < RW; ++h) {
                    if (mm >= M)
                        v[m][h] = make_uint4(0u, 0u, 0u, 0u);
                    else if constexpr (XB)
                        v[m][h] = __ldg(reinterpret_cast<const uint4*>(
                            static_cast<const uint16_t*>(X) + static_cast<int64_t>(mm) * K + k));
                    else
                        v[m][h] = __ldg(reinterpret_cast<const uint4*>(
                            static_cast<const float*>(X) + static_cast<int64_t>(mm) * K + k) + h);
                }
            }
        };
        auto unpack = [&](const uint4 (&w)[RW], float (&f)[8]) {
            if constexpr (XB) {
                const uint32_t wv[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    f[2 * e] = __uint_as_float(wv[e] << 16);
                    f[2 * e + 1] = __uint_as_float(wv[e] & 0xFFFF0000u);
                }
            } else {
                const uint32_t wv[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[RW - 1].x, w[RW - 1].y, w[RW - 1].z, w[RW - 1].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(wv[e]);
            }
        };
        if (total > 0) load(0, nxt);
        for (int sb = 0; sb < total; ++sb) {
            uint4 curw[XR][RW];
#pragma unroll
            for (int m = 0; m < XR; ++m)
#pragma unroll
                for (int h = 0; h < RW; ++h) curw[m][h] = nxt[m][h];
            if (sb + 1 < total) load(sb + 1, nxt);
            const int hs = sb % HR;
            // the slots of this super-block's four chunks and its side-data entry
            bool ok = mbar_wait(b_hempty + 8 * hs, ((sb / HR) & 1) ^ 1, err);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int st = 4 * sb + cc;
                ok = ok && mbar_wait(b_bempty + 8 * (st % BS), ((st / BS) & 1) ^ 1, err);
            }
            if (!__all_sync(0xffffffffu, ok)) break;
            uint8_t* bt = smem + Cfg::kOffB + ((4 * sb + c) % BS) * Cfg::kBStepBytes;
            float* xsum = reinterpret_cast<float*>(smem + Cfg::kOffXs) + hs * MT * 8;
            float* gf = reinterpret_cast<float*>(smem + Cfg::kOffG) + hs * MT * 2;
#pragma unroll
            for (int m = 0; m < XR; ++m) {
                const int mm = mx0 + m;
                float cur[8];
                unpack(curw[m], cur);
                uint32_t amax_bits = 0;
                float sum = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    amax_bits = max(amax_bits, __float_as_uint(cur[e]) & 0x7FFFFFFFu);
                    sum += cur[e];
                }
                amax_bits = __reduce_max_sync(0xffffffffu, amax_bits);
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                // S: the block's largest |x| to [2^120, 2^121); 133 - S back in the readout
                int e = static_cast<int>(amax_bits >> 23) - 127;
                e = e < -126 ? -126 : e;
                const int S = 120 - e;
                float s1, s2, g1, g2;
                exp2_pair(S, s1, s2);
                exp2_pair(133 - S, g1, g2);
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    // positions 2p, 2p+1 of this lane's 8 take k (0, 2), (1, 3), (4, 6), (5, 7)
                    const int ka = (p & 1) + 4 * (p >> 1), kb = ka + 2;
                    const float xa = (cur[ka] * s1) * s2, xb = (cur[kb] * s1) * s2;
                    const __nv_bfloat162 hh = __floats2bfloat162_rn(xa, xb);
                    const float2 hf = __bfloat1622float2(hh);
                    const __nv_bfloat162 ll = __floats2bfloat162_rn(xa - hf.x, xb - hf.y);
                    hw[p] = *reinterpret_cast<const uint32_t*>(&hh);
                    lw[p] = *reinterpret_cast<const uint32_t*>(&ll);
                }
                *reinterpret_cast<uint4*>(bt + sw128_offset(Cfg::kCPM * mm, lane & 7)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                if constexpr (Cfg::kLo)
                    *reinterpret_cast<uint4*>(bt + sw128_offset(2 * mm + 1, lane & 7)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                if ((lane & 3) == 0) xsum[mm * 8 + (lane >> 2)] = sum;
                if (lane == 0) {
                    gf[2 * mm] = g1;
                    gf[2 * mm + 1] = g2;
                }
            }
            fence_proxy_async_smem();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) mbar_arrive(b_bfull + 8 * ((4 * sb + cc) % BS));
            mbar_arrive(b_hfull + 8 * hs);
        }
    }
    if (C > 1 && !(warp >= Cfg::kWarpRead && warp < Cfg::kWarpX)) cluster_wait();  // each arrival waits once
    tc_fence_before();
    __syncthreads();
    if (warp == Cfg::kWarpMma) {
        mbar_wait(b_fin, 0, err);
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

// ------------------------------------------------------------------ host ---

template <int MT, bool XB>
static cudaError_t tc_set_attr(DeviceInfo& dev, int slot) {
    using Cfg = TcCfg<MT, XB>;
    cudaError_t e = cudaFuncSetAttribute(q4k_tcgemv_kernel<MT, XB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, q4k_tcgemv_kernel<MT, XB>, Cfg::kThreads, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    dev.tc_occ[XB ? 1 : 0][slot] = occ < 1 ? 1 : occ;
    for (int c = 2; c <= Cfg::kMaxSplit; ++c) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c, 1, 1);
        cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cfg::kSmem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = c;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, q4k_tcgemv_kernel<MT, XB>, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        dev.tc_clusters[XB ? 1 : 0][slot][c] = n;
    }
    return cudaSuccess;
}

cudaError_t tcgemv_setup(DeviceInfo& dev) {
    cudaError_t e = cudaSuccess, r;
#define Q4K_SET(MT, SLOT)                                                   \
    if ((r = tc_set_attr<MT, false>(dev, SLOT)) != cudaSuccess) e = r;      \
    if ((r = tc_set_attr<MT, true>(dev, SLOT)) != cudaSuccess) e = r;
    Q4K_SET(1, 0) Q4K_SET(2, 1) Q4K_SET(4, 2) Q4K_SET(8, 3) Q4K_SET(16, 4)
#undef Q4K_SET
    return e;
}

template <int MT, bool XB>
static cudaError_t tc_launch_mt(const WeightGroup& grp, const void* X, int M, int K, cudaStream_t stream,
                                const DeviceInfo& dev, int slot, int pdl, unsigned long long* amax) {
    using Cfg = TcCfg<MT, XB>;
    const int KB = K / kBlockWeights;
    const int tiles = grp.tile_start[grp.count];
    const int slots = dev.num_sms * dev.tc_occ[XB ? 1 : 0][slot];
    int C = 1, kb_per = KB, grid;
    if (tiles >= slots) {
        grid = slots;  // persistent: CTA c takes tiles c, c + grid, ...
    } else {
        // split K across a cluster (at least one super-block per CTA), as wide
        // as the CTA slots allow while every cluster is resident at once
        int c = slots / tiles;
        c = c > Cfg::kMaxSplit ? Cfg::kMaxSplit : c;
        c = c > KB ? KB : c;
        for (; c >= 2; --c) {
            const int kp = (KB + c - 1) / c;
            const int ce = (KB + kp - 1) / kp;
            if (dev.tc_clusters[XB ? 1 : 0][slot][ce] >= tiles) {
                C = ce;
                kb_per = kp;
                break;
            }
        }
        grid = tiles * C;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmem;
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
    const int pdl_flags = (pdl == 2) ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, q4k_tcgemv_kernel<MT, XB>, grp, X, M, K, C, kb_per, pdl_flags, amax,
                              dev.err);
}

cudaError_t launch_tcgemv(const WeightGroup& grp, const void* X, bool x_bf16, int M, int K,
                          cudaStream_t stream, const DeviceInfo& dev, int pdl, unsigned long long* amax) {
    const int mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : 0;
#define Q4K_CASE(MT, SLOT)                                                                  \
    case MT:                                                                                \
        return x_bf16 ? tc_launch_mt<MT, true>(grp, X, M, K, stream, dev, SLOT, pdl, amax)  \
                      : tc_launch_mt<MT, false>(grp, X, M, K, stream, dev, SLOT, pdl, amax);
    switch (mt) {
        Q4K_CASE(1, 0) Q4K_CASE(2, 1) Q4K_CASE(4, 2) Q4K_CASE(8, 3) Q4K_CASE(16, 4)
    }
#undef Q4K_CASE
    return cudaErrorInvalidValue;
}

}  // namespace q4k
