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
// Warp roles (640 threads, one CTA per SM):
//   warp 0      TMA producer of the packed W super-block tiles {144 B, 128
//               rows}, into their own ring, refilled as the dequantisers
//               release a stage
//   warp 19     TMA producer of the X tiles (k-major, 128-byte swizzle, into
//               their own ring of k-steps): one copy brings kXSteps
//               consecutive 64-k tiles of BN token rows ({64 k, BN rows,
//               kXSteps} of a 3-D view of X), refilled as the MMAs of the
//               copy it replaces complete. (A TMA issue costs its thread
//               150-350 cycles; one copy per 64-k step, from a thread that
//               also fed the W ring, came only every ~800 cycles, slower than
//               the MMAs of a small-BN step.)
//   warps 1, 18 MMA issuers: warp 1 takes the even k-steps, warp 18 the odd
//               ones, each into its own TMEM accumulator (the epilogue adds
//               the two), so the barrier waits and issue latencies of two
//               steps overlap (the warp runs the loop, one elected lane
//               issues 4 MMAs of K = 16 and a commit per step, plus one at
//               its last step of an X copy); warp 1 also allocates TMEM
//   warps 2..17 dequantisers, four groups of 128 threads: thread t <-> weight
//               row t % 128 of the 64-k chunk c = t / 128 of every super-block
//               (k-step 4 sb + c). A thread reads its row's header and the
//               chunk's 32 qs bytes into registers, releases the W stage, and
//               writes the whole 128-byte A row of its k-step (64 bf16
//               weights, both nibble halves): one stage wait, one proxy fence
//               and one arrival per 64 weights. The four chunks of a
//               super-block are dequantised in parallel. Then the epilogue
//               (TMEM -> registers -> Y, 128-byte coalesced stores per token
//               column; four warps per TMEM lane quadrant).
// When the tiles alone cannot fill the GPU, K is split across a thread-block
// cluster of C CTAs: each CTA pushes the accumulator rows owned by rank r
// (rows [r*rows, (r+1)*rows), rows = ceil(128/C) rounded up to a multiple of 4)
// from TMEM into rank r's shared memory through distributed shared memory, and
// rank r adds the C partials in rank order (deterministic). Several matrices
// sharing K and X run as one launch (global tile -> matrix, as for the GEMV).
// All pipeline waits are bounded (see mbar_wait).
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

constexpr int kGemmBM = 128;
constexpr int kGemmKStep = 64;                       // bf16 k per A/B stage (one 128-byte row)
constexpr int kGemmDequantWarps = 16;
constexpr int kGemmDequantThreads = 32 * kGemmDequantWarps;   // 512
constexpr int kGemmWarpMma2 = 2 + kGemmDequantWarps;          // the second MMA warp (18)
constexpr int kGemmWarpX = kGemmWarpMma2 + 1;                  // the X producer (19)
constexpr int kGemmThreads = 32 * (kGemmWarpX + 1);            // 640
constexpr int kGemmWStageBytes = kGemmBM * kBlockBytes;   // 18432
constexpr int kGemmAStageBytes = kGemmBM * 128;           // 16384

// Two rings of k-steps: dequantised A tiles (S stages) and TMA-loaded X (B)
// tiles (kXRing stages, kXSteps per copy). An MMA-issuing warp waits on the
// A tile's full barrier (its dequantising group has arrived; one per (MMA
// warp, stage): k-step ks is warp ks % 2's, visited every lcm(2, S) steps)
// and the X copy's full barrier, and its commit releases the A stage; its
// last commit in an X copy releases the copy's X stages.
//
// Release barriers: an mbarrier wait names only the parity of the phase it
// waits for, so a waiter must never find its barrier two phases behind that
// phase. A dequantising group writes every fourth k-step; with a ring of S < 4
// stages a per-stage release barrier could be two phases behind when the group
// comes back to the stage. So the release of k-step ks (the commit of k-step
// ks - S) goes to a barrier of its own pair (group ks % 4, stage ks % S): the
// group visits that pair every L = lcm(4, S) steps and each visit is released
// by exactly one commit, the (ks - S) / L -th on that barrier. The producer
// waits on the same barriers for the X tiles. Both barrier families see one
// MMA warp each (L is even), so their phases follow the steps in order.
template <int BN>
struct GemmCfg {
    // A ring (k-steps): a dequantising group writes every fourth step, so a
    // ring of 4 gives each group one stage and chains its writes to the MMAs
    // of its previous step; 6 lets it run ahead (32-token tiles: 83 -> 80 us
    // per Qwen3-8B-shaped layer)
    static constexpr int kStages = BN == 256 ? 3 : BN == 32 ? 6 : 4;
    // 64-k steps per X copy (the stages of one copy are consecutive in the ring)
    static constexpr int kXSteps = BN == 256 ? 1 : 4;
    // X ring (k-steps), apart from the A ring: for narrow tiles two copies are
    // in flight, so the next super-block's X lands while this one is consumed;
    // at BN = 256 the 32 KB copy of each k-step paces the MMAs, and a fourth X
    // stage (with 2 W stages to make room) measured 169 -> 163 us per
    // Qwen3-8B-shaped layer of 512 rows
    static constexpr int kXRing = BN <= 64 ? 8 : BN == 256 ? 4 : kStages;
    static_assert(kXRing % kXSteps == 0, "X copies tile the ring");
    static constexpr int kXSlots = kXRing / kXSteps;  // X copies in flight
    // X-full barriers: with kXSteps > 1 (even) both MMA warps wait on every
    // copy, one barrier per slot; with one step per copy each warp waits only
    // on its own steps' copies, so (as for the A tiles) one per (warp, slot)
    static constexpr int kXBars = kXSteps == 1 ? 2 * kXSlots : kXSlots;
    static constexpr int kXL2 = kXSlots % 2 == 0 ? kXSlots : 2 * kXSlots;  // lcm(2, kXSlots)
    // packed-W ring (super-blocks), the rest of shared memory: a W box takes
    // several microseconds from issue to landing under load
    static constexpr int kWStages = BN == 256 ? 2 : 5;
    static constexpr int kL = kStages % 4 == 0 ? kStages : kStages % 2 == 0 ? 2 * kStages : 4 * kStages;  // lcm(4, S)
    static constexpr int kL2 = kStages % 2 == 0 ? kStages : 2 * kStages;  // lcm(2, S)
    static constexpr int kBStageBytes = BN * 128;
    static constexpr int kOffA = 0;                                            // 1024-aligned
    static constexpr int kOffB = kOffA + kStages * kGemmAStageBytes;           // 1024-aligned
    static constexpr int kOffW = kOffB + kXRing * kBStageBytes;
    static constexpr int kOffBar = kOffW + kWStages * kGemmWStageBytes;
    // barriers: w_full[W], w_empty[W], full[2][S] (A tiles), release[4][S] (A tiles),
    // x_full[kXBars], x_release[kXSlots], acc_full
    static constexpr int kNumBars = 2 * kWStages + 6 * kStages + kXBars + kXSlots + 1;
    static constexpr int kOffTmem = kOffBar + kNumBars * 8;  // TMEM address; +8: a word holding 0
    static constexpr int kSmem = kOffTmem + 16 + 1024;   // + alignment slack
    static_assert(kSmem <= 232448, "shared memory per CTA");
    static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators of BN columns
    // split-K slots: C <= 8 slots of BN x rows floats in the A/B region, rows =
    // ceil(128 / C) rounded up to a multiple of 4; C * rows <= 144 for C <= 8
    static_assert((kGemmBM + 16) * BN * 4 <= kOffW, "split-K slots must fit in the A/B region");
};

// Eight weights of one nibble half (hh) from the qs word pair P = (w0, w1)
// (bytes b0..b7, little-endian): w = d1*q - m1 in fp32, rounded to bf16.
// A nibble masked in place at bit s of a word, OR'ed with 0x4B000000, is the
// float 2^23 + 2^s*q exactly (s + 4 <= 23); pairs are handled with 64-bit
// masks and the paired fp32 ops: bytes (i, i+4) of the pair form one fp32 pair.
// Bytes 2 and 3 are first brought down by a 64-bit shift by 16. d1s0 / d1s1 are
// (d1*2^-s, d1*2^-s) for s = 4*hh and 8 + 4*hh; nm1 is (-m1, -m1).
__device__ __forceinline__ uint4 dequant8x(uint64_t P, int hh, uint64_t d1s0, uint64_t d1s1,
                                           uint64_t nm1) {
    const uint64_t magic = 0x4B0000004B000000ull;
    const uint64_t neg = 0xCB000000CB000000ull;  // (-2^23, -2^23)
    const uint64_t m0 = 0x0000000F0000000Full << (4 * hh);
    const uint64_t m1 = 0x00000F0000000F00ull << (4 * hh);
    const uint64_t S = P >> 16;
    const uint64_t f0 = fma2(add2((P & m0) | magic, neg), d1s0, nm1);  // (w_b0, w_b4)
    const uint64_t f1 = fma2(add2((P & m1) | magic, neg), d1s1, nm1);  // (w_b1, w_b5)
    const uint64_t f2 = fma2(add2((S & m0) | magic, neg), d1s0, nm1);  // (w_b2, w_b6)
    const uint64_t f3 = fma2(add2((S & m1) | magic, neg), d1s1, nm1);  // (w_b3, w_b7)
    const float2 a = unpack2(f0), b = unpack2(f1), c = unpack2(f2), d = unpack2(f3);
    uint32_t o[4];
    __nv_bfloat162 t;
    t = __floats2bfloat162_rn(a.x, b.x); o[0] = *reinterpret_cast<uint32_t*>(&t);
    t = __floats2bfloat162_rn(c.x, d.x); o[1] = *reinterpret_cast<uint32_t*>(&t);
    t = __floats2bfloat162_rn(a.y, b.y); o[2] = *reinterpret_cast<uint32_t*>(&t);
    t = __floats2bfloat162_rn(c.y, d.y); o[3] = *reinterpret_cast<uint32_t*>(&t);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 32 columns of a lane's accumulator row: the sum of the two MMA warps'
// accumulators (columns c and BN + c), 16 columns of each per load.
template <int BN>
__device__ __forceinline__ void load_acc_sum(uint32_t taddr, float (&v)[32]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t a[16], b[16];
        tmem_ld_32x32b(taddr + 16 * h, a);
        tmem_ld_32x32b(taddr + BN + 16 * h, b);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[16 * h + j] = __uint_as_float(a[j]) + __uint_as_float(b[j]);
    }
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    q4k_gemm_kernel(const __grid_constant__ WeightGroup grp, const __grid_constant__ CUtensorMap tmapX,
                int M, int K, int tile0, int C, int kb_per, int pdl_flags, unsigned int* err) {
    using Cfg = GemmCfg<BN>;
    constexpr int S = Cfg::kStages, WS = Cfg::kWStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // blockIdx.x = (weight tile - tile0) x (token tiles) + token tile: the CTAs of
    // one weight tile are adjacent in launch order, so they run together and
    // the tile's packed bytes come from DRAM once (the others hit L2)
    const int mtiles = (M + BN - 1) / BN;
    const int wt = tile0 + static_cast<int>(blockIdx.x) / mtiles;
    const int mi = group_matrix(grp, wt);
    const CUtensorMap* tmapW = &grp.maps[mi];
    const int N = grp.N[mi];
    float* __restrict__ Y = grp.Y[mi];
    const int n0 = (wt - grp.tile_start[mi]) * kGemmBM;
    const int m0 = (static_cast<int>(blockIdx.x) - (wt - tile0) * mtiles) * BN;
    const int rank = blockIdx.z;  // cluster rank along z = K-slice
    const int kb0 = rank * kb_per;
    const int KB = min(K / kBlockWeights, kb0 + kb_per) - kb0;  // super-blocks of this K-slice
    const int nks = 4 * KB;                                       // 64-k steps of this K-slice
    const int ks0 = 4 * kb0;

    const uint32_t bw_full = sbase + Cfg::kOffBar;
    const uint32_t bw_empty = bw_full + 8 * WS;
    const uint32_t bfull = bw_empty + 8 * WS;
    const uint32_t brel = bfull + 8 * 2 * S;  // [4][S], see GemmCfg
    const uint32_t bxfull = brel + 8 * 4 * S;  // [kXBars], see GemmCfg
    const uint32_t bxrel = bxfull + 8 * Cfg::kXBars;  // [kXSlots]: the MMAs of copy j done
    const uint32_t bacc = bxrel + 8 * Cfg::kXSlots;
    constexpr int XS = Cfg::kXSteps, XQ = Cfg::kXSlots, SX = Cfg::kXRing;
    // the full barrier of X copy j and the parity of its phase
    auto xfull_bar = [&](int j) {
        return bxfull + 8u * static_cast<uint32_t>(XS == 1 ? (j & 1) * XQ + (j >> 1) % XQ : j % XQ);
    };
    auto xfull_parity = [](int j) {
        return static_cast<uint32_t>((XS == 1 ? (j >> 1) / XQ : j / XQ) & 1);
    };
    auto rel_bar = [&](int ks) { return brel + 8u * static_cast<uint32_t>((ks & 3) * S + ks % S); };
    auto rel_parity = [](int ks) { return static_cast<uint32_t>(((ks - S) / Cfg::kL) & 1); };
    // the full barrier of k-step ks's A tile (MMA warp ks % 2) and the parity of its phase
    auto full_bar = [&](int ks) { return bfull + 8u * static_cast<uint32_t>((ks & 1) * S + ks % S); };
    auto full_parity = [](int ks) { return static_cast<uint32_t>((ks / Cfg::kL2) & 1); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffTmem);
    uint32_t* zero_slot = tmem_slot + 2;

    if (threadIdx.x == 0) {
        *zero_slot = 0u;
        for (int i = 0; i < WS; ++i) {
            mbar_init(bw_full + 8 * i, 1);
            mbar_init(bw_empty + 8 * i, kGemmDequantThreads);
        }
        for (int i = 0; i < 2 * S; ++i) mbar_init(bfull + 8 * i, kGemmBM);  // one dequantising group
        for (int i = 0; i < Cfg::kXBars; ++i) mbar_init(bxfull + 8 * i, 1);  // the X producer, with the bytes
        // a copy's stages are free once every MMA warp with steps in it has
        // committed its last one (both warps for 4-step copies)
        for (int i = 0; i < XQ; ++i) mbar_init(bxrel + 8 * i, XS == 1 ? 1 : 2);
        for (int i = 0; i < 4 * S; ++i) mbar_init(brel + 8 * i, 1);  // one MMA commit
        mbar_init(bacc, 2);  // the last commit of each MMA warp
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
    // epilogue assignment of the dequantising warps (set in their branch)
    bool acc_ok = false;
    int epi_cols = 0, epi_c0 = 0, epi_row = 0;
    // Every warp except the W producer waits for the preceding grid here; the
    // W producer waits only unless weight prefetch is allowed.
    if (warp != 0) pdl_wait();

    if (warp == 0) {
        // ---------------------------------------------- W producer (TMA) ---
        if (lane == 0) {
            tma_prefetch_desc(tmapW);
            const uint64_t pol_w = policy_evict_first();
            if (pdl_flags & 1) pdl_wait();
            int sb = 0;
            for (; sb < KB; ++sb) {
                const int ws = sb % WS;
                if (!mbar_wait(bw_empty + 8 * ws, ((sb / WS) & 1) ^ 1, err)) break;
                mbar_arrive_expect_tx(bw_full + 8 * ws, kGemmWStageBytes);
                tma_load_2d_hint(sbase + Cfg::kOffW + ws * kGemmWStageBytes, tmapW,
                                 (kb0 + sb) * kBlockBytes, n0, bw_full + 8 * ws, pol_w);
            }
            // On a timeout the CTA must still not exit while a copy it issued is
            // landing. A stage is reissued only after its previous use was
            // released, which follows the landing of that use's bytes, so at
            // most the last WS stages issued can be in flight: wait for those.
            if (sb < KB)
                for (int i = sb - WS < 0 ? 0 : sb - WS; i < sb; ++i)
                    mbar_wait(bw_full + 8 * (i % WS), (i / WS) & 1, err, kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == kGemmWarpX) {
        // ---------------------------------------------- X producer (TMA) ---
        // (after the preceding grid, like every warp but 0: X is its output).
        // Copy j fills the X stages of k-steps XS*j .. XS*j + XS - 1; they are
        // free once the MMAs of copy j - XQ have completed (its X-release
        // barrier: the last commit of each MMA warp with steps in that copy).
        if (lane == 0) {
            tma_prefetch_desc(&tmapX);
            const uint64_t pol_x = policy_evict_last();
            const int nx = nks / XS;
            int j = 0;
            for (; j < nx; ++j) {
                if (j >= XQ && !mbar_wait(bxrel + 8 * (j % XQ), ((j / XQ) - 1) & 1, err)) break;
                const uint32_t xb = xfull_bar(j);
                mbar_arrive_expect_tx(xb, XS * Cfg::kBStageBytes);
                tma_load_3d_hint(sbase + Cfg::kOffB + ((XS * j) % SX) * Cfg::kBStageBytes, &tmapX, 0, m0,
                                 ks0 + XS * j, xb, pol_x);
            }
            // as for W: at most the last XQ copies issued can be landing
            if (j < nx)
                for (int i = j - XQ < 0 ? 0 : j - XQ; i < j; ++i)
                    mbar_wait(xfull_bar(i), xfull_parity(i), err, kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == 1 || warp == kGemmWarpMma2) {
        // ------------------------------------------------ MMA issuers ---
        // The whole warp runs the loop and the waits (so stage indices and
        // descriptors stay warp-uniform); one elected lane issues. Warp
        // mw = 0 / 1 takes k-steps mw, mw + 2, ... into accumulator mw.
        constexpr uint32_t idesc = idesc_bf16_f32(kGemmBM, BN);
        const int mw = warp == 1 ? 0 : 1;
        const uint32_t dacc = tmem + static_cast<uint32_t>(mw * BN);
        for (int ks = mw; ks < nks; ks += 2) {
            const int s = ks % S;
            const bool ok = mbar_wait(xfull_bar(ks / XS), xfull_parity(ks / XS), err) &&
                            mbar_wait(full_bar(ks), full_parity(ks), err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            if (elect_one()) {
                const uint64_t a0 = sw128_desc(sbase + Cfg::kOffA + s * kGemmAStageBytes);
                const uint64_t b0 = sw128_desc(sbase + Cfg::kOffB + (ks % SX) * Cfg::kBStageBytes);
#pragma unroll
                for (int kk = 0; kk < kGemmKStep / 16; ++kk)  // +32 bytes per k16 = +2 in the address field
                    tc_mma_bf16(dacc, a0 + 2 * kk, b0 + 2 * kk, idesc, (ks >= 2) || kk != 0);
                tc_commit(rel_bar(ks + S));  // releases the A stage for k-step ks + S
                // this warp's last step of its X copy releases the copy's X stages
                if (XS == 1 || (ks % XS) >= XS - 2) tc_commit(bxrel + 8 * ((ks / XS) % XQ));
            }
            __syncwarp();
        }
        if (elect_one()) tc_commit(bacc);
        __syncwarp();
    } else {
        // ------------------------------------------ dequantisers (A) ---
        const int t = threadIdx.x - 64;
        const int r = t & (kGemmBM - 1);  // weight row within the tile
        const int c = t >> 7;             // 64-k chunk of the super-block (warp-uniform)
        // 0, read from shared memory so that the compiler cannot fold the
        // data dependence built from it below
        const uint32_t zero = *reinterpret_cast<volatile uint32_t*>(zero_slot);
        bool ok = true;
        for (int sb = 0; sb < KB && ok; ++sb) {
            const int ws = sb % WS;
            if (!mbar_wait(bw_full + 8 * ws, (sb / WS) & 1, err)) { ok = false; break; }
            // the row's header and the chunk's 32 qs bytes into registers at
            // once, and the W stage released before any arithmetic. The
            // release must not overtake these reads: issued while they were
            // still outstanding, it let the next super-block's TMA write
            // overwrite the stage first (seen as sporadic stale rows with
            // 3-stage rings). Its barrier address depends on the loaded values
            // (and-ed with 0), so it cannot issue before all three loads have
            // returned -- the ordering a proxy fence gives, at a fraction of
            // its cost (measured: 5 % on a 32-row prefill sweep)
            const uint8_t* P = smem + Cfg::kOffW + ws * kGemmWStageBytes + r * kBlockBytes;
            const uint4 hd = *reinterpret_cast<const uint4*>(P);
            const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(P + 16 + 32 * c);
            const ulonglong2 qb = *reinterpret_cast<const ulonglong2*>(P + 32 + 32 * c);
            const uint32_t dep =
                (hd.x ^ static_cast<uint32_t>(qa.x) ^ static_cast<uint32_t>(qb.x)) & zero;
            mbar_arrive(bw_empty + 8 * ws + dep);
            const ScaleBytes scb = decode_scales(hd.y, hd.z, hd.w);
            const float d = half_lo(hd.x), dmin = half_hi(hd.x);
            const uint64_t qw[4] = {qa.x, qa.y, qb.x, qb.y};  // qs bytes 8v .. 8v+7 of the chunk
            uint4 o[2][4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                // low nibbles (hh = 0) are sub-block 2c, k = b; high nibbles sub-block
                // 2c + 1, k = 32 + b, for qs byte b of the chunk
                const int j = 2 * c + hh;
                const uint32_t scw = j < 4 ? scb.sc_lo : scb.sc_hi;
                const uint32_t mw = j < 4 ? scb.m_lo : scb.m_hi;
                const float d1 = d * byte_to_float(scw, j & 3);
                const float m1 = dmin * byte_to_float(mw, j & 3);
                const float d1s0 = d1 * exp2i(-4 * hh), d1s1 = d1 * exp2i(-8 - 4 * hh);
                const uint64_t D0 = pack2(d1s0, d1s0), D1 = pack2(d1s1, d1s1), NM = pack2(-m1, -m1);
#pragma unroll
                for (int v = 0; v < 4; ++v) o[hh][v] = dequant8x(qw[v], hh, D0, D1, NM);
            }
            const int ks = sb * 4 + c;
            const int s = ks % S;
            if (ks >= S && !mbar_wait(rel_bar(ks), rel_parity(ks), err)) { ok = false; break; }
            // 16-byte chunk 4hh + v of the A row holds k = 32hh + 8v .. +7
            uint8_t* arow = smem + Cfg::kOffA + s * kGemmAStageBytes + r * 128;
            const int sw = r & 7;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    *reinterpret_cast<uint4*>(arow + (((4 * hh + v) ^ sw) << 4)) = o[hh][v];
            fence_proxy_async_smem();
            mbar_arrive(full_bar(ks));
        }

        // ------------------------------------------------- epilogue ---
        // four warps per TMEM lane quadrant, each taking a quarter of the BN columns
        const int q = warp & 3;                      // TMEM lane quadrant this warp may access
        const int half = (warp - 2) >> 2;            // column slice 0..3
        epi_cols = BN >= 128 ? BN / 4 : 32;
        epi_c0 = half * epi_cols;
        epi_row = 32 * q + lane;
        acc_ok = ok && mbar_wait(bacc, 0, err) && epi_c0 < BN;
        if (acc_ok) {
            tc_fence_after();
            if (C == 1) {
                const int n = n0 + epi_row;
#pragma unroll 1
                for (int cc = epi_c0; cc < epi_c0 + epi_cols; cc += 32) {
                    float v[32];
                    load_acc_sum<BN>(tmem + (static_cast<uint32_t>(32 * q) << 16) + cc, v);
                    if (n < N) {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const int m = m0 + cc + jj;
                            if (m < M) Y[static_cast<int64_t>(m) * N + n] = v[jj];
                        }
                    }
                }
            }
        }
    }
    if (C > 1) {
        // Split K: rank r owns rows [r*rows, min(128, (r+1)*rows)) of the tile. Once
        // every CTA's MMAs are complete (first cluster barrier) the A/B region
        // of every CTA is free, and each CTA pushes the rows it does not own
        // straight from TMEM into the owner's region (posted remote stores:
        // slot [source rank][column][owned row]); after the second barrier
        // each owner adds the C slots in rank order (deterministic).
        const int rows = ((kGemmBM + C - 1) / C + 3) & ~3;  // a multiple of 4 (float4 groups)
        const uint32_t slot_bytes = 4u * static_cast<uint32_t>(BN * rows);
        const uint32_t pbase = sbase + Cfg::kOffA;
        cluster_sync_all();
        if (acc_ok) {
            tc_fence_after();
            const int owner = epi_row / rows;
            const uint32_t dst = map_shared_rank(pbase, owner) + rank * slot_bytes +
                                 4u * static_cast<uint32_t>(epi_row - owner * rows);
#pragma unroll 1
            for (int cc = epi_c0; cc < epi_c0 + epi_cols; cc += 32) {
                float v[32];
                load_acc_sum<BN>(tmem + (static_cast<uint32_t>(epi_row & ~31) << 16) + cc, v);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    st_shared_cluster_f32(dst + 4u * static_cast<uint32_t>((cc + jj) * rows), v[jj]);
            }
        }
        cluster_sync_all();
        const int r0 = rank * rows;
        const int nr4 = (min(kGemmBM, r0 + rows) - r0) >> 2;  // owned rows / 4 (> 0 for C <= 8)
        const float* part = reinterpret_cast<const float*>(smem + Cfg::kOffA);
        const bool vec = (N & 3) == 0;  // Y rows 16-byte aligned
        for (int idx = threadIdx.x; idx < nr4 * BN; idx += kGemmThreads) {
            const int col = idx / nr4;
            const int rl = 4 * (idx - col * nr4);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int src = 0; src < C; ++src) {
                const float4 v = *reinterpret_cast<const float4*>(part + src * (BN * rows) + col * rows + rl);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            const int n = n0 + r0 + rl, m = m0 + col;
            if (m >= M) continue;
            float* y = Y + static_cast<int64_t>(m) * N + n;
            if (vec && n + 3 < N) {
                *reinterpret_cast<float4*>(y) = acc;
            } else {
                if (n < N) y[0] = acc.x;
                if (n + 1 < N) y[1] = acc.y;
                if (n + 2 < N) y[2] = acc.z;
                if (n + 3 < N) y[3] = acc.w;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // every MMA this CTA issued has completed before its accumulator is
        // freed (the epilogue's own wait is skipped after a timeout)
        mbar_wait(bacc, 0, err);
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

// ------------------------------------------------------------------ host ---

// Tile width BN (tokens) and K-split C for M token rows over `ntiles` 128-row
// weight tiles, from a cost model fitted to measurements of this kernel: a CTA
// costs ~4 us of launch, pipeline fill and epilogue plus ~0.38 us per 64-k
// step whatever BN is (the dequantising side sets the pace), and a K-split adds
// the DSMEM reduction (~0.5 us + 0.018 us per token column, twice that above
// four ranks). Waves come from the number of clusters the occupancy API says
// can be resident at once. A launch whose unsplit CTAs would end in a partial
// wave may instead run as two: the tiles of the full waves unsplit, then the
// remaining tiles split in K, so that the last wave is short (the second launch
// starts when the first completes; ~2 us between them).
namespace {
struct PlanCost {
    double cost;
    int C, kb_per;
};
PlanCost best_split(int bi, int bn, int M, int ntiles, int KB, const DeviceInfo& dev) {
    const int cs[6] = {1, 2, 3, 4, 6, 8};
    PlanCost best{1e300, 1, KB};
    const int mtiles = (M + bn - 1) / bn;
    for (int c : cs) {
        if (c > KB) break;
        const int kb_per = (KB + c - 1) / c;
        const int ce = (KB + kb_per - 1) / kb_per;
        const int resident = dev.gemm_clusters[bi][ce];
        if (resident < 1) continue;
        const long clusters = static_cast<long>(ntiles) * mtiles;
        const long waves = (clusters + resident - 1) / resident;
        double per = 4.0 + 0.38 * 4.0 * kb_per;
        if (ce > 1) per += (0.5 + 0.018 * bn) * (ce <= 4 ? 1.0 : 2.0);
        const double cost = static_cast<double>(waves) * per;
        if (cost < best.cost * 0.999) best = PlanCost{cost, ce, kb_per};
    }
    return best;
}
}  // namespace

GemmPlan gemm_plan(int M, int ntiles, int K, const DeviceInfo& dev) {
    const int KB = K / kBlockWeights;
    GemmPlan best{32, 1, {{0, ntiles, 1, KB}, {0, 0, 1, KB}}};
    double best_cost = 1e300;
    for (int bi = 0; bi < 4; ++bi) {
        const int bn = 32 << bi;
        if (bn > 32 && bn / 2 >= M) break;  // a narrower tile already covers M
        const int mtiles = (M + bn - 1) / bn;
        const PlanCost one = best_split(bi, bn, M, ntiles, KB, dev);
        if (one.cost < best_cost * 0.999) {
            best_cost = one.cost;
            best = GemmPlan{bn, 1, {{0, ntiles, one.C, one.kb_per}, {0, 0, 1, KB}}};
        }
        // full waves of unsplit tiles, then the rest split
        const int r1 = dev.gemm_clusters[bi][1];
        const long units = static_cast<long>(ntiles) * mtiles;
        if (r1 < 1 || units <= r1) continue;
        const int t1 = static_cast<int>((units / r1) * r1 / mtiles);
        if (t1 < 1 || t1 >= ntiles) continue;
        const double full = static_cast<double>((static_cast<long>(t1) * mtiles + r1 - 1) / r1) *
                            (4.0 + 0.38 * 4.0 * KB);
        const PlanCost rest = best_split(bi, bn, M, ntiles - t1, KB, dev);
        const double cost = full + rest.cost + 2.0;
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            best = GemmPlan{bn, 2, {{0, t1, 1, KB}, {t1, ntiles, rest.C, rest.kb_per}}};
        }
    }
    return best;
}

int gemm_x_steps(int BN) {
    switch (BN) {
        case 32: return GemmCfg<32>::kXSteps;
        case 64: return GemmCfg<64>::kXSteps;
        case 128: return GemmCfg<128>::kXSteps;
        case 256: return GemmCfg<256>::kXSteps;
    }
    return 1;
}

template <int BN>
static cudaError_t setup_bn(DeviceInfo& dev, int bi) {
    cudaError_t e = cudaFuncSetAttribute(q4k_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GemmCfg<BN>::kSmem);
    if (e != cudaSuccess) return e;
    for (int c = 1; c <= 8; ++c) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, c);
        cfg.blockDim = dim3(kGemmThreads, 1, 1);
        cfg.dynamicSmemBytes = GemmCfg<BN>::kSmem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 1;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = c;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, q4k_gemm_kernel<BN>, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = c == 1 ? dev.num_sms : 0;  // plain launches need no co-scheduling
        }
        dev.gemm_clusters[bi][c] = n;
    }
    return cudaSuccess;
}

cudaError_t gemm_setup(DeviceInfo& dev) {
    cudaError_t e = cudaSuccess, r;
    if ((r = setup_bn<32>(dev, 0)) != cudaSuccess) e = r;
    if ((r = setup_bn<64>(dev, 1)) != cudaSuccess) e = r;
    if ((r = setup_bn<128>(dev, 2)) != cudaSuccess) e = r;
    if ((r = setup_bn<256>(dev, 3)) != cudaSuccess) e = r;
    return e;
}

template <int BN>
static cudaError_t launch_bn(const WeightGroup& grp, const CUtensorMap& tmapX, int M, int K,
                             const GemmLaunch& plan, cudaStream_t stream, unsigned int* err, int pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((plan.t1 - plan.t0) * ((M + BN - 1) / BN), 1, plan.C);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = GemmCfg<BN>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (plan.C > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = plan.C;
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
    return cudaLaunchKernelEx(&cfg, q4k_gemm_kernel<BN>, grp, tmapX, M, K, plan.t0, plan.C, plan.kb_per,
                              pdl_flags, err);
}

cudaError_t launch_gemm(const WeightGroup& grp, const CUtensorMap& tmapX, int M, int K, int BN,
                        const GemmLaunch& part, cudaStream_t stream, const DeviceInfo& dev, int pdl) {
    switch (BN) {
        case 32: return launch_bn<32>(grp, tmapX, M, K, part, stream, dev.err, pdl);
        case 64: return launch_bn<64>(grp, tmapX, M, K, part, stream, dev.err, pdl);
        case 128: return launch_bn<128>(grp, tmapX, M, K, part, stream, dev.err, pdl);
        case 256: return launch_bn<256>(grp, tmapX, M, K, part, stream, dev.err, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace q4k
