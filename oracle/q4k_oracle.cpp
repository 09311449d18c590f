// q4k_oracle.cpp -- CPU oracle for the packed Q4_K dequant-matmul.
//
// TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct reference
// that the GPU library is checked against. Only the test suite, the smoke check
// and the benchmark's CPU-baseline and reference legs may load it. It shares no code, header,
// table or constant with the CUDA library, and it never calls it.
//
// What it computes (the Op::DequantMatMul of the rlx pages: "rlx-qwen3" crate
// page, packed-GGUF note under "Quick start" -- K-quant tensors stay packed and
// every matmul dequantises them; "rlx-llama32" page, section "Packed GGUF"):
//
//   Q4_K super-block, 144 bytes for 256 consecutive weights of one row:
//     bytes 0..1    d     (IEEE binary16, little-endian)
//     bytes 2..3    dmin  (IEEE binary16, little-endian)
//     bytes 4..15   s[12] six-bit sub-block scales and mins, packed
//     bytes 16..143 qs[128] four-bit quants
//   Sub-block j (0..7) covers weights 32j..32j+31 of the super-block.
//     j < 4 : sc = s[j] & 63,                             m = s[j+4] & 63
//     j >= 4: sc = (s[j+4] & 15) | ((s[j-4] >> 6) << 4),  m = (s[j+4] >> 4) | ((s[j] >> 6) << 4)
//   Chunk c (0..3) is qs[32c .. 32c+31]; byte l of it holds weight 64c+l in its
//   low nibble and weight 64c+32+l in its high nibble.
//   w = d*sc*q - dmin*m, evaluated as fp32 round-to-nearest-even operations in
//   the order ((d*sc)*q) - (dmin*m), no fused multiply-add (this file must be
//   compiled with -ffp-contract=off).
//
//   Matmul: Y[m][n] = sum_k X[m][k] * w(n, k), accumulated in double with k
//   ascending; A[m][n] = sum_k |X[m][k] * w(n, k)| (the tolerance scale).
//
// The six-bit unpack rule, byte layout and weight order are this library's
// stated Q4_K contract (the pages name Q4_K -- "lazy Q4_K weights" in the
// nx_f32_llm_run_v3 listing header, "Q4_K_M" in the rlx-llama32 page's
// "Cross-utterance decode-graph reuse" -- but print no layout).
//
// Parity pins (tests/test_oracle_pins.py): hand-worked blocks from
// tests/golden/, per-bit isolation of all 96 scale bits, pack/unpack
// round-trips, exact power-of-two weights, brute force against an independent
// numpy matmul, and matmul invariants; tests/test_oracle_mutants.py plants
// plausible mistakes in a copy of this file and checks that a pin catches each.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

extern "C" {

// IEEE 754 binary16 -> binary32, from the format definition: 1 sign bit,
// 5 exponent bits (bias 15), 10 fraction bits. Exact for every input.
float oracle_f16_to_f32(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 31;
    const int frac = h & 1023;
    double v;
    if (expo == 0) {
        v = std::ldexp((double)frac, -24);                  // zero / subnormal: frac * 2^-24
    } else if (expo == 31) {
        v = frac == 0 ? INFINITY : NAN;                     // infinity / NaN
    } else {
        v = std::ldexp((double)(1024 + frac), expo - 25);   // (1 + frac/1024) * 2^(expo-15)
    }
    return (float)(sign ? -v : v);
}

// bfloat16 -> binary32: bfloat16 is the upper half of a binary32.
float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// The 12 packed scale bytes -> eight (sc, m) six-bit pairs.
void oracle_unpack_scales(const uint8_t* s, uint8_t* sc, uint8_t* m) {
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            sc[j] = s[j] & 63;
            m[j] = s[j + 4] & 63;
        } else {
            sc[j] = (uint8_t)((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4));
            m[j] = (uint8_t)((s[j + 4] >> 4) | ((s[j] >> 6) << 4));
        }
    }
}

// One 144-byte super-block -> 256 fp32 weights in k order.
void oracle_dequant_block(const uint8_t* blk, float* out) {
    const float d = oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    const float dmin = oracle_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t* s = blk + 4;
    const uint8_t* qs = blk + 16;
    uint8_t sc[8], m[8];
    oracle_unpack_scales(s, sc, m);
    for (int c = 0; c < 4; ++c) {
        for (int l = 0; l < 32; ++l) {
            const uint8_t byte = qs[32 * c + l];
            const int q_lo = byte & 15, q_hi = byte >> 4;
            const int j_lo = 2 * c, j_hi = 2 * c + 1;
            // ((d * sc) * q) - (dmin * m): each product and the difference is
            // one fp32 round-to-nearest-even operation.
            const float t_lo = (d * (float)sc[j_lo]) * (float)q_lo;
            const float u_lo = dmin * (float)m[j_lo];
            out[64 * c + l] = t_lo - u_lo;
            const float t_hi = (d * (float)sc[j_hi]) * (float)q_hi;
            const float u_hi = dmin * (float)m[j_hi];
            out[64 * c + 32 + l] = t_hi - u_hi;
        }
    }
}

static int check_dims(int64_t N, int64_t K) {
    if (N < 1 || K < 256 || K % 256 != 0) return -2;
    return 0;
}

// Whole matrix: W is [N][K/256][144] bytes, out is fp32 [N][K] row-major.
int oracle_dequant(const uint8_t* W, int64_t N, int64_t K, float* out) {
    if (!W || !out) return -1;
    if (check_dims(N, K)) return -2;
    const int64_t KB = K / 256;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < KB; ++b)
            oracle_dequant_block(W + (n * KB + b) * 144, out + n * K + b * 256);
    return 0;
}

// Matmul over a subset of rows of W (columns of Y).
//   X      fp32 [M][K] row-major (bf16 inputs are passed as their exact fp32 values)
//   rows   indices n of the rows of W to evaluate (nrows of them); NULL = all N rows
//   Y, A   double [M][nrows]: Y = sum_k x*w, A = sum_k |x*w|, k ascending
//   threads  worker threads over rows (<= 0: hardware concurrency); the
//            arithmetic of each output does not depend on it
int oracle_matmul(const uint8_t* W, int64_t N, int64_t K, const float* X, int64_t M,
                  const int64_t* rows, int64_t nrows, double* Y, double* A, int threads) {
    if (!W || !X || !Y) return -1;
    if (check_dims(N, K) || M < 1) return -2;
    if (!rows) nrows = N;
    if (nrows < 0) return -2;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -2;
    const int64_t KB = K / 256;
    int nt = threads > 0 ? threads : (int)std::max(1u, std::thread::hardware_concurrency());
    nt = (int)std::min<int64_t>(nt, std::max<int64_t>(1, nrows));
    auto work = [&](int64_t r0, int64_t r1) {
        std::vector<float> w((size_t)K);
        for (int64_t r = r0; r < r1; ++r) {
            const int64_t n = rows ? rows[r] : r;
            for (int64_t b = 0; b < KB; ++b)
                oracle_dequant_block(W + (n * KB + b) * 144, w.data() + b * 256);
            for (int64_t mi = 0; mi < M; ++mi) {
                const float* x = X + mi * K;
                double acc = 0.0, aab = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const double p = (double)w[(size_t)k] * (double)x[k];
                    acc += p;
                    aab += std::fabs(p);
                }
                Y[mi * nrows + r] = acc;
                if (A) A[mi * nrows + r] = aab;
            }
        }
    };
    if (nt == 1) {
        work(0, nrows);
    } else {
        std::vector<std::thread> pool;
        const int64_t per = (nrows + nt - 1) / nt;
        for (int t = 0; t < nt; ++t) {
            const int64_t r0 = t * per, r1 = std::min(nrows, r0 + per);
            if (r0 < r1) pool.emplace_back(work, r0, r1);
        }
        for (auto& th : pool) th.join();
    }
    return 0;
}

}  // extern "C"
