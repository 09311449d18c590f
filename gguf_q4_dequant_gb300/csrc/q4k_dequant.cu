// q4k_dequant.cu -- K1: standalone Q4_K -> fp32 dequantisation.
//
// The GPU form of the rlx-llama32 page's "CPU F32 (parity)" prefill mode: the
// packed weights are expanded to dense fp32, bit-exact. HBM-bound on its
// writes (4 bytes out per 0.5625 bytes in).
//
// Mapping: one warp per super-block per step, one lane per 4-byte qs word.
// Lane u reads qs bytes 4u..4u+3 (32 lanes = 128 contiguous bytes) and writes
// weights 64c+4v .. +3 (low nibbles) and 64c+32+4v .. +3 (high nibbles),
// c = u/8, v = u%8: each warp store instruction covers four full 128-byte lines.
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

__global__ void __launch_bounds__(256) q4k_dequant_kernel(const uint8_t* __restrict__ W,
                                                      float* __restrict__ out, int64_t nblocks) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int c = lane >> 3;       // chunk 0..3
    const int v = lane & 7;        // word within the chunk

    for (int64_t g = warp; g < nblocks; g += nwarps) {
        const uint8_t* blk = W + g * kBlockBytes;
        const uint4 h = __ldg(reinterpret_cast<const uint4*>(blk));
        const uint32_t q = __ldg(reinterpret_cast<const uint32_t*>(blk + 16) + lane);
        const ScaleBytes sb = decode_scales(h.y, h.z, h.w);
        const float d = half_lo(h.x), dmin = half_hi(h.x);
        // this lane's two sub-blocks: 2c (low nibbles) and 2c+1 (high nibbles)
        const uint32_t scw = c < 2 ? sb.sc_lo : sb.sc_hi;
        const uint32_t mw = c < 2 ? sb.m_lo : sb.m_hi;
        const int jb = (2 * c) & 3;
        const float sc0 = static_cast<float>(byte_of(scw, jb));
        const float sc1 = static_cast<float>(byte_of(scw, jb + 1));
        const float m0 = static_cast<float>(byte_of(mw, jb));
        const float m1 = static_cast<float>(byte_of(mw, jb + 1));
        // ((d*sc)*q) - (dmin*m), each operation rounded to nearest even
        const float d1_lo = __fmul_rn(d, sc0), mm_lo = __fmul_rn(dmin, m0);
        const float d1_hi = __fmul_rn(d, sc1), mm_hi = __fmul_rn(dmin, m1);
        float4 lo, hi;
        lo.x = __fsub_rn(__fmul_rn(d1_lo, static_cast<float>(q & 15u)), mm_lo);
        lo.y = __fsub_rn(__fmul_rn(d1_lo, static_cast<float>((q >> 8) & 15u)), mm_lo);
        lo.z = __fsub_rn(__fmul_rn(d1_lo, static_cast<float>((q >> 16) & 15u)), mm_lo);
        lo.w = __fsub_rn(__fmul_rn(d1_lo, static_cast<float>((q >> 24) & 15u)), mm_lo);
        hi.x = __fsub_rn(__fmul_rn(d1_hi, static_cast<float>((q >> 4) & 15u)), mm_hi);
        hi.y = __fsub_rn(__fmul_rn(d1_hi, static_cast<float>((q >> 12) & 15u)), mm_hi);
        hi.z = __fsub_rn(__fmul_rn(d1_hi, static_cast<float>((q >> 20) & 15u)), mm_hi);
        hi.w = __fsub_rn(__fmul_rn(d1_hi, static_cast<float>(q >> 28)), mm_hi);
        float* o = out + g * kBlockWeights + 64 * c + 4 * v;
        __stcs(reinterpret_cast<float4*>(o), lo);
        __stcs(reinterpret_cast<float4*>(o + 32), hi);
    }
}

cudaError_t launch_dequant(const uint8_t* W, int64_t N, int64_t K, float* out, cudaStream_t stream,
                           int num_sms) {
    const int64_t nblocks = N * (K / kBlockWeights);
    const int threads = 256;
    const int64_t want = (nblocks + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    const int grid = static_cast<int>(want < cap ? want : cap);
    q4k_dequant_kernel<<<grid, threads, 0, stream>>>(W, out, nblocks);
    return cudaGetLastError();
}

}  // namespace q4k
