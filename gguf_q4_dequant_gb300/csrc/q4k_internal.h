// q4k_internal.h -- host-side launchers shared between the C ABI shim and the
// kernel translation units. Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q4k {

struct DeviceInfo {
    int num_sms = 0;
    int max_smem_optin = 0;
    unsigned int* err = nullptr;  // device address of the device error word
    // GEMM: clusters of C CTAs that can be resident at once, per tile width
    // BN = 32 << i (i < 4) and split C (index C, 1..8), from the occupancy API.
    int gemm_clusters[4][9] = {};
    // GEMV, per (bf16 activations?, M slot 1/2/4/8/16): resident CTAs per SM,
    // and resident clusters of C CTAs (index C, 2..16).
    int gemv_occ[2][5] = {};
    int gemv_clusters[2][5][17] = {};
    // tensor-core decode kernel, same indexing (C up to 8)
    int tc_occ[2][5] = {};
    int tc_clusters[2][5][9] = {};
};

cudaError_t launch_dequant(const uint8_t* W, int64_t N, int64_t K, float* out, cudaStream_t stream,
                           int num_sms);

// Programmatic-dependent-launch mode of a call (see q4k_set_pdl in q4k.h):
// 0 = plain launch, 1 = overlap the launch with the preceding kernel,
// 2 = also stream W before the preceding kernel has finished.
//
// Split-K GEMV for 1 <= M <= 16 rows of activations (fp32 or bf16 bit patterns)
// over up to kMaxGroup weight matrices that share K and X (one launch).
constexpr int kMaxGroup = 8;
// Up to kMaxGroup weight matrices that share K and X, as one launch: global
// 128-row tile t belongs to matrix i with tile_start[i] <= t < tile_start[i+1].
struct WeightGroup {  // aligned as its CUtensorMap members
    CUtensorMap maps[kMaxGroup];     // W_i: 2-D uint8 map {K/256*144, N_i}, box {144, 128}
    float* Y[kMaxGroup];             // Y_i: fp32 [M][N_i]
    int N[kMaxGroup];
    int tile_start[kMaxGroup + 1];   // prefix sums of ceil(N_i / 128)
    int count;
};

// Matrix of the group that owns global tile t.
__host__ __device__ inline int group_matrix(const WeightGroup& g, int t) {
    int i = 0;
    while (i + 1 < g.count && t >= g.tile_start[i + 1]) ++i;
    return i;
}
// amax != nullptr: no Y is written; the argmax key of each activation row's
// outputs (see argmax_key) is combined into amax[m] instead (count == 1).
cudaError_t launch_gemv(const WeightGroup& grp, const void* X, bool x_bf16, int M, int K,
                        cudaStream_t stream, const DeviceInfo& dev, int pdl,
                        unsigned long long* amax = nullptr);
// The same product on the tensor cores (1 <= M <= 16): the 4-bit codes are the
// MMA's A operand; fp32 X is split into bf16 hi + lo to keep fp32 accuracy.
cudaError_t launch_tcgemv(const WeightGroup& grp, const void* X, bool x_bf16, int M, int K,
                          cudaStream_t stream, const DeviceInfo& dev, int pdl,
                          unsigned long long* amax = nullptr);
// Sets its attributes and fills dev.tc_occ / dev.tc_clusters.
cudaError_t tcgemv_setup(DeviceInfo& dev);
cudaError_t launch_argmax_init(unsigned long long* keys, int M, cudaStream_t stream);
cudaError_t launch_argmax_finish(unsigned long long* keys, int M, cudaStream_t stream);
// Sets the kernels' attributes and fills dev.gemv_occ / dev.gemv_clusters.
cudaError_t gemv_setup(DeviceInfo& dev);

// tcgen05 GEMM for M >= 17 rows of bf16 activations over a group of weight
// matrices (grp.maps as for the GEMV); tmapX: 3-D bf16 map {64, M, K / 64},
// box {64, BN, gemm_x_steps(BN)}, 128-byte swizzle.
struct GemmLaunch {
    int t0, t1;  // global weight tiles [t0, t1) of the launch
    int C;       // K-split factor (cluster size along z)
    int kb_per;  // super-blocks per K-slice
};
struct GemmPlan {
    int BN;             // tokens per tile (MMA N)
    int nlaunch;        // 1, or 2: full waves of unsplit tiles, then the rest split in K
    GemmLaunch part[2];
};
// ntiles: total 128-row weight tiles of the group.
GemmPlan gemm_plan(int M, int ntiles, int K, const DeviceInfo& dev);
// 64-k steps of X that one TMA copy of the GEMM brings for tile width BN: the
// X tensor map is a 3-D view {64 k, M rows, K / 64} with box {64, BN, this}.
int gemm_x_steps(int BN);
cudaError_t launch_gemm(const WeightGroup& grp, const CUtensorMap& tmapX, int M, int K, int BN,
                        const GemmLaunch& part, cudaStream_t stream, const DeviceInfo& dev, int pdl);
// Sets the kernels' attributes and fills dev.gemm_clusters.
cudaError_t gemm_setup(DeviceInfo& dev);

}  // namespace q4k
