// Cluster-split forward kernels for small batches.
//
// When there are few rows, one CTA per row leaves most SMs idle ("optimize
// inner persistent scheduler for static fusion", description item 2(2):
// small batches do not use all SMs, so give a row more warps).  Here a row
// is split across a thread-block cluster of C CTAs, each on its own SM:
// CTA `rank` holds vectors [rank * NV/C, (rank+1) * NV/C) of the row in
// registers, reduces them inside the CTA, publishes its partial in shared
// memory and, after a cluster barrier, reads all C partials through
// distributed shared memory in rank order (so every CTA computes the same
// bit-identical total).  A final cluster barrier keeps each CTA's shared
// memory alive until its peers have read it.  The "Llu/ln bwd" discussion
// lists grid-parallel inner normalization as not yet built; this is its
// cluster-scoped form.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace nf {

template <int H> struct ClusterShape;
// C = CTAs per row (cluster size, <= 8 so no opt-in is needed),
// T = threads per CTA, VPT = vectors per thread.
template <> struct ClusterShape<1024>  { static constexpr int C = 2, T = 32; };
template <> struct ClusterShape<2048>  { static constexpr int C = 4, T = 32; };
template <> struct ClusterShape<4096>  { static constexpr int C = 8, T = 32; };
template <> struct ClusterShape<5120>  { static constexpr int C = 5, T = 64; };
template <> struct ClusterShape<8192>  { static constexpr int C = 8, T = 64; };
template <> struct ClusterShape<12288> { static constexpr int C = 8, T = 96; };

bool cluster_shape(int64_t hidden, int* c, int* t) {
    switch (hidden) {
        case 1024:  *c = ClusterShape<1024>::C;  *t = ClusterShape<1024>::T;  return true;
        case 2048:  *c = ClusterShape<2048>::C;  *t = ClusterShape<2048>::T;  return true;
        case 4096:  *c = ClusterShape<4096>::C;  *t = ClusterShape<4096>::T;  return true;
        case 5120:  *c = ClusterShape<5120>::C;  *t = ClusterShape<5120>::T;  return true;
        case 8192:  *c = ClusterShape<8192>::C;  *t = ClusterShape<8192>::T;  return true;
        case 12288: *c = ClusterShape<12288>::C; *t = ClusterShape<12288>::T; return true;
        default: return false;
    }
}

namespace {

template <int H>
struct CGeo {
    static constexpr int C = ClusterShape<H>::C;
    static constexpr int T = ClusterShape<H>::T;
    static constexpr int NV = H / kVec;
    static constexpr int SLICE = NV / C;      // vectors per CTA
    static constexpr int VPT = SLICE / T;     // vectors per thread
    static constexpr int W = T / 32;
    static_assert(NV % C == 0 && SLICE % T == 0, "row must split evenly over the cluster");
    static_assert(T % 32 == 0, "whole warps");
};

// Sum one value over the CTA, then over the cluster.  `red` holds W floats,
// `part` one float in this CTA's shared memory.  Returns the cluster total
// in every thread.  Contains two cluster barriers: the first publishes the
// partials, the second (by the caller, via cluster_done) protects them.
template <int T>
__device__ __forceinline__ float cluster_sum(float v, float* red, float* part, cg::cluster_group& cl) {
    float a[1] = {v};
    group_sum<T, 1>(a, red, 0, threadIdx.x);
    if (threadIdx.x == 0) *part = a[0];
    cl.sync();
    float tot = 0.f;
    const int n = static_cast<int>(cl.num_blocks());
    for (int r = 0; r < n; ++r) tot += *cl.map_shared_rank(part, r);
    return tot;
}

template <int H>
__global__ void __launch_bounds__(CGeo<H>::T)
fused_add_rmsnorm_cluster(uint16_t* __restrict__ x, uint16_t* __restrict__ res,
                          const uint16_t* __restrict__ w, int64_t rows, float eps) {
    using G = CGeo<H>;
    __shared__ float red[G::W];
    __shared__ float part[2];
    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int t = threadIdx.x;
    const int64_t stride = gridDim.x / G::C;
    int iter = 0;
    for (int64_t row = blockIdx.x / G::C; row < rows; row += stride, ++iter) {
        uint16_t* xr = x + row * H + rank * G::SLICE * kVec;
        uint16_t* rr = res + row * H + rank * G::SLICE * kVec;
        uint4 xv[G::VPT], rv[G::VPT];
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            xv[k] = ld_stream(xr + (k * G::T + t) * kVec);
            rv[k] = ld_stream(rr + (k * G::T + t) * kVec);
        }
        float s[G::VPT][8];
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            float a[8], b[8];
            unpack8(xv[k], a);
            unpack8(rv[k], b);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                s[k][e] = a[e] + b[e];
                ss += s[k][e] * s[k][e];
            }
            st_stream(rr + (k * G::T + t) * kVec, pack8(s[k]));
        }
        // alternate the partial slot per row so a fast CTA cannot overwrite
        // a value a peer has not read yet
        const float tot = cluster_sum<G::T>(ss, red, &part[iter & 1], cl);
        const float rstd = rsqrtf(tot * (1.0f / H) + eps);
        const int vbase = rank * G::SLICE;
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            float wf[8], o[8];
            unpack8(ld_param(w + (vbase + k * G::T + t) * kVec), wf);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = s[k][e] * rstd * wf[e];
            st_stream(xr + (k * G::T + t) * kVec, pack8(o));
        }
        if constexpr (G::W > 1) __syncthreads();
    }
    cl.sync();  // no CTA leaves while a peer may still read its `part`
}

template <int H>
__global__ void __launch_bounds__(CGeo<H>::T)
rmsnorm_fwd_cluster(uint16_t* y, const uint16_t* x, const uint16_t* __restrict__ w,
                    int64_t rows, float eps) {
    using G = CGeo<H>;
    __shared__ float red[G::W];
    __shared__ float part[2];
    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int t = threadIdx.x;
    const int64_t stride = gridDim.x / G::C;
    int iter = 0;
    for (int64_t row = blockIdx.x / G::C; row < rows; row += stride, ++iter) {
        const int64_t base = row * H + rank * G::SLICE * kVec;
        float f[G::VPT][8];
        float ss = 0.f;
        uint4 xv[G::VPT];
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) xv[k] = ld_stream(x + base + (k * G::T + t) * kVec);
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            unpack8(xv[k], f[k]);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss += f[k][e] * f[k][e];
        }
        const float tot = cluster_sum<G::T>(ss, red, &part[iter & 1], cl);
        const float rstd = rsqrtf(tot * (1.0f / H) + eps);
        const int vbase = rank * G::SLICE;
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            float wf[8], o[8];
            unpack8(ld_param(w + (vbase + k * G::T + t) * kVec), wf);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = f[k][e] * rstd * wf[e];
            st_stream(y + base + (k * G::T + t) * kVec, pack8(o));
        }
        if constexpr (G::W > 1) __syncthreads();
    }
    cl.sync();
}

template <int H>
__global__ void __launch_bounds__(CGeo<H>::T)
layernorm_fwd_cluster(uint16_t* y, float* __restrict__ mean_out, float* __restrict__ rstd_out,
                      const uint16_t* x, const uint16_t* __restrict__ gamma,
                      const uint16_t* __restrict__ beta, int64_t rows, float eps) {
    using G = CGeo<H>;
    __shared__ float red1[G::W];
    __shared__ float red2[G::W];
    __shared__ float part[4];
    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int t = threadIdx.x;
    const int64_t stride = gridDim.x / G::C;
    int iter = 0;
    for (int64_t row = blockIdx.x / G::C; row < rows; row += stride, ++iter) {
        const int64_t base = row * H + rank * G::SLICE * kVec;
        float f[G::VPT][8];
        float sum = 0.f;
        uint4 xv[G::VPT];
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) xv[k] = ld_stream(x + base + (k * G::T + t) * kVec);
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            unpack8(xv[k], f[k]);
#pragma unroll
            for (int e = 0; e < 8; ++e) sum += f[k][e];
        }
        const float mean = cluster_sum<G::T>(sum, red1, &part[(iter & 1) * 2], cl) * (1.0f / H);
        float sq = 0.f;
#pragma unroll
        for (int k = 0; k < G::VPT; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float d = f[k][e] - mean;
                sq += d * d;
            }
        const float var = cluster_sum<G::T>(sq, red2, &part[(iter & 1) * 2 + 1], cl) * (1.0f / H);
        const float rstd = rsqrtf(var + eps);
        const int vbase = rank * G::SLICE;
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            float gf[8], bf[8], o[8];
            unpack8(ld_param(gamma + (vbase + k * G::T + t) * kVec), gf);
            unpack8(ld_param(beta + (vbase + k * G::T + t) * kVec), bf);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = (f[k][e] - mean) * rstd * gf[e] + bf[e];
            st_stream(y + base + (k * G::T + t) * kVec, pack8(o));
        }
        if (rank == 0 && t == 0) {
            if (mean_out) mean_out[row] = mean;
            if (rstd_out) rstd_out[row] = rstd;
        }
        if constexpr (G::W > 1) __syncthreads();
    }
    cl.sync();
}

template <typename Kernel, typename... Args>
cudaError_t launch_clustered(Kernel k, int c, int threads, int grid, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(c);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace

// `grid` must be a multiple of the cluster size; the caller (plan) ensures it.
cudaError_t launch_fused_cluster(int64_t hidden, void* x, void* res, const void* w, int64_t rows,
                                 float eps, int grid, cudaStream_t st) {
    NF_HIDDEN_SWITCH(hidden, {
        return launch_clustered(fused_add_rmsnorm_cluster<H>, CGeo<H>::C, CGeo<H>::T, grid, st,
                                static_cast<uint16_t*>(x), static_cast<uint16_t*>(res),
                                static_cast<const uint16_t*>(w), rows, eps);
    })
}

cudaError_t launch_rms_cluster(int64_t hidden, void* y, const void* x, const void* w, int64_t rows,
                               float eps, int grid, cudaStream_t st) {
    NF_HIDDEN_SWITCH(hidden, {
        return launch_clustered(rmsnorm_fwd_cluster<H>, CGeo<H>::C, CGeo<H>::T, grid, st,
                                static_cast<uint16_t*>(y), static_cast<const uint16_t*>(x),
                                static_cast<const uint16_t*>(w), rows, eps);
    })
}

cudaError_t launch_ln_fwd_cluster(int64_t hidden, void* y, float* mean, float* rstd, const void* x,
                                  const void* gamma, const void* beta, int64_t rows, float eps,
                                  int grid, cudaStream_t st) {
    NF_HIDDEN_SWITCH(hidden, {
        return launch_clustered(layernorm_fwd_cluster<H>, CGeo<H>::C, CGeo<H>::T, grid, st,
                                static_cast<uint16_t*>(y), mean, rstd,
                                static_cast<const uint16_t*>(x),
                                static_cast<const uint16_t*>(gamma),
                                static_cast<const uint16_t*>(beta), rows, eps);
    })
}

}  // namespace nf
