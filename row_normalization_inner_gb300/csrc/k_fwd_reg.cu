// Register-persistent forward kernels: fused residual add + RMSNorm (in
// place), RMSNorm forward, LayerNorm forward.
//
// One row per group of TPR threads, RPC groups per CTA.  The hidden size is
// a template constant, so the thread count, the vectors per thread and the
// loops are all static ("optimize inner persistent scheduler for static
// fusion", description item 2(1): static bdimx when the hidden size is
// fixed; bdimx a multiple of the warp size).  Each thread loads its VPT
// 128-bit vectors once, keeps the row in registers (fp32 for the fused
// kernel and for LayerNorm at hidden 1024, packed bf16 widened per pass
// otherwise), and reduces it
// in the same pass that loads it (the page's compute-with-first-consumer
// change): sum of squares for RMSNorm; for LayerNorm the sum, then the
// centered sum of squares over the resident values (two passes, no reload).
#include "common.cuh"
#include "pairs.cuh"
#include "pdl.cuh"
#include "launch.h"

namespace nf {
namespace {

// SMALL: the geometry of calls of at most kSmallCallRows rows: one row per
// CTA, so that a few rows spread over as many SMs (8 x 4096 fused: 1.89 ->
// 1.76 us; at 16384 rows one row per CTA was slower at hidden 4096), and
// twice the threads per row, two vectors each, so each thread's chain of
// loads and sums is shorter (fused 1 x 8192: 2.01 -> 1.79 us, 256 x 8192:
// 3.97 -> 3.47 us).
template <int H, bool SMALL = false>
struct Geo {
    static constexpr int TPR = SMALL ? 2 * RegShape<H>::TPR : RegShape<H>::TPR;
    static constexpr int RPC = SMALL ? 1 : RegShape<H>::RPC;
    static constexpr int NV = H / kVec;
    static constexpr int VPT = NV / TPR;
    static constexpr int W = TPR / 32;
    static_assert(NV % TPR == 0, "hidden/8 must be a multiple of the row's thread count");
    static_assert(TPR % 32 == 0, "a row uses whole warps");
};

// Minimum resident CTAs per SM the RMSNorm / LayerNorm forward kernels are
// compiled for: 5 at hidden 4096 (48 registers, 62.5 % occupancy instead of
// 50 %; measured 40.9 -> 39.6 us and 42.6 -> 41.3 us at 16384 rows), 1
// elsewhere (forcing it at 1024 or 8192, or on the fused kernel, was
// slower), and never for the small-call variants (PRE), whose parameter
// registers would spill.  0 leaves the register count to the compiler's
// default for the block size (an explicit 1 instead lets it grow the count:
// LayerNorm 1024 60 -> 84 registers, RMSNorm 8192 64 -> 75, both slower).
template <int H, bool PRE> struct FwdMinBlocks { static constexpr int v = (H == 4096 && !PRE) ? 5 : 0; };

// [kernel-span fused_add_rmsnorm_reg]
// A parameter vector (weight, gamma or beta) of this thread's columns.
// With PRE the thread loads all VPT vectors once, before its first row, so
// a call with few rows makes one memory round trip (the row and the
// parameters together) instead of loading the parameters after the row
// reduction; without it each is read when it is used, costing no registers
// across the reduction (the choice for large row counts, where occupancy
// matters and the parameters sit in L1).
template <int VPT, bool PRE>
struct ParamVecs {
    uint4 v[PRE ? VPT : 1];
    __device__ __forceinline__ ParamVecs(const uint16_t* p, int tpr, int t) {
        if constexpr (PRE) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) v[k] = ld_param(p + (k * tpr + t) * kVec);
        }
    }
    // vector k of this thread, which is vector `vi` of the row
    __device__ __forceinline__ uint4 get(int k, const uint16_t* p, int vi) const {
        if constexpr (PRE) return v[k];
        else return ld_param(p + vi * kVec);
    }
};

// Before waiting for the kernel ahead of it in the stream, warm L2 with
// this thread's vectors of its CTA's first row (of `a`, and of `b` when
// given): a hint, no data is read.
template <typename G>
__device__ __forceinline__ void prefetch_first_row(const uint16_t* a, const uint16_t* b,
                                                   int64_t rows, int group, int t,
                                                   int64_t first_wave) {
    // Only the first wave of CTAs (first_wave = resident CTAs per SM x SMs)
    // can be resident before the kernel ahead finishes; later CTAs start
    // after it and would only duplicate their own loads.
    if (static_cast<int64_t>(blockIdx.x) >= first_wave) return;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * G::RPC + group;
    if (row >= rows) return;
    constexpr int H = G::NV * kVec;
#pragma unroll
    for (int k = 0; k < G::VPT; ++k) {
        const int64_t off = row * H + (k * G::TPR + t) * kVec;
        prefetch_l2(a + off);
        if (b) prefetch_l2(b + off);
    }
}

// residual <- x + residual ; x <- bf16(s * rsqrt(mean(s^2) + eps) * w)
template <int H, bool PRE>
__global__ void __launch_bounds__(Geo<H, PRE>::TPR * Geo<H, PRE>::RPC)
fused_add_rmsnorm_reg(uint16_t* __restrict__ x, uint16_t* __restrict__ res,
                      const uint16_t* __restrict__ w, int64_t rows, float eps, int64_t first_wave) {
    using G = Geo<H, PRE>;
    __shared__ float red[G::RPC * G::W];
    const int group = threadIdx.x / G::TPR, t = threadIdx.x % G::TPR;
    prefetch_first_row<G>(x, res, rows, group, t, first_wave);
    grid_dep_wait();
    grid_dep_release();
    ParamVecs<G::VPT, PRE> wp(w, G::TPR, t);
    const int64_t nblk = (rows + G::RPC - 1) / G::RPC;
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const int64_t row = blk * G::RPC + group;
        const bool active = row < rows;
        uint16_t* xr = x + row * H;
        uint16_t* rr = res + row * H;
        float s[G::VPT][8];
        float ss[1] = {0.f};
        if (active) {
            uint4 xv[G::VPT], rv[G::VPT];
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                const int v = k * G::TPR + t;
                xv[k] = ld_stream(xr + v * kVec);
                rv[k] = ld_stream(rr + v * kVec);
            }
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float a[8], b[8];
                unpack8(xv[k], a);
                unpack8(rv[k], b);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    s[k][e] = a[e] + b[e];
                    ss[0] += s[k][e] * s[k][e];
                }
                st_stream(rr + (k * G::TPR + t) * kVec, pack8(s[k]));
            }
        }
        group_sum<G::TPR, 1>(ss, red, group, t);
        if (active) {
            const float rstd = rsqrtf(ss[0] * (1.0f / H) + eps);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                const int v = k * G::TPR + t;
                float wf[8], o[8];
                unpack8(wp.get(k, w, v), wf);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = s[k][e] * rstd * wf[e];
                st_stream(xr + v * kVec, pack8(o));
            }
        }
        if constexpr (G::W > 1) __syncthreads();  // `red` is reused by the next row block
    }
}
// [end kernel-span fused_add_rmsnorm_reg]

// y <- bf16(x * rsqrt(mean(x^2) + eps) * w)
template <int H, bool PRE>
__global__ void __launch_bounds__(Geo<H, PRE>::TPR * Geo<H, PRE>::RPC, FwdMinBlocks<H, PRE>::v)
rmsnorm_fwd_reg(uint16_t* y, const uint16_t* x, const uint16_t* __restrict__ w,
                int64_t rows, float eps, int64_t first_wave) {
    using G = Geo<H, PRE>;
    __shared__ float red[G::RPC * G::W];
    const int group = threadIdx.x / G::TPR, t = threadIdx.x % G::TPR;
    prefetch_first_row<G>(x, nullptr, rows, group, t, first_wave);
    grid_dep_wait();
    grid_dep_release();
    ParamVecs<G::VPT, PRE> wp(w, G::TPR, t);
    const int64_t nblk = (rows + G::RPC - 1) / G::RPC;
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const int64_t row = blk * G::RPC + group;
        const bool active = row < rows;
        // the row stays packed (bf16) in registers and is widened per pass;
        // the arithmetic runs on fp32 pairs
        uint4 xv[G::VPT];
        float2 s2 = make_float2(0.f, 0.f);
        if (active) {
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) xv[k] = ld_stream(x + row * H + (k * G::TPR + t) * kVec);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float2 f[4];
                unpack8x2(xv[k], f);
#pragma unroll
                for (int q = 0; q < 4; ++q) s2 = __ffma2_rn(f[q], f[q], s2);
            }
        }
        float ss[1] = {s2.x + s2.y};
        group_sum<G::TPR, 1>(ss, red, group, t);
        if (active) {
            const float rstd = rsqrtf(ss[0] * (1.0f / H) + eps);
            const float2 rstd2 = make_float2(rstd, rstd);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                const int v = k * G::TPR + t;
                float2 f[4], wf[4], o[4];
                unpack8x2(xv[k], f);
                unpack8x2(wp.get(k, w, v), wf);
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = __fmul2_rn(__fmul2_rn(f[q], rstd2), wf[q]);
                st_stream(y + row * H + v * kVec, pack8x2(o));
            }
        }
        if constexpr (G::W > 1) __syncthreads();
    }
}

// mean = sum(x)/H ; var = sum((x-mean)^2)/H ; rstd = rsqrt(var + eps)
// y <- bf16((x - mean) * rstd * gamma + beta)
template <int H, bool PRE>
__global__ void __launch_bounds__(Geo<H, PRE>::TPR * Geo<H, PRE>::RPC, FwdMinBlocks<H, PRE>::v)
layernorm_fwd_reg(uint16_t* y, float* __restrict__ mean_out, float* __restrict__ rstd_out,
                  const uint16_t* x, const uint16_t* __restrict__ gamma,
                  const uint16_t* __restrict__ beta, int64_t rows, float eps, int64_t first_wave) {
    using G = Geo<H, PRE>;
    __shared__ float red1[G::RPC * G::W];
    __shared__ float red2[G::RPC * G::W];
    const int group = threadIdx.x / G::TPR, t = threadIdx.x % G::TPR;
    prefetch_first_row<G>(x, nullptr, rows, group, t, first_wave);
    grid_dep_wait();
    grid_dep_release();
    ParamVecs<G::VPT, PRE> gp(gamma, G::TPR, t), bp(beta, G::TPR, t);
    const int64_t nblk = (rows + G::RPC - 1) / G::RPC;
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const int64_t row = blk * G::RPC + group;
        const bool active = row < rows;
        // Small rows are instruction-bound: widen the row once and center it
        // in place.  Larger rows are occupancy-bound: keep it packed (half
        // the registers) and widen it on each pass.  Either way
        // y = fma(x - mean, rstd * gamma, beta), on fp32 pairs.
        constexpr bool kWide = H <= 1024;
        float2 f[kWide ? G::VPT : 1][4];
        uint4 xv[G::VPT];
        float2 s1 = make_float2(0.f, 0.f);
        if (active) {
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) xv[k] = ld_stream(x + row * H + (k * G::TPR + t) * kVec);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float2 tmp[4];
                unpack8x2(xv[k], tmp);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (kWide) f[k][q] = tmp[q];
                    s1 = __fadd2_rn(s1, tmp[q]);
                }
            }
        }
        float acc[1] = {s1.x + s1.y};
        group_sum<G::TPR, 1>(acc, red1, group, t);
        const float mean = acc[0] * (1.0f / H);
        const float2 nmean2 = make_float2(-mean, -mean);
        float2 s2 = make_float2(0.f, 0.f);
        if (active) {
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float2 tmp[4];
                if constexpr (!kWide) unpack8x2(xv[k], tmp);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (kWide) {
                        f[k][q] = __fadd2_rn(f[k][q], nmean2);
                        s2 = __ffma2_rn(f[k][q], f[k][q], s2);
                    } else {
                        const float2 d = __fadd2_rn(tmp[q], nmean2);
                        s2 = __ffma2_rn(d, d, s2);
                    }
                }
            }
        }
        float sq[1] = {s2.x + s2.y};
        group_sum<G::TPR, 1>(sq, red2, group, t);
        if (active) {
            const float rstd = rsqrtf(sq[0] * (1.0f / H) + eps);
            const float2 rstd2 = make_float2(rstd, rstd);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                const int v = k * G::TPR + t;
                float2 gf[4], bf[4], o[4], xm[4];
                if constexpr (kWide) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) xm[q] = f[k][q];
                } else {
                    unpack8x2(xv[k], xm);
#pragma unroll
                    for (int q = 0; q < 4; ++q) xm[q] = __fadd2_rn(xm[q], nmean2);
                }
                unpack8x2(gp.get(k, gamma, v), gf);
                unpack8x2(bp.get(k, beta, v), bf);
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = __ffma2_rn(xm[q], __fmul2_rn(rstd2, gf[q]), bf[q]);
                st_stream(y + row * H + v * kVec, pack8x2(o));
            }
            if (t == 0) {
                if (mean_out) mean_out[row] = mean;
                if (rstd_out) rstd_out[row] = rstd;
            }
        }
        if constexpr (G::W > 1) __syncthreads();
    }
}

// [kernel-span layernorm_fwd_shift]
// LayerNorm forward with one reduction per row: each warp shifts its values
// by one of them (c = the first element its lane 0 holds) and sums d = x - c
// and d^2; the warp's (mean, M2) = (c + sum d / n, sum d^2 - (sum d)^2 / n)
// over its n elements, and the warps of a row are combined with Chan,
// Golub and LeVeque's pairwise update in warp order.  Because c is one of
// the warp's own values, (c - mean)^2 <= n * var, so the cancellation in
// sum d^2 - (sum d)^2 / n costs at most about n fp32 roundings relative to
// M2 (n <= 1024 here): far below the bf16 output rounding.
template <int H, bool PRE>
__global__ void __launch_bounds__(Geo<H, PRE>::TPR * Geo<H, PRE>::RPC, FwdMinBlocks<H, PRE>::v)
layernorm_fwd_shift(uint16_t* y, float* __restrict__ mean_out, float* __restrict__ rstd_out,
                    const uint16_t* x, const uint16_t* __restrict__ gamma,
                    const uint16_t* __restrict__ beta, int64_t rows, float eps, int64_t first_wave) {
    using G = Geo<H, PRE>;
    constexpr float kNW = 32.0f * G::VPT * kVec;  // elements per warp
    __shared__ float red[G::W > 1 ? G::RPC * G::W * 2 : 1];
    const int group = threadIdx.x / G::TPR, t = threadIdx.x % G::TPR;
    prefetch_first_row<G>(x, nullptr, rows, group, t, first_wave);
    grid_dep_wait();
    grid_dep_release();
    ParamVecs<G::VPT, PRE> gp(gamma, G::TPR, t), bp(beta, G::TPR, t);
    const int warp = t >> 5, lane = t & 31;
    const int64_t nblk = (rows + G::RPC - 1) / G::RPC;
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const int64_t row = blk * G::RPC + group;
        const bool active = row < rows;
        uint4 xv[G::VPT];
        float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
        float c = 0.f;
        if (active) {
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) xv[k] = ld_stream(x + row * H + (k * G::TPR + t) * kVec);
            c = __shfl_sync(0xFFFFFFFFu, bf_lo(xv[0].x), 0);
            const float2 nc2 = make_float2(-c, -c);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float2 f[4];
                unpack8x2(xv[k], f);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 d = __fadd2_rn(f[q], nc2);
                    s1 = __fadd2_rn(s1, d);
                    s2 = __ffma2_rn(d, d, s2);
                }
            }
        }
        float v[2] = {s1.x + s1.y, s2.x + s2.y};
        warp_sum<2>(v);
        const float dm = v[0] * (1.0f / kNW);
        float mean = c + dm;
        float m2 = fmaxf(v[1] - v[0] * dm, 0.f);
        if constexpr (G::W > 1) {
            float* rb = red + group * G::W * 2;
            if (lane == 0) {
                rb[warp * 2] = mean;
                rb[warp * 2 + 1] = m2;
            }
            __syncthreads();
            mean = rb[0];
            m2 = rb[1];
            float n = kNW;
#pragma unroll
            for (int w = 1; w < G::W; ++w) {
                const float d = rb[w * 2] - mean;
                const float nt = n + kNW;
                const float fb = kNW / nt;
                mean = fmaf(d, fb, mean);
                m2 += rb[w * 2 + 1] + d * d * n * fb;
                n = nt;
            }
        }
        if (active) {
            const float rstd = rsqrtf(m2 * (1.0f / H) + eps);
            const float2 rstd2 = make_float2(rstd, rstd), nmean2 = make_float2(-mean, -mean);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                const int vi = k * G::TPR + t;
                float2 xm[4], gf[4], bf[4], o[4];
                unpack8x2(xv[k], xm);
                unpack8x2(gp.get(k, gamma, vi), gf);
                unpack8x2(bp.get(k, beta, vi), bf);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    o[q] = __ffma2_rn(__fadd2_rn(xm[q], nmean2), __fmul2_rn(rstd2, gf[q]), bf[q]);
                st_stream(y + row * H + vi * kVec, pack8x2(o));
            }
            if (t == 0) {
                if (mean_out) mean_out[row] = mean;
                if (rstd_out) rstd_out[row] = rstd;
            }
        }
        if constexpr (G::W > 1) __syncthreads();  // `red` is reused by the next row block
    }
}

// [end kernel-span layernorm_fwd_shift]

// Which LayerNorm forward statistics the register path uses (two passes
// over the resident row, or one shifted pass).
constexpr bool kLnFwdShifted = true;


}  // namespace

// CTAs of a kernel's first wave on this device (resident per SM x SMs).
// `slot` caches the occupancy of one kernel instantiation (a benign race at
// worst repeats the query).
template <typename K>
int64_t first_wave_ctas(K kernel, int threads, int sms, int* slot) {
    int o = *slot;
    if (o <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, threads, 0) != cudaSuccess || o <= 0)
            o = 1;
        *slot = o;
    }
    return static_cast<int64_t>(o) * sms;
}

cudaError_t launch_fused_reg(int64_t hidden, void* x, void* res, const void* w, int64_t rows,
                             float eps, int grid, int sms, cudaStream_t st) {
    const bool pre = rows <= kSmallCallRows;
    NF_HIDDEN_SWITCH(hidden, {
        static int occ[2] = {0, 0};
        const auto k = pre ? fused_add_rmsnorm_reg<H, true> : fused_add_rmsnorm_reg<H, false>;
        const int threads = pre ? Geo<H, true>::TPR * Geo<H, true>::RPC : Geo<H>::TPR * Geo<H>::RPC;
        return launch_with_pdl(k, dim3(grid), dim3(threads), 0, st, static_cast<uint16_t*>(x),
                               static_cast<uint16_t*>(res), static_cast<const uint16_t*>(w), rows,
                               eps, first_wave_ctas(k, threads, sms, &occ[pre]));
    })
}

cudaError_t launch_rms_reg(int64_t hidden, void* y, const void* x, const void* w, int64_t rows,
                           float eps, int grid, int sms, cudaStream_t st) {
    const bool pre = rows <= kSmallCallRows;
    NF_HIDDEN_SWITCH(hidden, {
        static int occ[2] = {0, 0};
        const auto k = pre ? rmsnorm_fwd_reg<H, true> : rmsnorm_fwd_reg<H, false>;
        const int threads = pre ? Geo<H, true>::TPR * Geo<H, true>::RPC : Geo<H>::TPR * Geo<H>::RPC;
        return launch_with_pdl(k, dim3(grid), dim3(threads), 0, st, static_cast<uint16_t*>(y),
                               static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(w),
                               rows, eps, first_wave_ctas(k, threads, sms, &occ[pre]));
    })
}

cudaError_t launch_ln_fwd_reg(int64_t hidden, void* y, float* mean, float* rstd, const void* x,
                              const void* gamma, const void* beta, int64_t rows, float eps,
                              int grid, int sms, cudaStream_t st) {
    const bool pre = rows <= kSmallCallRows;
    NF_HIDDEN_SWITCH(hidden, {
        static int occ[2] = {0, 0};
        const auto k = kLnFwdShifted ? (pre ? layernorm_fwd_shift<H, true> : layernorm_fwd_shift<H, false>)
                                     : (pre ? layernorm_fwd_reg<H, true> : layernorm_fwd_reg<H, false>);
        const int threads = pre ? Geo<H, true>::TPR * Geo<H, true>::RPC : Geo<H>::TPR * Geo<H>::RPC;
        return launch_with_pdl(k, dim3(grid), dim3(threads), 0, st, static_cast<uint16_t*>(y), mean,
                               rstd, static_cast<const uint16_t*>(x),
                               static_cast<const uint16_t*>(gamma), static_cast<const uint16_t*>(beta),
                               rows, eps, first_wave_ctas(k, threads, sms, &occ[pre]));
    })
}

}  // namespace nf
