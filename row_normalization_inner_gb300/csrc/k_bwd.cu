// LayerNorm backward: the combined inner + outer reduction of "Llu/ln bwd"
// (NVIDIA/Fuser PR #207, whose discussion treats the layer norm backward as
// the special case of a grid-parallel normalization that reduces both
// within rows and across them), with the cross-CTA partials kept in a
// workspace (the workspace support of "TMA inner persistent scheduler",
// description).
//
// Stage 1 (register path): `grid` persistent CTAs of RPC row groups.  Row
// group `slot` owns the contiguous row stripe
//     [rows * slot / nslots, rows * (slot + 1) / nslots),  nslots = grid * RPC,
// so which rows feed which partial depends only on (rows, nslots).  For each
// row it computes, with xhat = (x - mean) * rstd and g = dy * gamma,
//     inner:  A = sum_j g_j / H,  B = sum_j g_j xhat_j / H  (one row reduction of 2 values)
//             dx_j = rstd * (g_j - A - xhat_j * B)
//     outer:  acc_gamma_j += dy_j * xhat_j,  acc_beta_j += dy_j  (per-thread registers)
// and at the end writes its column partials to ws[slot][0][:], ws[slot][1][:].
// Stage 2 sums the nslots partials of every column in slot order, so dgamma
// and dbeta are bit-identical from run to run.
#include "common.cuh"
#include "pdl.cuh"
#include "launch.h"

namespace nf {
namespace {

template <int H>
struct BGeo {
    static constexpr int TPR = RegShape<H>::TPR;
    static constexpr int RPC = RegShape<H>::RPC;
    static constexpr int NV = H / kVec;
    static constexpr int VPT = NV / TPR;
    static constexpr int W = TPR / 32;
    static_assert(NV % TPR == 0 && TPR % 32 == 0, "static row split");
};

template <int H>
__global__ void __launch_bounds__(BGeo<H>::TPR * BGeo<H>::RPC)
layernorm_bwd_reg(uint16_t* dx, float* __restrict__ ws, const uint16_t* dy, const uint16_t* x,
                  const float* __restrict__ mean, const float* __restrict__ rstd,
                  const uint16_t* __restrict__ gamma, int64_t rows) {
    using G = BGeo<H>;
    __shared__ float red[2][G::RPC * G::W * 2];
    grid_dep_wait();
    const int group = threadIdx.x / G::TPR, t = threadIdx.x % G::TPR;
    const int64_t nslots = static_cast<int64_t>(gridDim.x) * G::RPC;
    const int64_t slot = static_cast<int64_t>(blockIdx.x) * G::RPC + group;
    const int64_t r0 = rows * slot / nslots;
    const int64_t r1 = rows * (slot + 1) / nslots;
    const int64_t maxlen = (rows + nslots - 1) / nslots;  // >= every stripe's length

    uint4 gm[G::VPT];
#pragma unroll
    for (int k = 0; k < G::VPT; ++k) gm[k] = ld_param(gamma + (k * G::TPR + t) * kVec);
    float acc_g[G::VPT][8], acc_b[G::VPT][8];
#pragma unroll
    for (int k = 0; k < G::VPT; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e) { acc_g[k][e] = 0.f; acc_b[k][e] = 0.f; }

    for (int64_t it = 0; it < maxlen; ++it) {
        const int64_t r = r0 + it;
        const bool active = r < r1;
        uint4 xv[G::VPT], dv[G::VPT];
        float mu = 0.f, rs = 0.f;
        float v[2] = {0.f, 0.f};
        if (active) {
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                const int vi = k * G::TPR + t;
                xv[k] = ld_stream(x + r * H + vi * kVec);
                dv[k] = ld_stream(dy + r * H + vi * kVec);
            }
            mu = __ldg(mean + r);
            rs = __ldg(rstd + r);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float xf[8], df[8], gf[8];
                unpack8(xv[k], xf);
                unpack8(dv[k], df);
                unpack8(gm[k], gf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float xh = (xf[e] - mu) * rs;
                    const float g = df[e] * gf[e];
                    v[0] += g;
                    v[1] += g * xh;
                    acc_g[k][e] += df[e] * xh;
                    acc_b[k][e] += df[e];
                }
            }
        }
        group_sum<G::TPR, 2>(v, red[it & 1], group, t);
        if (active) {
            const float A = v[0] * (1.0f / H);
            const float B = v[1] * (1.0f / H);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float xf[8], df[8], gf[8], o[8];
                unpack8(xv[k], xf);
                unpack8(dv[k], df);
                unpack8(gm[k], gf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float xh = (xf[e] - mu) * rs;
                    o[e] = rs * (df[e] * gf[e] - A - xh * B);
                }
                st_stream(dx + r * H + (k * G::TPR + t) * kVec, pack8(o));
            }
        }
    }

    float* wg = ws + slot * 2 * H;
    float* wb = wg + H;
#pragma unroll
    for (int k = 0; k < G::VPT; ++k) {
        const int j = (k * G::TPR + t) * kVec;
        float4* pg = reinterpret_cast<float4*>(wg + j);
        float4* pb = reinterpret_cast<float4*>(wb + j);
        pg[0] = make_float4(acc_g[k][0], acc_g[k][1], acc_g[k][2], acc_g[k][3]);
        pg[1] = make_float4(acc_g[k][4], acc_g[k][5], acc_g[k][6], acc_g[k][7]);
        pb[0] = make_float4(acc_b[k][0], acc_b[k][1], acc_b[k][2], acc_b[k][3]);
        pb[1] = make_float4(acc_b[k][4], acc_b[k][5], acc_b[k][6], acc_b[k][7]);
    }
}

// RMSNorm backward, stage 1 (register path), same stripes and slots as the
// LayerNorm kernel above.  rstd is recomputed from the resident row (one
// more sum in the same reduction), so the forward need not save it:
//     rstd = rsqrt(sum_j x_j^2 / H + eps),  g = dy * w,  P = sum_j g_j x_j
//     dx_j = rstd * g_j - x_j * rstd^3 * P / H     (= rstd * (g_j - xhat_j * mean(g * xhat)))
//     acc_w_j += dy_j * x_j * rstd                  -> ws[slot][0][:]
template <int H>
__global__ void __launch_bounds__(BGeo<H>::TPR * BGeo<H>::RPC)
rmsnorm_bwd_reg(uint16_t* dx, float* __restrict__ ws, const uint16_t* dy, const uint16_t* x,
                const uint16_t* dres, const uint16_t* __restrict__ w, int64_t rows, float eps) {
    using G = BGeo<H>;
    __shared__ float red[2][G::RPC * G::W * 2];
    grid_dep_wait();
    const int group = threadIdx.x / G::TPR, t = threadIdx.x % G::TPR;
    const int64_t nslots = static_cast<int64_t>(gridDim.x) * G::RPC;
    const int64_t slot = static_cast<int64_t>(blockIdx.x) * G::RPC + group;
    const int64_t r0 = rows * slot / nslots;
    const int64_t r1 = rows * (slot + 1) / nslots;
    const int64_t maxlen = (rows + nslots - 1) / nslots;

    uint4 wv[G::VPT];
#pragma unroll
    for (int k = 0; k < G::VPT; ++k) wv[k] = ld_param(w + (k * G::TPR + t) * kVec);
    float acc[G::VPT][8];
#pragma unroll
    for (int k = 0; k < G::VPT; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[k][e] = 0.f;

    for (int64_t it = 0; it < maxlen; ++it) {
        const int64_t r = r0 + it;
        const bool active = r < r1;
        uint4 xv[G::VPT], dv[G::VPT];
        float v[2] = {0.f, 0.f};
        if (active) {
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                const int vi = k * G::TPR + t;
                xv[k] = ld_stream(x + r * H + vi * kVec);
                dv[k] = ld_stream(dy + r * H + vi * kVec);
            }
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float xf[8], df[8], wf[8];
                unpack8(xv[k], xf);
                unpack8(dv[k], df);
                unpack8(wv[k], wf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    v[0] += xf[e] * xf[e];
                    v[1] += df[e] * wf[e] * xf[e];
                }
            }
        }
        group_sum<G::TPR, 2>(v, red[it & 1], group, t);
        if (active) {
            const float rs = rsqrtf(v[0] * (1.0f / H) + eps);
            const float c = rs * rs * rs * v[1] * (1.0f / H);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float xf[8], df[8], wf[8], o[8];
                unpack8(xv[k], xf);
                unpack8(dv[k], df);
                unpack8(wv[k], wf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    o[e] = rs * df[e] * wf[e] - xf[e] * c;
                    acc[k][e] += df[e] * xf[e] * rs;
                }
                if (dres) {  // fused-add backward: + the residual-stream gradient
                    float af[8];
                    unpack8(ld_stream(dres + r * H + (k * G::TPR + t) * kVec), af);
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] += af[e];
                }
                st_stream(dx + r * H + (k * G::TPR + t) * kVec, pack8(o));
            }
        }
    }

    float* wp = ws + slot * H;
#pragma unroll
    for (int k = 0; k < G::VPT; ++k) {
        const int j = (k * G::TPR + t) * kVec;
        reinterpret_cast<float4*>(wp + j)[0] = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
        reinterpret_cast<float4*>(wp + j)[1] = make_float4(acc[k][4], acc[k][5], acc[k][6], acc[k][7]);
    }
}

// out0[j] = sum_{slot} ws[slot][0][j] and, with two planes,
// out1[j] = sum_{slot} ws[slot][1][j], in a fixed order.  Each float4
// column gets Y slot lanes of one warp (Y = 16 or 32, so a warp covers
// 32 / Y columns): lane ly sums slots ly, ly + Y, ly + 2Y, ... in that
// order, issuing up to eight loads before it adds them, and the Y lane sums are
// combined by a shuffle butterfly.  Every butterfly step adds the same two
// values on both partner lanes, so all Y lanes end with the same bits and
// the result does not depend on the launch.  No shared memory and no CTA
// barrier: the reduction is a few loads deep plus log2(Y) shuffles.
constexpr int kColT = 64;  // two warps: many small CTAs spread the columns evenly over the SMs

template <int Y>
__global__ void __launch_bounds__(kColT, 16)
column_reduce(const float* __restrict__ ws, float* __restrict__ dgamma,
              float* __restrict__ dbeta, int nslots, int hidden, int planes) {
    static_assert(Y == 16 || Y == 32, "slot lanes per column");
    constexpr int CPW = 32 / Y;  // float4 columns per warp
    // Launched as a programmatic dependent of stage 1: wait until stage 1
    // has finished and its partials are visible (a no-op otherwise), then
    // let the next kernel in the stream be scheduled while this one runs.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ly = lane % Y, lx = lane / Y;
    const int64_t c4 = (static_cast<int64_t>(blockIdx.x) * (kColT / 32) + warp) * CPW + lx;
    const int64_t total4 = static_cast<int64_t>(planes) * hidden / 4;
    const bool ok = c4 < total4;
    const int which = ok ? static_cast<int>((c4 * 4) / hidden) : 0;
    const int64_t j = ok ? (c4 * 4) % hidden : 0;
    // slot p of this column is float4 number p * total4 + c4
    const float4* src = reinterpret_cast<const float4*>(ws) + (ok ? c4 : 0);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ok) {
        // up to kColU slots per lane are loaded before any is added, so a
        // lane waits for one L2 round trip per kColU slots (152 slots: one)
        constexpr int kColU = 8;
        for (int p0 = ly; p0 < nslots; p0 += kColU * Y) {
            float4 v[kColU];
#pragma unroll
            for (int u = 0; u < kColU; ++u) {
                const int p = p0 + u * Y;
                v[u] = p < nslots ? __ldcs(src + static_cast<int64_t>(p) * total4)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kColU; ++u) {
                if (p0 + u * Y < nslots) {
                    s.x += v[u].x; s.y += v[u].y; s.z += v[u].z; s.w += v[u].w;
                }
            }
        }
    }
#pragma unroll
    for (int off = Y / 2; off > 0; off >>= 1) {
        s.x += __shfl_xor_sync(0xFFFFFFFFu, s.x, off);
        s.y += __shfl_xor_sync(0xFFFFFFFFu, s.y, off);
        s.z += __shfl_xor_sync(0xFFFFFFFFu, s.z, off);
        s.w += __shfl_xor_sync(0xFFFFFFFFu, s.w, off);
    }
    if (ok && ly == 0) *reinterpret_cast<float4*>((which == 0 ? dgamma : dbeta) + j) = s;
}

// The same sums when there are many slots (> kWideSlots, the runtime-hidden
// backward's one slot per resident CTA): kSplitW warps per float4 column,
// warp w adding the contiguous slot range [n w / kSplitW, n (w + 1) /
// kSplitW) with 32 slot lanes as above, then the warps' totals added in
// warp order.  A lane then waits for one or two L2 round trips instead of
// n / 256, and four times as many warps share the work.
constexpr int kWideSlots = 256;
constexpr int kSplitW = 4;

__global__ void __launch_bounds__(kSplitW * 32)
column_reduce_split(const float* __restrict__ ws, float* __restrict__ dgamma,
                    float* __restrict__ dbeta, int nslots, int hidden, int planes) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float4 part[kSplitW];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t c4 = blockIdx.x;  // one float4 column per CTA
    const int64_t total4 = static_cast<int64_t>(planes) * hidden / 4;
    const int which = static_cast<int>((c4 * 4) / hidden);
    const int64_t j = (c4 * 4) % hidden;
    const float4* src = reinterpret_cast<const float4*>(ws) + c4;
    const int p_lo = static_cast<int>(static_cast<int64_t>(nslots) * warp / kSplitW);
    const int p_hi = static_cast<int>(static_cast<int64_t>(nslots) * (warp + 1) / kSplitW);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int kColU = 8;
    for (int p0 = p_lo + lane; p0 < p_hi; p0 += kColU * 32) {
        float4 v[kColU];
#pragma unroll
        for (int u = 0; u < kColU; ++u) {
            const int p = p0 + u * 32;
            v[u] = p < p_hi ? __ldcs(src + static_cast<int64_t>(p) * total4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kColU; ++u) {
            if (p0 + u * 32 < p_hi) {
                s.x += v[u].x; s.y += v[u].y; s.z += v[u].z; s.w += v[u].w;
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        s.x += __shfl_xor_sync(0xFFFFFFFFu, s.x, off);
        s.y += __shfl_xor_sync(0xFFFFFFFFu, s.y, off);
        s.z += __shfl_xor_sync(0xFFFFFFFFu, s.z, off);
        s.w += __shfl_xor_sync(0xFFFFFFFFu, s.w, off);
    }
    if (lane == 0) part[warp] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float4 t = part[0];
#pragma unroll
        for (int w = 1; w < kSplitW; ++w) {
            t.x += part[w].x; t.y += part[w].y; t.z += part[w].z; t.w += part[w].w;
        }
        *reinterpret_cast<float4*>((which == 0 ? dgamma : dbeta) + j) = t;
    }
}

// The same sums when there are few slots (<= kNarrowSlots): one float4
// column per thread, the slots added in order, so a CTA covers 1024
// contiguous columns (the wide form would leave at least half of each
// column's 16 slot lanes idle).
constexpr int kNarrowSlots = 8;
constexpr int kNarrowT = 256;

__global__ void __launch_bounds__(kNarrowT)
column_reduce_narrow(const float* __restrict__ ws, float* __restrict__ dgamma,
                     float* __restrict__ dbeta, int nslots, int hidden, int planes) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t c4 = static_cast<int64_t>(blockIdx.x) * kNarrowT + threadIdx.x;
    if (c4 * 4 >= planes * static_cast<int64_t>(hidden)) return;
    const int which = static_cast<int>((c4 * 4) / hidden);
    const int64_t j = (c4 * 4) % hidden;
    float4 s = __ldcs(reinterpret_cast<const float4*>(ws + static_cast<int64_t>(which) * hidden + j));
    for (int p = 1; p < nslots; ++p) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(
            ws + (static_cast<int64_t>(p) * planes + which) * hidden + j));
        s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    *reinterpret_cast<float4*>((which == 0 ? dgamma : dbeta) + j) = s;
}

}  // namespace

cudaError_t launch_ln_bwd_reg(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                              const float* mean, const float* rstd, const void* gamma,
                              int64_t rows, int grid, cudaStream_t st) {
    NF_HIDDEN_SWITCH(hidden, {
        return launch_with_pdl(layernorm_bwd_reg<H>, dim3(grid), dim3(BGeo<H>::TPR * BGeo<H>::RPC), 0,
                               st, static_cast<uint16_t*>(dx), ws, static_cast<const uint16_t*>(dy),
                               static_cast<const uint16_t*>(x), mean, rstd,
                               static_cast<const uint16_t*>(gamma), rows);
    })
}

// Stage 2 is launched with programmatic stream serialization: its launch
// overlaps the tail of stage 1, and the kernel's griddepcontrol.wait keeps
// every read after stage 1 has completed.
cudaError_t launch_column_reduce_planes(const float* ws, float* out0, float* out1, int nslots,
                                        int64_t hidden, int planes, cudaStream_t st) {
    const int64_t cols4 = planes * hidden / 4;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kColT, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (nslots <= kNarrowSlots) {
        cfg.gridDim = dim3(static_cast<unsigned>((cols4 + kNarrowT - 1) / kNarrowT), 1, 1);
        cfg.blockDim = dim3(kNarrowT, 1, 1);
        return cudaLaunchKernelEx(&cfg, column_reduce_narrow, ws, out0, out1, nslots,
                                  static_cast<int>(hidden), planes);
    }
    // slot lanes per column: 16 up to 64 slots (at most 4 loads a lane),
    // else 32
    const auto launch = [&](auto kernel, int y) {
        const int64_t per_cta = (kColT / 32) * (32 / y);  // float4 columns per CTA
        cfg.gridDim = dim3(static_cast<unsigned>((cols4 + per_cta - 1) / per_cta), 1, 1);
        return cudaLaunchKernelEx(&cfg, kernel, ws, out0, out1, nslots, static_cast<int>(hidden),
                                  planes);
    };
    if (nslots <= 64) return launch(column_reduce<16>, 16);
    if (nslots <= kWideSlots) return launch(column_reduce<32>, 32);
    cfg.gridDim = dim3(static_cast<unsigned>(cols4), 1, 1);
    cfg.blockDim = dim3(kSplitW * 32, 1, 1);
    return cudaLaunchKernelEx(&cfg, column_reduce_split, ws, out0, out1, nslots, static_cast<int>(hidden),
                              planes);
}

cudaError_t launch_column_reduce(const float* ws, float* dgamma, float* dbeta, int nslots,
                                 int64_t hidden, cudaStream_t st) {
    return launch_column_reduce_planes(ws, dgamma, dbeta, nslots, hidden, 2, st);
}

cudaError_t launch_column_reduce1(const float* ws, float* out, int nslots, int64_t hidden,
                                  cudaStream_t st) {
    return launch_column_reduce_planes(ws, out, nullptr, nslots, hidden, 1, st);
}

cudaError_t launch_rms_bwd_reg(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                               const void* dres, const void* w, int64_t rows, float eps, int grid,
                               cudaStream_t st) {
    NF_HIDDEN_SWITCH(hidden, {
        return launch_with_pdl(rmsnorm_bwd_reg<H>, dim3(grid), dim3(BGeo<H>::TPR * BGeo<H>::RPC), 0,
                               st, static_cast<uint16_t*>(dx), ws, static_cast<const uint16_t*>(dy),
                               static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(dres),
                               static_cast<const uint16_t*>(w), rows, eps);
    })
}

}  // namespace nf
