// Runtime-hidden ("dynamic block dimension") kernels: any hidden that is a
// multiple of 8, up to a per-op maximum.  "TMA inner persistent scheduler"
// (NVIDIA/Fuser PR #5587, description) adds manual scheduling for dynamic
// block dimensions beside the static-size path of "optimize inner
// persistent scheduler for static fusion"; this is that counterpart here.
//
// The hidden size is a kernel argument.  A CTA of T threads (a multiple of
// 32, chosen on the host so that T * MAXV covers the row's NV = hidden / 8
// vectors) owns one row at a time; thread t holds vectors v = k * T + t for
// k < MAXV, predicated on v < NV, so the row still stays in registers
// (MAXV is a compile-time bound, which keeps the per-thread arrays in
// registers).  Reductions: warp shuffles, then a fixed-order sum over the
// CTA's warps through shared memory.
//
// Backward kernels run a persistent grid; CTA b owns the contiguous row
// stripe [rows * b / G, rows * (b + 1) / G) and one column-partial slot, as
// in the static-size backward kernels, and the same fixed-order column
// reduction finishes dgamma/dbeta (or dw).
#include "common.cuh"
#include "pdl.cuh"
#include "launch.h"

namespace nf {

namespace {

constexpr int kDynMaxWarps = 32;
constexpr int kDynMaxV = 4;          // vectors per thread (a 1024-thread CTA covers hidden 32768)
constexpr int kDynBwdMaxT = 512;     // backward CTAs keep column accumulators: at most 512 threads

// Sum N values over the CTA; every thread gets the totals (fixed order).
// `red` holds kDynMaxWarps * N floats and is private to this call site and
// row parity; the caller keeps a trailing __syncthreads before reuse.
template <int N>
__device__ __forceinline__ void cta_sum(float (&v)[N], float* red) {
    warp_sum<N>(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i) red[warp * N + i] = v[i];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < N; ++i) {
        float s = 0.f;
        for (int w = 0; w < nw; ++w) s += red[w * N + i];
        v[i] = s;
    }
}

// OP: 0 fused add + RMSNorm, 1 RMSNorm fwd, 2 LayerNorm fwd.  MAXT bounds
// the CTA size (so small rows keep a large register budget).
template <int OP, int MAXV, int MAXT>
__global__ void __launch_bounds__(MAXT) norm_dyn_fwd(DynArgs a) {
    __shared__ float red[2][kDynMaxWarps];
    grid_dep_wait();
    grid_dep_release();
    const int H = a.hidden;
    const int NV = H / kVec;
    const int T = blockDim.x, t = threadIdx.x;
    const float invH = 1.0f / static_cast<float>(H);
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        uint4 v0[MAXV], v1[MAXV];
        float s1[1] = {0.f};
#pragma unroll
        for (int k = 0; k < MAXV; ++k) {
            const int v = k * T + t;
            v0[k] = make_uint4(0, 0, 0, 0);
            v1[k] = make_uint4(0, 0, 0, 0);
            if (v < NV) {
                v0[k] = ld_stream(a.in0 + row * H + v * kVec);
                if constexpr (OP == 0) v1[k] = ld_stream(a.in1 + row * H + v * kVec);
            }
        }
        float f[MAXV][8];
#pragma unroll
        for (int k = 0; k < MAXV; ++k) {
            unpack8(v0[k], f[k]);  // zero vectors beyond the row add nothing
            if constexpr (OP == 0) {
                float b[8];
                unpack8(v1[k], b);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[k][e] += b[e];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) s1[0] += (OP == 2) ? f[k][e] : f[k][e] * f[k][e];
        }
        cta_sum<1>(s1, red[0]);
        float mean = 0.f, rstd;
        if constexpr (OP == 2) {
            mean = s1[0] * invH;
            float s2[1] = {0.f};
#pragma unroll
            for (int k = 0; k < MAXV; ++k) {
                if (k * T + t < NV) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float d = f[k][e] - mean;
                        s2[0] += d * d;
                    }
                }
            }
            cta_sum<1>(s2, red[1]);
            rstd = rsqrtf(s2[0] * invH + a.eps);
        } else {
            rstd = rsqrtf(s1[0] * invH + a.eps);
        }
#pragma unroll
        for (int k = 0; k < MAXV; ++k) {
            const int v = k * T + t;
            if (v < NV) {
                if constexpr (OP == 0) st_stream(a.out1 + row * H + v * kVec, pack8(f[k]));
                float g[8], o[8];
                unpack8(ld_param(a.p0 + v * kVec), g);
                if constexpr (OP == 2) {
                    float b[8];
                    unpack8(ld_param(a.p1 + v * kVec), b);
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = (f[k][e] - mean) * rstd * g[e] + b[e];
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = f[k][e] * rstd * g[e];
                }
                st_stream(a.out0 + row * H + v * kVec, pack8(o));
            }
        }
        if constexpr (OP == 2) {
            if (t == 0) {
                if (a.mean) a.mean[row] = mean;
                if (a.rstd) a.rstd[row] = rstd;
            }
        }
        __syncthreads();  // `red` is reused by the next row
    }
}

// OP: 3 LayerNorm backward, 4 RMSNorm backward (rstd recomputed from x)
template <int OP, int MAXV>
__global__ void __launch_bounds__(kDynBwdMaxT) norm_dyn_bwd(DynArgs a) {
    constexpr int NP = OP == 3 ? 2 : 1;  // partial planes
    __shared__ float red[2][kDynMaxWarps * 2];
    grid_dep_wait();
    const int H = a.hidden;
    const int NV = H / kVec;
    const int T = blockDim.x, t = threadIdx.x;
    const float invH = 1.0f / static_cast<float>(H);
    const int64_t G = gridDim.x;
    const int64_t r0 = a.rows * blockIdx.x / G, r1 = a.rows * (blockIdx.x + 1) / G;

    uint4 pv[MAXV];
    float acc0[MAXV][8], acc1[NP == 2 ? MAXV : 1][8];
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
        const int v = k * T + t;
        pv[k] = v < NV ? ld_param(a.p0 + v * kVec) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc0[k][e] = 0.f;
        if constexpr (NP == 2) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc1[k][e] = 0.f;
        }
    }
    int it = 0;
    for (int64_t r = r0; r < r1; ++r, ++it) {
        uint4 xv[MAXV], dv[MAXV];
#pragma unroll
        for (int k = 0; k < MAXV; ++k) {
            const int v = k * T + t;
            xv[k] = make_uint4(0, 0, 0, 0);
            dv[k] = make_uint4(0, 0, 0, 0);
            if (v < NV) {
                xv[k] = ld_stream(a.in0 + r * H + v * kVec);
                dv[k] = ld_stream(a.in1 + r * H + v * kVec);
            }
        }
        const float mu = OP == 3 ? __ldg(a.mean + r) : 0.f;
        const float rs_in = OP == 3 ? __ldg(a.rstd + r) : 0.f;
        float s[2] = {0.f, 0.f};
#pragma unroll
        for (int k = 0; k < MAXV; ++k) {
            if (k * T + t < NV) {
                float xf[8], df[8], gf[8];
                unpack8(xv[k], xf);
                unpack8(dv[k], df);
                unpack8(pv[k], gf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if constexpr (OP == 3) {
                        const float xh = (xf[e] - mu) * rs_in;
                        const float g = df[e] * gf[e];
                        s[0] += g;
                        s[1] += g * xh;
                        acc0[k][e] += df[e] * xh;
                        acc1[k][e] += df[e];
                    } else {
                        s[0] += xf[e] * xf[e];
                        s[1] += df[e] * gf[e] * xf[e];
                    }
                }
            }
        }
        cta_sum<2>(s, red[it & 1]);
        float rs, A, B;
        if constexpr (OP == 3) {
            rs = rs_in;
            A = s[0] * invH;
            B = s[1] * invH;
        } else {
            rs = rsqrtf(s[0] * invH + a.eps);
            A = 0.f;
            B = rs * rs * rs * s[1] * invH;
        }
#pragma unroll
        for (int k = 0; k < MAXV; ++k) {
            const int v = k * T + t;
            if (v < NV) {
                float xf[8], df[8], gf[8], o[8];
                unpack8(xv[k], xf);
                unpack8(dv[k], df);
                unpack8(pv[k], gf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if constexpr (OP == 3) {
                        const float xh = (xf[e] - mu) * rs;
                        o[e] = rs * (df[e] * gf[e] - A - xh * B);
                    } else {
                        o[e] = rs * df[e] * gf[e] - xf[e] * B;
                        acc0[k][e] += df[e] * xf[e] * rs;
                    }
                }
                if (OP == 4 && a.add) {  // fused-add backward: + the residual-stream gradient
                    float af[8];
                    unpack8(ld_stream(a.add + r * H + v * kVec), af);
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] += af[e];
                }
                st_stream(a.out0 + r * H + v * kVec, pack8(o));
            }
        }
    }
    float* wp = a.ws + static_cast<int64_t>(blockIdx.x) * NP * H;
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
        const int v = k * T + t;
        if (v < NV) {
            float4* p0 = reinterpret_cast<float4*>(wp + v * kVec);
            p0[0] = make_float4(acc0[k][0], acc0[k][1], acc0[k][2], acc0[k][3]);
            p0[1] = make_float4(acc0[k][4], acc0[k][5], acc0[k][6], acc0[k][7]);
            if constexpr (NP == 2) {
                float4* p1 = reinterpret_cast<float4*>(wp + H + v * kVec);
                p1[0] = make_float4(acc1[k][0], acc1[k][1], acc1[k][2], acc1[k][3]);
                p1[1] = make_float4(acc1[k][4], acc1[k][5], acc1[k][6], acc1[k][7]);
            }
        }
    }
}

}  // namespace

// Threads per CTA and the per-thread vector bound for a runtime hidden
// size, or false if the op has no dynamic kernel for it.
bool dyn_shape(int op, int64_t hidden, int* threads) {
    if (hidden < kVec || hidden % kVec != 0) return false;
    const int64_t nv = hidden / kVec;
    const int64_t maxt = (op == 3 || op == 4) ? kDynBwdMaxT : 1024;
    if (nv > maxt * kDynMaxV) return false;
    int64_t t = (nv + kDynMaxV - 1) / kDynMaxV;
    t = (t + 31) / 32 * 32;
    *threads = static_cast<int>(t < 32 ? 32 : t);
    return true;
}

int64_t dyn_max_hidden(int op) {
    return static_cast<int64_t>((op == 3 || op == 4) ? kDynBwdMaxT : 1024) * kDynMaxV * kVec;
}

cudaError_t launch_dyn(int op, const DynArgs& a, int grid, cudaStream_t st) {
    int threads;
    if (!dyn_shape(op, a.hidden, &threads)) return cudaErrorInvalidValue;
    const bool big = threads > 256;
    const dim3 g(grid), b(threads);
    switch (op) {
        case 0:
            return big ? launch_with_pdl(norm_dyn_fwd<0, kDynMaxV, 1024>, g, b, 0, st, a)
                       : launch_with_pdl(norm_dyn_fwd<0, kDynMaxV, 256>, g, b, 0, st, a);
        case 1:
            return big ? launch_with_pdl(norm_dyn_fwd<1, kDynMaxV, 1024>, g, b, 0, st, a)
                       : launch_with_pdl(norm_dyn_fwd<1, kDynMaxV, 256>, g, b, 0, st, a);
        case 2:
            return big ? launch_with_pdl(norm_dyn_fwd<2, kDynMaxV, 1024>, g, b, 0, st, a)
                       : launch_with_pdl(norm_dyn_fwd<2, kDynMaxV, 256>, g, b, 0, st, a);
        case 3: return launch_with_pdl(norm_dyn_bwd<3, kDynMaxV>, g, b, 0, st, a);
        case 4: return launch_with_pdl(norm_dyn_bwd<4, kDynMaxV>, g, b, 0, st, a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nf
