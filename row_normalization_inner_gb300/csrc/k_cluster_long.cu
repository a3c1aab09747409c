// Grid-parallel inner normalization for long rows: one row split across a
// thread-block cluster, with a runtime hidden size.  The "Llu/ln bwd"
// discussion lists "grid-parallel inner normalization" among the
// normalization variants and notes it does not exist yet; here it covers
// rows too long for one CTA (forward hidden above 32768 up to 262144,
// backward above 16384 up to 131072), and any other multiple of 8 when the
// cluster family is forced.
//
// CTA `rank` of a C-CTA cluster owns vectors [rank * slice, rank * slice +
// slice) of the row (slice = ceil(NV / C), NV = hidden / 8); thread t holds
// vectors rank * slice + k * T + t, k < 4, predicated.  Row sums: warp
// shuffles, a fixed-order sum over the CTA's warps, then every CTA reads
// the C partials through distributed shared memory in rank order (so all C
// CTAs hold the same total).  Partial slots alternate with the row parity
// and a final cluster barrier keeps each CTA's shared memory alive until
// its peers have read it.
//
// Backward: persistent clusters; cluster c owns the row stripe
// [rows * c / NC, rows * (c + 1) / NC) and partial slot c, each CTA writing
// its own column slice of the slot; the fixed-order column reduction
// finishes dgamma/dbeta (or dw).
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace nf {
namespace {

constexpr int kLongV = 4;            // vectors per thread
constexpr int kLongFwdMaxT = 1024;
constexpr int kLongBwdMaxT = 512;
constexpr int kLongMaxC = 8;         // portable cluster size

template <int N>
__device__ __forceinline__ void block_sum(float (&v)[N], float* red) {
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

// Block sums of N values, published in `part` (N floats of this CTA's
// shared memory), then summed over the cluster in rank order.
template <int N>
__device__ __forceinline__ void cluster_total(float (&v)[N], float* red, float* part,
                                              cg::cluster_group& cl) {
    block_sum<N>(v, red);
    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i) part[i] = v[i];
    }
    cl.sync();
    const int C = static_cast<int>(cl.num_blocks());
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = 0.f;
    for (int r = 0; r < C; ++r) {
        const float* pr = cl.map_shared_rank(part, r);
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] += pr[i];
    }
}

// OP: 0 fused add + RMSNorm, 1 RMSNorm fwd, 2 LayerNorm fwd
template <int OP>
__global__ void __launch_bounds__(kLongFwdMaxT) norm_long_fwd(DynArgs a, int slice) {
    __shared__ float red[2][32];
    __shared__ float part[2][2];  // [row parity][round]
    cg::cluster_group cl = cg::this_cluster();
    const int C = static_cast<int>(cl.num_blocks());
    const int rank = static_cast<int>(cl.block_rank());
    const int H = a.hidden, NV = H / kVec, T = blockDim.x, t = threadIdx.x;
    const int vbeg = rank * slice;
    const int vend = min(NV, vbeg + slice);
    const float invH = 1.0f / static_cast<float>(H);
    int iter = 0;
    for (int64_t row = blockIdx.x / C; row < a.rows; row += gridDim.x / C, ++iter) {
        float f[kLongV][8];
        float s1[1] = {0.f};
#pragma unroll
        for (int k = 0; k < kLongV; ++k) {
            const int v = vbeg + k * T + t;
            uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
            if (v < vend) {
                x0 = ld_stream(a.in0 + row * H + v * kVec);
                if constexpr (OP == 0) x1 = ld_stream(a.in1 + row * H + v * kVec);
            }
            unpack8(x0, f[k]);
            if constexpr (OP == 0) {
                float b[8];
                unpack8(x1, b);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[k][e] += b[e];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) s1[0] += (OP == 2) ? f[k][e] : f[k][e] * f[k][e];
        }
        cluster_total<1>(s1, red[0], &part[iter & 1][0], cl);
        float mean = 0.f, rstd;
        if constexpr (OP == 2) {
            mean = s1[0] * invH;
            float s2[1] = {0.f};
#pragma unroll
            for (int k = 0; k < kLongV; ++k) {
                if (vbeg + k * T + t < vend) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float d = f[k][e] - mean;
                        s2[0] += d * d;
                    }
                }
            }
            cluster_total<1>(s2, red[1], &part[iter & 1][1], cl);
            rstd = rsqrtf(s2[0] * invH + a.eps);
        } else {
            rstd = rsqrtf(s1[0] * invH + a.eps);
        }
#pragma unroll
        for (int k = 0; k < kLongV; ++k) {
            const int v = vbeg + k * T + t;
            if (v < vend) {
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
            if (rank == 0 && t == 0) {
                if (a.mean) a.mean[row] = mean;
                if (a.rstd) a.rstd[row] = rstd;
            }
        }
        __syncthreads();  // `red` is reused by the next row
    }
    cl.sync();  // no CTA leaves while a peer may still read its `part`
}

// OP: 3 LayerNorm backward (saved mean/rstd), 4 RMSNorm backward (rstd recomputed)
template <int OP>
__global__ void __launch_bounds__(kLongBwdMaxT) norm_long_bwd(DynArgs a, int slice) {
    constexpr int NP = OP == 3 ? 2 : 1;
    __shared__ float red[2][64];
    __shared__ float part[2][2];
    cg::cluster_group cl = cg::this_cluster();
    const int C = static_cast<int>(cl.num_blocks());
    const int rank = static_cast<int>(cl.block_rank());
    const int H = a.hidden, NV = H / kVec, T = blockDim.x, t = threadIdx.x;
    const int vbeg = rank * slice;
    const int vend = min(NV, vbeg + slice);
    const float invH = 1.0f / static_cast<float>(H);
    const int64_t NC = gridDim.x / C, cid = blockIdx.x / C;
    const int64_t r0 = a.rows * cid / NC, r1 = a.rows * (cid + 1) / NC;

    uint4 pv[kLongV];
    float acc0[kLongV][8], acc1[NP == 2 ? kLongV : 1][8];
#pragma unroll
    for (int k = 0; k < kLongV; ++k) {
        const int v = vbeg + k * T + t;
        pv[k] = v < vend ? ld_param(a.p0 + v * kVec) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc0[k][e] = 0.f;
        if constexpr (NP == 2) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc1[k][e] = 0.f;
        }
    }
    int it = 0;
    for (int64_t r = r0; r < r1; ++r, ++it) {
        uint4 xv[kLongV], dv[kLongV];
#pragma unroll
        for (int k = 0; k < kLongV; ++k) {
            const int v = vbeg + k * T + t;
            xv[k] = make_uint4(0, 0, 0, 0);
            dv[k] = make_uint4(0, 0, 0, 0);
            if (v < vend) {
                xv[k] = ld_stream(a.in0 + r * H + v * kVec);
                dv[k] = ld_stream(a.in1 + r * H + v * kVec);
            }
        }
        const float mu = OP == 3 ? __ldg(a.mean + r) : 0.f;
        const float rs_in = OP == 3 ? __ldg(a.rstd + r) : 0.f;
        float s[2] = {0.f, 0.f};
#pragma unroll
        for (int k = 0; k < kLongV; ++k) {
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
        cluster_total<2>(s, red[it & 1], part[it & 1], cl);
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
        for (int k = 0; k < kLongV; ++k) {
            const int v = vbeg + k * T + t;
            if (v < vend) {
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
    float* wp = a.ws + cid * NP * H;
#pragma unroll
    for (int k = 0; k < kLongV; ++k) {
        const int v = vbeg + k * T + t;
        if (v < vend) {
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
    cl.sync();  // no CTA leaves while a peer may still read its `part`
}

template <typename Kernel>
cudaError_t launch_in_clusters(Kernel k, int c, int threads, int grid, cudaStream_t st,
                               const DynArgs& a, int slice) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(c);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a, slice);
}

}  // namespace

bool long_shape(int op, int64_t hidden, int* ctas, int* threads, int* slice) {
    if (hidden < kVec || hidden % kVec != 0) return false;
    const int64_t nv = hidden / kVec;
    const int64_t maxt = (op == 3 || op == 4) ? kLongBwdMaxT : kLongFwdMaxT;
    for (int c = 2; c <= kLongMaxC; c *= 2) {
        const int64_t sl = (nv + c - 1) / c;
        int64_t t = (sl + kLongV - 1) / kLongV;
        t = (t + 31) / 32 * 32;
        if (t < 32) t = 32;
        if (t <= maxt) {
            *ctas = c;
            *threads = static_cast<int>(t);
            *slice = static_cast<int>(sl);
            return true;
        }
    }
    return false;
}

int64_t long_max_hidden(int op) {
    return static_cast<int64_t>((op == 3 || op == 4) ? kLongBwdMaxT : kLongFwdMaxT) * kLongV *
           kVec * kLongMaxC;
}

cudaError_t launch_long(int op, const DynArgs& a, int grid, cudaStream_t st) {
    int c, threads, slice;
    if (!long_shape(op, a.hidden, &c, &threads, &slice)) return cudaErrorInvalidValue;
    switch (op) {
        case 0: return launch_in_clusters(norm_long_fwd<0>, c, threads, grid, st, a, slice);
        case 1: return launch_in_clusters(norm_long_fwd<1>, c, threads, grid, st, a, slice);
        case 2: return launch_in_clusters(norm_long_fwd<2>, c, threads, grid, st, a, slice);
        case 3: return launch_in_clusters(norm_long_bwd<3>, c, threads, grid, st, a, slice);
        case 4: return launch_in_clusters(norm_long_bwd<4>, c, threads, grid, st, a, slice);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nf
