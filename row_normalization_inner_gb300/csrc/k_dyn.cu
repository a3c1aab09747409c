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
// Backward kernels run a persistent grid of one wave (the CTAs that stay
// resident); CTA b owns the contiguous row stripe [rows * b / G,
// rows * (b + 1) / G) and one column-partial slot, as in the static-size
// backward kernels, and the same fixed-order column reduction finishes
// dgamma/dbeta (or dw).  Each thread streams its vectors of the next row
// through a per-thread cp.async ring in shared memory while it reduces the
// current one, and the arithmetic runs on packed fp32 pairs.  Measured on
// GB300 at 16384 rows against one-row-at-a-time loads in registers and a
// grid sized for 1024 threads per SM (two waves): RMSNorm backward 6144
// 151.7 -> 99.5 us, fused-add backward 6144 276.8 -> 123.4 us, LayerNorm
// backward 1000 50.1 -> 29.7 us.
#include "common.cuh"
#include "pdl.cuh"
#include "pairs.cuh"
#include "launch.h"

namespace nf {

namespace {

constexpr int kDynMaxWarps = 32;
constexpr int kDynMaxV = 4;          // vectors per thread (a 1024-thread CTA covers hidden 32768)
constexpr int kDynBwdMaxT = 512;     // backward CTAs keep column accumulators: at most 512 threads

// Backward copy ring: each thread copies its own vectors of the row ahead
// of the one it computes into kDynBwdStages stages of dynamic shared memory
// (16-byte cp.async, layout [stage][tensor][vector][thread]; the tensors
// are x, dy and, for the fused-add backward, the residual-stream
// gradient), so a row's loads are in flight while the row before it is
// reduced.  A thread only reads what it copied, so cp.async.wait_group is
// the only synchronization.  Two stages measured as fast as three or
// faster, with half the shared memory.
constexpr int kDynBwdStages = 2;
constexpr int kDynFwdStages = 2;  // the forward ring (RMSNorm and LayerNorm)

__device__ __forceinline__ void dyn_cp16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void dyn_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void dyn_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Sum N values over the CTA; every thread gets the totals (fixed order).
// `red` holds kDynMaxWarps * N floats and is private to this call site and
// row parity; the caller keeps a trailing __syncthreads before reuse.
template <int N>
__device__ __forceinline__ void cta_sum(float (&v)[N], float* red) {
    warp_sum<N>(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (nw == 1) {
        // one warp: its shuffle totals are the CTA's; 0 + v keeps the bits of
        // the loop below (a -0 total becomes +0).  Rows of one warp at 16384
        // rows: 3-9 % faster (LayerNorm forward 264 10.1 -> 9.3 us, RMSNorm
        // backward 24 12.8 -> 12.0 us)
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] = 0.f + v[i];
        return;
    }
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
// the CTA size (so small rows keep a large register budget).  LayerNorm
// makes one reduction per row: the sums of d = x - c and d^2, with c the
// row's first element (read by every thread; one cached line), give
// mean = c + sum d / H and M2 = sum d^2 - (sum d)^2 / H.  The arithmetic
// runs on packed fp32 pairs (16384 x 3072 LayerNorm 35.5 -> 34.7 us,
// RMSNorm 14336 161.4 -> 156.8 us against scalar fp32).
//
// A CTA takes one row at a time with plain loads, the grid as large as the
// rows, so the hardware keeps as many rows in flight per SM as CTAs fit.
// Rows of one warp (hidden up to 1024: 32 threads of four vectors) hit the
// limit of 32 resident CTAs per SM, so the forward ops then run RING (when
// the row's inputs are at most 2 KB, see dyn_fwd_smem): one wave of resident
// CTAs that walk rows blockIdx.x, + gridDim.x, ... and
// stream each thread's vectors of the row ahead (x, and for the fused op
// the residual) through a per-thread cp.async ring (kDynFwdStages stages
// of dynamic shared memory, layout [stage][tensor][vector][thread]) while
// the current row is reduced (16384 x 1000: RMSNorm 17.3 -> 14.0 us,
// LayerNorm 17.3 -> 15.7 us).  For wider rows the ring measured slower
// than one CTA per row (LayerNorm 16384 x 3072: 43.2 against 34.5 us, with
// two or three stages).

// One row of the forward once this thread's vectors are in registers:
// v0 = x (fused: plus v1 = the residual), c = LayerNorm's shift.
template <int OP, int MAXV>
__device__ __forceinline__ void dyn_fwd_row(const DynArgs& a, int64_t row, const uint4 (&v0)[MAXV],
                                            const uint4 (&v1)[MAXV], float c, float* red) {
    const int H = a.hidden;
    const int NV = H / kVec;
    const int T = blockDim.x, t = threadIdx.x;
    const float invH = 1.0f / static_cast<float>(H);
    float2 f[MAXV][4];
    float2 p1 = make_float2(0.f, 0.f), p2 = make_float2(0.f, 0.f);
    const float2 nc2 = make_float2(-c, -c);
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
        unpack8x2(v0[k], f[k]);  // zero vectors beyond the row add nothing
        if constexpr (OP == 0) {
            float2 b[4];
            unpack8x2(v1[k], b);
#pragma unroll
            for (int q = 0; q < 4; ++q) f[k][q] = __fadd2_rn(f[k][q], b[q]);
        }
        if constexpr (OP == 2) {
            if (k * T + t < NV) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 d = __fadd2_rn(f[k][q], nc2);
                    p1 = __fadd2_rn(p1, d);
                    p2 = __ffma2_rn(d, d, p2);
                }
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) p1 = __ffma2_rn(f[k][q], f[k][q], p1);
        }
    }
    float sv[2] = {p1.x + p1.y, p2.x + p2.y};
    float mean = 0.f, rstd;
    if constexpr (OP == 2) {
        cta_sum<2>(sv, red);
        const float dm = sv[0] * invH;
        mean = c + dm;
        rstd = rsqrtf(fmaxf(sv[1] - sv[0] * dm, 0.f) * invH + a.eps);
    } else {
        float s1[1] = {sv[0]};
        cta_sum<1>(s1, red);
        rstd = rsqrtf(s1[0] * invH + a.eps);
    }
    const float2 rstd2 = make_float2(rstd, rstd), nmean2 = make_float2(-mean, -mean);
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
        const int v = k * T + t;
        if (v < NV) {
            if constexpr (OP == 0) st_stream(a.out1 + row * H + v * kVec, pack8x2(f[k]));
            float2 g[4], o[4];
            unpack8x2(ld_param(a.p0 + v * kVec), g);
            if constexpr (OP == 2) {
                float2 b[4];
                unpack8x2(ld_param(a.p1 + v * kVec), b);
#pragma unroll
                for (int q = 0; q < 4; ++q)  // (x - mean) (rstd gamma) + beta: a constant row gives beta
                    o[q] = __ffma2_rn(__fadd2_rn(f[k][q], nmean2), __fmul2_rn(rstd2, g[q]), b[q]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = __fmul2_rn(__fmul2_rn(f[k][q], rstd2), g[q]);
            }
            st_stream(a.out0 + row * H + v * kVec, pack8x2(o));
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

template <int OP, int MAXV, int MAXT, bool RING>
__global__ void __launch_bounds__(MAXT, 1024 / MAXT) norm_dyn_fwd(DynArgs a) {
    __shared__ float red[kDynMaxWarps * 2];
    grid_dep_wait();
    grid_dep_release();
    const int H = a.hidden;
    const int NV = H / kVec;
    const int T = blockDim.x, t = threadIdx.x;
    if constexpr (!RING) {
        for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
            uint4 v0[MAXV], v1[MAXV];
            const float c = OP == 2 ? __uint_as_float(static_cast<uint32_t>(__ldg(a.in0 + row * H)) << 16) : 0.f;
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
            dyn_fwd_row<OP, MAXV>(a, row, v0, v1, c, red);
        }
    } else {
        constexpr int S = kDynFwdStages;
        constexpr int NT = OP == 0 ? 2 : 1;              // x (and the residual)
        extern __shared__ __align__(16) uint4 fring[];  // [S][NT][MAXV][T]
        const int64_t G = gridDim.x;
        const auto slot = [&](int st, int tsr, int k) { return fring + ((st * NT + tsr) * MAXV + k) * T + t; };
        // one commit group per row: this thread's vectors (empty past the end)
        const auto issue = [&](int64_t r, int st) {
            if (r < a.rows) {
#pragma unroll
                for (int k = 0; k < MAXV; ++k) {
                    const int v = k * T + t;
                    if (v < NV) {
                        dyn_cp16(slot(st, 0, k), a.in0 + r * H + v * kVec);
                        if constexpr (OP == 0) dyn_cp16(slot(st, 1, k), a.in1 + r * H + v * kVec);
                    }
                }
            }
            dyn_commit();
        };
        // LayerNorm's shift (the row's first element), fetched one row ahead
        const auto shift = [&](int64_t r) {
            return OP == 2 && r < a.rows
                       ? __uint_as_float(static_cast<uint32_t>(__ldg(a.in0 + r * H)) << 16) : 0.f;
        };
#pragma unroll
        for (int i = 0; i < S - 1; ++i) issue(blockIdx.x + i * G, i);
        float c_next = shift(blockIdx.x);
        int it = 0;
        for (int64_t row = blockIdx.x; row < a.rows; row += G, ++it) {
            const float c = c_next;
            c_next = shift(row + G);
            issue(row + (S - 1) * G, (it + S - 1) % S);
            dyn_wait<S - 1>();
            const int st = it % S;
            uint4 v0[MAXV], v1[MAXV];
#pragma unroll
            for (int k = 0; k < MAXV; ++k) {
                const bool in = k * T + t < NV;
                v0[k] = in ? *slot(st, 0, k) : make_uint4(0, 0, 0, 0);
                v1[k] = OP == 0 && in ? *slot(st, NT - 1, k) : make_uint4(0, 0, 0, 0);
            }
            dyn_fwd_row<OP, MAXV>(a, row, v0, v1, c, red);
        }
        dyn_wait<0>();  // only empty groups remain
    }
}

// OP: 3 LayerNorm backward, 4 RMSNorm backward (rstd recomputed from x).
// MAXV is the vectors per thread (dyn_bwd_vecs): 1 for rows of at most 256
// vectors, 2 up to 768, else 4.  The launch bound guarantees 1024 resident
// threads per SM with one vector, 768 with two (at most 384 threads, two
// CTAs) and 512 with four (dyn_bwd_per_sm).
template <int OP, int MAXV, bool ADD>
__global__ void __launch_bounds__(MAXV == 2 ? 384 : kDynBwdMaxT, MAXV == 4 ? 1 : 2) norm_dyn_bwd(DynArgs a) {
    constexpr int NP = OP == 3 ? 2 : 1;  // partial planes
    // The LayerNorm backward with four vectors per thread (OP 3, MAXV 4)
    // reads gamma again (through L1) where it is used instead of holding it:
    // that frees the registers its two planes of column sums need (128
    // registers and a spill -> 106 and none; 16384 x 8200 / 14336: 265 / 333
    // -> 218 / 277 us).  Elsewhere the reload cost more than it saved
    // (RMSNorm 16384 x 8200: 170 -> 272 us): the copy ring leaves L1 little
    // room.
    constexpr int NT = ADD ? 3 : 2;      // tensors in the ring
    __shared__ float red[2][kDynMaxWarps * 2];
    grid_dep_wait();
    const int H = a.hidden;
    const int NV = H / kVec;
    const int T = blockDim.x, t = threadIdx.x;
    const float invH = 1.0f / static_cast<float>(H);
    const int64_t G = gridDim.x;
    const int64_t r0 = a.rows * blockIdx.x / G, r1 = a.rows * (blockIdx.x + 1) / G;

    // the arithmetic runs on packed fp32 pairs (add / mul / fma .f32x2),
    // which halves the floating-point instructions of this issue-bound loop
    uint4 pv[MAXV];
    float2 acc0[MAXV][4], acc1[NP == 2 ? MAXV : 1][4];
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
        const int v = k * T + t;
        pv[k] = v < NV ? ld_param(a.p0 + v * kVec) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc0[k][q] = make_float2(0.f, 0.f);
            if constexpr (NP == 2) acc1[k][q] = make_float2(0.f, 0.f);
        }
    }
    constexpr int S = kDynBwdStages;
    extern __shared__ __align__(16) uint4 ring[];  // [S][NT][MAXV][T]
    const auto slot = [&](int st, int tsr, int k) { return ring + ((st * NT + tsr) * MAXV + k) * T + t; };
    // one commit group per row: its vectors of every tensor (empty past the stripe)
    const auto issue = [&](int64_t r, int st) {
        if (r < r1) {
#pragma unroll
            for (int k = 0; k < MAXV; ++k) {
                const int v = k * T + t;
                if (v < NV) {
                    dyn_cp16(slot(st, 0, k), a.in0 + r * H + v * kVec);
                    dyn_cp16(slot(st, 1, k), a.in1 + r * H + v * kVec);
                    if constexpr (ADD) dyn_cp16(slot(st, 2, k), a.add + r * H + v * kVec);
                }
            }
        }
        dyn_commit();
    };
#pragma unroll
    for (int i = 0; i < S - 1; ++i) issue(r0 + i, i);
    // LayerNorm's saved statistics, fetched one row ahead
    float mu_n = 0.f, rs_n = 0.f;
    if (OP == 3 && r0 < r1) {
        mu_n = __ldg(a.mean + r0);
        rs_n = __ldg(a.rstd + r0);
    }
    int it = 0;
    for (int64_t r = r0; r < r1; ++r, ++it) {
        // start the row S - 1 ahead (into the stage the previous row used),
        // then wait for this row's group
        issue(r + S - 1, (it + S - 1) % S);
        const float mu = mu_n, rs_in = rs_n;
        if (OP == 3 && r + 1 < r1) {
            mu_n = __ldg(a.mean + r + 1);
            rs_n = __ldg(a.rstd + r + 1);
        }
        dyn_wait<S - 1>();
        const int st = it % S;
        uint4 xv[MAXV], dv[MAXV];
#pragma unroll
        for (int k = 0; k < MAXV; ++k) {
            const bool in = k * T + t < NV;
            xv[k] = in ? *slot(st, 0, k) : make_uint4(0, 0, 0, 0);
            dv[k] = in ? *slot(st, 1, k) : make_uint4(0, 0, 0, 0);
        }
        const float2 nmu2 = make_float2(-mu, -mu), rsi2 = make_float2(rs_in, rs_in);
        float2 s0v = make_float2(0.f, 0.f), s1v = s0v;
#pragma unroll
        for (int k = 0; k < MAXV; ++k) {
            if (k * T + t < NV) {
                float2 xf[4], df[4], gf[4];
                unpack8x2(xv[k], xf);
                unpack8x2(dv[k], df);
                if constexpr (OP == 3 && MAXV == 4) unpack8x2(ld_param(a.p0 + (k * T + t) * kVec), gf);
                else unpack8x2(pv[k], gf);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (OP == 3) {
                        const float2 xh = __fmul2_rn(__fadd2_rn(xf[q], nmu2), rsi2);
                        const float2 g = __fmul2_rn(df[q], gf[q]);
                        s0v = __fadd2_rn(s0v, g);
                        s1v = __ffma2_rn(g, xh, s1v);
                        acc0[k][q] = __ffma2_rn(df[q], xh, acc0[k][q]);
                        acc1[k][q] = __fadd2_rn(acc1[k][q], df[q]);
                    } else {
                        s0v = __ffma2_rn(xf[q], xf[q], s0v);
                        s1v = __ffma2_rn(__fmul2_rn(df[q], gf[q]), xf[q], s1v);
                    }
                }
            }
        }
        float s[2] = {s0v.x + s0v.y, s1v.x + s1v.y};
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
        // LayerNorm: dx = rs dy w - rs A - (rs B) xhat; RMSNorm: dx = rs dy w - B x
        const float2 rs2 = make_float2(rs, rs);
        const float2 nra2 = make_float2(-rs * A, -rs * A);
        const float2 nb2 = OP == 3 ? make_float2(-rs * B, -rs * B) : make_float2(-B, -B);
#pragma unroll
        for (int k = 0; k < MAXV; ++k) {
            const int v = k * T + t;
            if (v < NV) {
                float2 xf[4], df[4], gf[4], o[4];
                if constexpr (MAXV >= 2) {
                    // read again from the ring (this row's stage is not refilled
                    // before the next iteration) instead of holding x and dy in
                    // registers across the row reduction: at 16384 rows LayerNorm
                    // backward 3072 / 6144 / 8200 / 14336 67.2 / 127.1 / 296 / 367
                    // -> 65.4 / 122.4 / 267 / 334.5 us, RMSNorm 14336 233.7 -> 215 us
                    // (LayerNorm 1000, one vector per thread: 27.8 -> 29.7 us, so
                    // one vector keeps them in registers)
                    unpack8x2(*slot(st, 0, k), xf);
                    unpack8x2(*slot(st, 1, k), df);
                } else {
                    unpack8x2(xv[k], xf);
                    unpack8x2(dv[k], df);
                }
                if constexpr (OP == 3 && MAXV == 4) unpack8x2(ld_param(a.p0 + (k * T + t) * kVec), gf);
                else unpack8x2(pv[k], gf);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 dw = __fmul2_rn(df[q], gf[q]);
                    if constexpr (OP == 3) {
                        const float2 xh = __fmul2_rn(__fadd2_rn(xf[q], nmu2), rs2);
                        o[q] = __ffma2_rn(xh, nb2, __ffma2_rn(rs2, dw, nra2));
                    } else {
                        o[q] = __ffma2_rn(xf[q], nb2, __fmul2_rn(rs2, dw));
                        acc0[k][q] = __ffma2_rn(__fmul2_rn(df[q], xf[q]), rs2, acc0[k][q]);
                    }
                }
                if constexpr (ADD) {  // fused-add backward: + the residual-stream gradient
                    float2 af[4];
                    unpack8x2(*slot(st, 2, k), af);
#pragma unroll
                    for (int q = 0; q < 4; ++q) o[q] = __fadd2_rn(o[q], af[q]);
                }
                st_stream(a.out0 + r * H + v * kVec, pack8x2(o));
            }
        }
    }
    dyn_wait<0>();  // only empty groups remain
    float* wp = a.ws + static_cast<int64_t>(blockIdx.x) * NP * H;
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
        const int v = k * T + t;
        if (v < NV) {
            float4* p0 = reinterpret_cast<float4*>(wp + v * kVec);
            p0[0] = make_float4(acc0[k][0].x, acc0[k][0].y, acc0[k][1].x, acc0[k][1].y);
            p0[1] = make_float4(acc0[k][2].x, acc0[k][2].y, acc0[k][3].x, acc0[k][3].y);
            if constexpr (NP == 2) {
                float4* p1 = reinterpret_cast<float4*>(wp + H + v * kVec);
                p1[0] = make_float4(acc1[k][0].x, acc1[k][0].y, acc1[k][1].x, acc1[k][1].y);
                p1[1] = make_float4(acc1[k][2].x, acc1[k][2].y, acc1[k][3].x, acc1[k][3].y);
            }
        }
    }
}

}  // namespace

// Vectors per thread of the backward kernel: one for rows of at most 256
// vectors, two up to 768, else four.  Measured on GB300 at 16384 rows (graph-timed):
// hidden 1000 LayerNorm backward 50.1 -> 32.6 us with one vector against
// four; from hidden 2560 up four were faster (RMSNorm 3072: 61.7 against
// 90.1 us), as a CTA then keeps more of a row in flight per thread.
//
// Two vectors per thread from 257 to 768 vectors: twice the threads per row
// and half the column sums per thread (75-79 registers, no spill, against
// 128 and a spill for the LayerNorm backward with four).  At 16384 rows:
// LayerNorm backward 2560 / 3072 / 4000 / 6144: 71.2 / 78.3 / 103.2 / 164.3
// -> 58.4 / 66.9 / 81.6 / 126.4 us; RMSNorm backward 1 % faster; fused-add
// backward 3072 / 4000: 68.4 / 88.8 -> 65.4 / 83.7 us (2560: 56.0 -> 58.0).
int dyn_bwd_vecs(int64_t nv) { return nv <= 256 ? 1 : nv <= 768 ? 2 : kDynMaxV; }

// Threads per CTA for a runtime hidden size, or false if the op has no
// dynamic kernel for it.  Forward: four vectors per thread; backward: see
// dyn_bwd_vecs.
bool dyn_shape(int op, int64_t hidden, int* threads) {
    if (hidden < kVec || hidden % kVec != 0) return false;
    const int64_t nv = hidden / kVec;
    const bool bwd = op == 3 || op == 4;
    const int64_t maxt = bwd ? kDynBwdMaxT : 1024;
    if (nv > maxt * kDynMaxV) return false;
    const int vecs = bwd ? dyn_bwd_vecs(nv) : kDynMaxV;
    int64_t t = (nv + vecs - 1) / vecs;
    t = (t + 31) / 32 * 32;
    *threads = static_cast<int>(t < 32 ? 32 : t);
    return true;
}

// Dynamic shared memory of the backward kernel: its copy ring.
size_t dyn_bwd_smem(int64_t hidden, bool add) {
    int t;
    if (!dyn_shape(3, hidden, &t)) return 0;
    return static_cast<size_t>(kDynBwdStages) * (add ? 3 : 2) * dyn_bwd_vecs(hidden / kVec) * t * 16;
}

// Resident CTAs per SM of the backward kernel: what its launch bound
// guarantees (1024 threads per SM with one vector per thread, 768 with two,
// 512 with four),
// and what its ring leaves room for (228 KB of shared memory per SM, 1 KB
// of it reserved per CTA, plus the kernel's static reduction buffer).
int dyn_bwd_per_sm(int64_t hidden, bool add) {
    int t;
    if (!dyn_shape(3, hidden, &t)) return 1;
    const int vecs = dyn_bwd_vecs(hidden / kVec);
    int per_sm = (vecs == 1 ? 1024 : vecs == 2 ? 768 : 512) / t;
    const size_t cta = dyn_bwd_smem(hidden, add) + 1024 + 2 * kDynMaxWarps * 2 * sizeof(float);
    const int by_smem = static_cast<int>((228 * 1024) / cta);
    if (by_smem < per_sm) per_sm = by_smem;
    return per_sm > 0 ? per_sm : 1;
}

// Dynamic shared memory of the forward kernel: the copy ring on rows of one
// warp whose inputs are at most 2 KB (x, and for the fused op the residual:
// hidden up to 512 there), else 0 (one CTA per row, no ring).  The fused op
// at 16384 x 264 took 17.0 -> 9.65 us on the ring, at 16384 x 1000
// 21.4 -> 24.1 us: with 4 KB of inputs per row one CTA per row already
// keeps enough in flight, and two-tensor rings fit only 24 CTAs per SM.
size_t dyn_fwd_smem(int op, int64_t hidden) {
    int t;
    if (op < 0 || op > 2 || !dyn_shape(op, hidden, &t) || t != 32) return 0;
    if ((op == 0 ? 2 : 1) * hidden * 2 > 2048) return 0;
    return static_cast<size_t>(kDynFwdStages) * (op == 0 ? 2 : 1) * kDynMaxV * t * 16;
}

// Resident CTAs per SM of the forward kernel on the ring: the launch bound
// keeps 1024 threads per SM, the ring takes shared memory (228 KB per SM,
// 1 KB reserved per CTA, plus the static reduction buffer), and an SM holds
// at most 32 CTAs.
int dyn_fwd_per_sm(int op, int64_t hidden) {
    int t;
    if (!dyn_shape(op, hidden, &t)) return 1;
    int per_sm = 1024 / t;
    const size_t cta = dyn_fwd_smem(op, hidden) + 1024 + kDynMaxWarps * 2 * sizeof(float);
    const int by_smem = static_cast<int>((228 * 1024) / cta);
    if (by_smem < per_sm) per_sm = by_smem;
    if (per_sm > 32) per_sm = 32;
    return per_sm > 0 ? per_sm : 1;
}

int64_t dyn_max_hidden(int op) {
    return static_cast<int64_t>((op == 3 || op == 4) ? kDynBwdMaxT : 1024) * kDynMaxV * kVec;
}

// Opt the backward kernels into their ring's shared memory, once per device.
cudaError_t dyn_bwd_attrs() {
    constexpr int kMaxDev = 64;
    static bool done[kMaxDev] = {};
    int dev;
    if (cudaError_t e = cudaGetDevice(&dev)) return e;
    if (dev >= 0 && dev < kMaxDev && done[dev]) return cudaSuccess;
    constexpr int most = kDynBwdStages * 3 * kDynMaxV * kDynBwdMaxT * 16;
    static_assert(most <= 227 * 1024, "the largest ring fits a CTA");
    const auto set = [](auto k) { return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, most); };
    cudaError_t e = set(norm_dyn_bwd<3, 1, false>);
    if (!e) e = set(norm_dyn_bwd<3, kDynMaxV, false>);
    if (!e) e = set(norm_dyn_bwd<4, 1, false>);
    if (!e) e = set(norm_dyn_bwd<4, kDynMaxV, false>);
    if (!e) e = set(norm_dyn_bwd<4, 1, true>);
    if (!e) e = set(norm_dyn_bwd<4, kDynMaxV, true>);
    if (!e) e = set(norm_dyn_bwd<3, 2, false>);
    if (!e) e = set(norm_dyn_bwd<4, 2, false>);
    if (!e) e = set(norm_dyn_bwd<4, 2, true>);
    if (!e && dev >= 0 && dev < kMaxDev) done[dev] = true;
    return e;
}

cudaError_t launch_dyn(int op, const DynArgs& a, int grid, cudaStream_t st) {
    int threads;
    if (!dyn_shape(op, a.hidden, &threads)) return cudaErrorInvalidValue;
    const bool big = threads > 256;
    const dim3 g(grid), b(threads);
    const size_t ring = dyn_fwd_smem(op, a.hidden);  // > 0: one-warp rows on the ring
    switch (op) {
        case 0:
            if (ring) return launch_with_pdl(norm_dyn_fwd<0, kDynMaxV, 256, true>, g, b, ring, st, a);
            return big ? launch_with_pdl(norm_dyn_fwd<0, kDynMaxV, 1024, false>, g, b, 0, st, a)
                       : launch_with_pdl(norm_dyn_fwd<0, kDynMaxV, 256, false>, g, b, 0, st, a);
        case 1:
            if (ring) return launch_with_pdl(norm_dyn_fwd<1, kDynMaxV, 256, true>, g, b, ring, st, a);
            return big ? launch_with_pdl(norm_dyn_fwd<1, kDynMaxV, 1024, false>, g, b, 0, st, a)
                       : launch_with_pdl(norm_dyn_fwd<1, kDynMaxV, 256, false>, g, b, 0, st, a);
        case 2:
            if (ring) return launch_with_pdl(norm_dyn_fwd<2, kDynMaxV, 256, true>, g, b, ring, st, a);
            return big ? launch_with_pdl(norm_dyn_fwd<2, kDynMaxV, 1024, false>, g, b, 0, st, a)
                       : launch_with_pdl(norm_dyn_fwd<2, kDynMaxV, 256, false>, g, b, 0, st, a);
        case 3:
        case 4: {
            const int v = dyn_bwd_vecs(a.hidden / kVec);
            const bool add = op == 4 && a.add != nullptr;
            const size_t smem = dyn_bwd_smem(a.hidden, add);
            if (cudaError_t e = dyn_bwd_attrs()) return e;
            if (op == 3)
                return v == 1 ? launch_with_pdl(norm_dyn_bwd<3, 1, false>, g, b, smem, st, a)
                     : v == 2 ? launch_with_pdl(norm_dyn_bwd<3, 2, false>, g, b, smem, st, a)
                              : launch_with_pdl(norm_dyn_bwd<3, kDynMaxV, false>, g, b, smem, st, a);
            if (add)
                return v == 1 ? launch_with_pdl(norm_dyn_bwd<4, 1, true>, g, b, smem, st, a)
                     : v == 2 ? launch_with_pdl(norm_dyn_bwd<4, 2, true>, g, b, smem, st, a)
                              : launch_with_pdl(norm_dyn_bwd<4, kDynMaxV, true>, g, b, smem, st, a);
            return v == 1 ? launch_with_pdl(norm_dyn_bwd<4, 1, false>, g, b, smem, st, a)
                 : v == 2 ? launch_with_pdl(norm_dyn_bwd<4, 2, false>, g, b, smem, st, a)
                          : launch_with_pdl(norm_dyn_bwd<4, kDynMaxV, false>, g, b, smem, st, a);
        }
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nf
