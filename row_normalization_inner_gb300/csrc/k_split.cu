// Grid-parallel inner normalization across any number of CTAs: a row is
// cut into chunks of 8192 elements, one CTA per (chunk, row), and the row
// statistics travel through global memory instead of a cluster's shared
// memory.  The "Llu/ln bwd" discussion names grid-parallel inner
// normalization as the missing normalization variant; the cluster kernels
// cover rows up to 8 CTAs, this family any length (the chunk count is not
// bounded by a cluster).
//
// Forward (fused add + RMSNorm, RMSNorm, LayerNorm), three launches:
//   1. split_stats: per (row, chunk) partial statistics -> part[row][chunk][2]
//      (RMS: sum of squares; LayerNorm: the chunk's mean and M2, two passes
//      over the chunk held in registers);
//   2. split_merge: one CTA per row merges its chunks in a fixed order
//      (thread t takes chunks t, t + 256, ..., then a fixed tree; Chan's
//      formula for LayerNorm) -> stat[row] = (mean, rstd);
//   3. split_apply: per (row, chunk) re-reads the chunk (from L2 when the
//      batch fits there) and writes the normalized output.
// The fused op reads x and residual in launches 1 and 3 and writes both in
// 3, so it normalizes the unrounded fp32 sum like every other family.
//
// Backward (LayerNorm, RMSNorm, fused-add RMSNorm), four launches: the row
// sums (LN: sum g, sum g * xhat; RMS: sum x^2, sum g * x) by (row, chunk),
// a per-row merge, then split_bwd_apply over (chunk, row block) CTAs that
// write dx and accumulate the column sums of their rows in registers (one
// workspace slot per row block), and the fixed-order column reduction.
//
// Every launch after the first is a programmatic dependent of the one
// before (griddepcontrol.wait before any read), and every sum runs in a
// fixed order, so results are deterministic.
#include "common.cuh"
#include "launch.h"

namespace nf {
namespace {

constexpr int kSpT = 256;                 // threads per CTA
constexpr int kSpV = 4;                   // vectors per thread
constexpr int kSpVecs = kSpT * kSpV;      // vectors per chunk
constexpr int kSpChunk = kSpVecs * kVec;  // elements per chunk
constexpr int kSpMaxGridY = 65535;

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Sum N values over the CTA (warp shuffles, then the 8 warps in order);
// every thread gets the totals.  `red` holds 8 * N floats; callers
// alternate two buffers between consecutive calls.
template <int N>
__device__ __forceinline__ void cta_sum(float (&v)[N], float* red) {
    warp_sum<N>(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i) red[warp * N + i] = v[i];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < N; ++i) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kSpT / 32; ++w) s += red[w * N + i];
        v[i] = s;
    }
}

struct Chan {
    float n, mean, m2;
};

__device__ __forceinline__ Chan chan_merge(Chan a, Chan b) {
    if (a.n == 0.f) return b;
    if (b.n == 0.f) return a;
    const float n = a.n + b.n;
    const float d = b.mean - a.mean;
    const float wb = b.n / n;
    return {n, a.mean + d * wb, a.m2 + b.m2 + d * d * a.n * wb};
}

// Elements of chunk c of a row of H elements.
__device__ __forceinline__ int chunk_len(int c, int H) {
    const int rest = H - c * kSpChunk;
    return rest < kSpChunk ? rest : kSpChunk;
}

// Load this thread's vectors of chunk c of row r, widened; invalid vectors
// are zero.  Vector k of thread t is chunk vector k * kSpT + t.  KEEP asks
// L2 to keep the lines (the statistics pass: the apply pass reads the same
// chunk again, from L2 when the batch fits there); otherwise the load
// streams (last use).
template <bool KEEP = false>
__device__ __forceinline__ void load_chunk(const uint16_t* src, int64_t r, int c, int H,
                                           float (&f)[kSpV][8]) {
    const int NV = H / kVec;
#pragma unroll
    for (int k = 0; k < kSpV; ++k) {
        const int v = c * kSpVecs + k * kSpT + threadIdx.x;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (v < NV) {
            const uint16_t* p = src + r * H + static_cast<int64_t>(v) * kVec;
            u = KEEP ? ld_keep(p) : ld_stream(p);
        }
        unpack8(u, f[k]);
    }
}

// Warm L2 with this thread's vectors of chunk c of row r (a hint, issued
// before waiting for the kernel ahead in the stream).
__device__ __forceinline__ void prefetch_chunk(const uint16_t* src, int64_t r, int c, int H) {
    const int NV = H / kVec;
#pragma unroll
    for (int k = 0; k < kSpV; ++k) {
        const int v = c * kSpVecs + k * kSpT + threadIdx.x;
        if (v < NV) prefetch_l2(src + r * H + static_cast<int64_t>(v) * kVec);
    }
}

// The apply passes take their (chunk, row) CTAs in the reverse of the
// statistics pass's order: the chunks the statistics pass read last are the
// ones still in L2 when the apply pass starts.
constexpr bool kSplitApplyLastFirst = true;

// ---- forward ----------------------------------------------------------------
// OP: 0 fused add + RMSNorm, 1 RMSNorm, 2 LayerNorm.
template <int OP>
__global__ void __launch_bounds__(kSpT) split_stats(DynArgs a, float* __restrict__ part, int nc) {
    __shared__ float red[(kSpT / 32) * 2];
    const int c = blockIdx.x, H = a.hidden;
    if (blockIdx.y < a.rows) {
        prefetch_chunk(a.in0, blockIdx.y, c, H);
        if (OP == 0) prefetch_chunk(a.in1, blockIdx.y, c, H);
    }
    pdl_wait();
    const int NV = H / kVec;
    for (int64_t r = blockIdx.y; r < a.rows; r += gridDim.y) {
        float f[kSpV][8];
        load_chunk<true>(a.in0, r, c, H, f);
        if constexpr (OP == 0) {
            float b[kSpV][8];
            load_chunk<true>(a.in1, r, c, H, b);
#pragma unroll
            for (int k = 0; k < kSpV; ++k)
#pragma unroll
                for (int e = 0; e < 8; ++e) f[k][e] += b[k][e];
        }
        float2 out;
        if constexpr (OP == 2) {
            // one reduction: the sums of d = x - K and d^2, K the chunk's first
            // element (every thread reads it; one cached line), give the
            // chunk's mean K + sum d / n and M2 = sum d^2 - (sum d)^2 / n
            const float K = __uint_as_float(static_cast<uint32_t>(
                                __ldg(a.in0 + r * H + static_cast<int64_t>(c) * kSpChunk)) << 16);
            float q[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < kSpV; ++k) {
                if (c * kSpVecs + k * kSpT + static_cast<int>(threadIdx.x) < NV) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float d = f[k][e] - K;
                        q[0] += d;
                        q[1] = fmaf(d, d, q[1]);
                    }
                }
            }
            cta_sum<2>(q, red);
            const float dm = q[0] / static_cast<float>(chunk_len(c, H));
            out = make_float2(K + dm, fmaxf(q[1] - q[0] * dm, 0.f));
        } else {
            float q[1] = {0.f};
#pragma unroll
            for (int k = 0; k < kSpV; ++k)
#pragma unroll
                for (int e = 0; e < 8; ++e) q[0] = fmaf(f[k][e], f[k][e], q[0]);
            cta_sum<1>(q, red);
            out = make_float2(q[0], 0.f);
        }
        if (threadIdx.x == 0) reinterpret_cast<float2*>(part)[r * nc + c] = out;
        __syncthreads();  // red is reused by the next row
    }
    // this CTA's partials are written: let the apply pass be scheduled (it
    // still waits for this grid to finish before reading them)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// LayerNorm forward: one CTA per row merges the row's chunk partials ->
// stat[row] = (mean, rstd) (Chan's pairwise update in a fixed order).  A
// separate launch measured faster for LayerNorm than every apply CTA
// repeating the Chan merge; RMSNorm merges inside the apply pass.
template <int OP>
__global__ void __launch_bounds__(kSpT) split_merge_fwd(DynArgs a, const float* __restrict__ part,
                                                        float2* __restrict__ stat, int nc) {
    __shared__ Chan sh[kSpT / 32];
    pdl_wait();
    const int H = a.hidden;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float2* p2 = reinterpret_cast<const float2*>(part);
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        Chan acc{0.f, 0.f, 0.f};
        for (int c = threadIdx.x; c < nc; c += kSpT) {
            const float2 p = __ldcg(p2 + r * nc + c);
            if constexpr (OP == 2) {
                acc = chan_merge(acc, Chan{static_cast<float>(chunk_len(c, H)), p.x, p.y});
            } else {
                acc.n = 1.f;
                acc.m2 += p.x;  // sum of squares
            }
        }
        // fixed tree: lanes, then warps in order
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const Chan o{__shfl_down_sync(0xffffffffu, acc.n, off),
                         __shfl_down_sync(0xffffffffu, acc.mean, off),
                         __shfl_down_sync(0xffffffffu, acc.m2, off)};
            if (lane < off) {
                if constexpr (OP == 2) {
                    acc = chan_merge(acc, o);
                } else {
                    acc.m2 += o.m2;
                }
            }
        }
        if (lane == 0) sh[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            Chan t = sh[0];
#pragma unroll
            for (int w = 1; w < kSpT / 32; ++w) {
                if constexpr (OP == 2) {
                    t = chan_merge(t, sh[w]);
                } else {
                    t.m2 += sh[w].m2;
                }
            }
            const float invH = 1.0f / static_cast<float>(H);
            const float rstd = rsqrtf(t.m2 * invH + a.eps);
            const float mean = OP == 2 ? t.mean : 0.f;
            stat[r] = make_float2(mean, rstd);
            if (OP == 2) {
                if (a.mean) a.mean[r] = mean;
                if (a.rstd) a.rstd[r] = rstd;
            }
        }
        __syncthreads();  // sh is reused by the next row
    }
}

// (mean, rstd) of row r from its nc chunk partials, merged by the whole CTA
// in a fixed order (thread t takes chunks t, t + 256, ..., then lanes and
// warps in a fixed tree), so every CTA that merges row r gets the same
// bits.  Every thread returns the result; `sh` is the CTA's scratch.
template <int OP>
__device__ __forceinline__ float2 merge_row_fwd(const DynArgs& a, const float* __restrict__ part,
                                                int64_t r, int nc, Chan* sh) {
    const int H = a.hidden;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float2* p2 = reinterpret_cast<const float2*>(part);
    Chan acc{0.f, 0.f, 0.f};
    for (int c = threadIdx.x; c < nc; c += kSpT) {
        const float2 p = __ldcg(p2 + r * nc + c);
        if constexpr (OP == 2) {
            acc = chan_merge(acc, Chan{static_cast<float>(chunk_len(c, H)), p.x, p.y});
        } else {
            acc.n = 1.f;
            acc.m2 += p.x;  // sum of squares
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const Chan o{__shfl_down_sync(0xffffffffu, acc.n, off),
                     __shfl_down_sync(0xffffffffu, acc.mean, off),
                     __shfl_down_sync(0xffffffffu, acc.m2, off)};
        if (lane < off) {
            if constexpr (OP == 2) {
                acc = chan_merge(acc, o);
            } else {
                acc.m2 += o.m2;
            }
        }
    }
    if (lane == 0) sh[warp] = acc;
    __syncthreads();
    Chan t = sh[0];
#pragma unroll
    for (int w = 1; w < kSpT / 32; ++w) {
        if constexpr (OP == 2) {
            t = chan_merge(t, sh[w]);
        } else {
            t.m2 += sh[w].m2;
        }
    }
    __syncthreads();  // sh is reused by the next row
    const float rstd = rsqrtf(t.m2 * (1.0f / static_cast<float>(H)) + a.eps);
    return make_float2(OP == 2 ? t.mean : 0.f, rstd);
}

// Apply pass.  RMSNorm (and the fused op) merge their row's chunk partials
// here (every CTA of the row does the same fixed-order merge), so their
// forward is two launches; LayerNorm reads `stat` from the merge launch.
template <int OP>
__global__ void __launch_bounds__(kSpT) split_apply_fwd(DynArgs a, const float* __restrict__ part,
                                                        const float2* __restrict__ stat, int nc) {
    __shared__ Chan sh[kSpT / 32];
    // CTAs take the grid last to first (see kSplitApplyLastFirst)
    const int c = kSplitApplyLastFirst ? gridDim.x - 1 - blockIdx.x : blockIdx.x, H = a.hidden;
    const int64_t rfirst = kSplitApplyLastFirst ? gridDim.y - 1 - blockIdx.y : blockIdx.y;
    if (rfirst < a.rows) {
        prefetch_chunk(a.in0, rfirst, c, H);
        if (OP == 0) prefetch_chunk(a.in1, rfirst, c, H);
    }
    pdl_wait();
    const int NV = H / kVec;
    for (int64_t r = rfirst; r < a.rows; r += gridDim.y) {
        float f[kSpV][8];
        load_chunk(a.in0, r, c, H, f);
        if constexpr (OP == 0) {
            float b[kSpV][8];
            load_chunk(a.in1, r, c, H, b);
#pragma unroll
            for (int k = 0; k < kSpV; ++k)
#pragma unroll
                for (int e = 0; e < 8; ++e) f[k][e] += b[k][e];
        }
        const float2 st = stat ? __ldcg(stat + r) : merge_row_fwd<OP>(a, part, r, nc, sh);
#pragma unroll
        for (int k = 0; k < kSpV; ++k) {
            const int v = c * kSpVecs + k * kSpT + threadIdx.x;
            if (v >= NV) continue;
            const int64_t off = r * H + static_cast<int64_t>(v) * kVec;
            float p[8], o[8];
            unpack8(ld_param(a.p0 + static_cast<int64_t>(v) * kVec), p);
            if constexpr (OP == 2) {
                float b[8];
                unpack8(ld_param(a.p1 + static_cast<int64_t>(v) * kVec), b);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = fmaf(f[k][e] - st.x, st.y * p[e], b[e]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = f[k][e] * st.y * p[e];
            }
            if constexpr (OP == 0) st_stream(a.out1 + off, pack8(f[k]));  // residual <- s
            st_stream(a.out0 + off, pack8(o));
        }
    }
}

// ---- backward -----------------------------------------------------------------
// OP: 3 LayerNorm (saved mean / rstd), 4 RMSNorm (rstd recomputed; a.add is
// the fused-add residual-stream gradient, or null).  in0 = x, in1 = dy.
template <int OP>
__global__ void __launch_bounds__(kSpT) split_stats_bwd(DynArgs a, float* __restrict__ part, int nc) {
    __shared__ float red[8 * 2];
    const int c = blockIdx.x, H = a.hidden;
    if (blockIdx.y < a.rows) {
        prefetch_chunk(a.in0, blockIdx.y, c, H);
        prefetch_chunk(a.in1, blockIdx.y, c, H);
    }
    pdl_wait();
    const int NV = H / kVec;
    for (int64_t r = blockIdx.y; r < a.rows; r += gridDim.y) {
        float x[kSpV][8], dy[kSpV][8];
        load_chunk<true>(a.in0, r, c, H, x);
        load_chunk<true>(a.in1, r, c, H, dy);
        const float mu = OP == 3 ? __ldg(a.mean + r) : 0.f;
        const float rs = OP == 3 ? __ldg(a.rstd + r) : 0.f;
        float s[2] = {0.f, 0.f};
#pragma unroll
        for (int k = 0; k < kSpV; ++k) {
            const int v = c * kSpVecs + k * kSpT + threadIdx.x;
            if (v >= NV) continue;
            float w[8];
            unpack8(ld_param(a.p0 + static_cast<int64_t>(v) * kVec), w);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float g = dy[k][e] * w[e];
                if constexpr (OP == 3) {
                    s[0] += g;
                    s[1] = fmaf(g, (x[k][e] - mu) * rs, s[1]);
                } else {
                    s[0] = fmaf(x[k][e], x[k][e], s[0]);
                    s[1] = fmaf(g, x[k][e], s[1]);
                }
            }
        }
        cta_sum<2>(s, red);
        if (threadIdx.x == 0) reinterpret_cast<float2*>(part)[r * nc + c] = make_float2(s[0], s[1]);
        __syncthreads();
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One CTA per row: stat[row] = LN (A, B) = (sum g / H, sum g xhat / H);
// RMS (rstd, rstd^3 * sum g x / H).
template <int OP>
__global__ void __launch_bounds__(kSpT) split_merge_bwd(DynArgs a, const float* __restrict__ part,
                                                        float2* __restrict__ stat, int nc) {
    __shared__ float red[8 * 2];
    pdl_wait();
    const float2* p2 = reinterpret_cast<const float2*>(part);
    const float invH = 1.0f / static_cast<float>(a.hidden);
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        float s[2] = {0.f, 0.f};
        for (int c = threadIdx.x; c < nc; c += kSpT) {
            const float2 p = __ldcg(p2 + r * nc + c);
            s[0] += p.x;
            s[1] += p.y;
        }
        cta_sum<2>(s, red);
        if (threadIdx.x == 0) {
            if constexpr (OP == 3) {
                stat[r] = make_float2(s[0] * invH, s[1] * invH);
            } else {
                const float rs = rsqrtf(s[0] * invH + a.eps);
                stat[r] = make_float2(rs, rs * rs * rs * s[1] * invH);
            }
        }
        __syncthreads();
    }
}

constexpr int kSpMergeRows = kSplitMergeRows;

// The per-row statistics of rows [r0, r0 + nrow) (nrow <= kSpMergeRows) from
// their chunk partials, into sh_stat[0 .. nrow): thread t adds chunks t,
// t + 256, ... of every row (all loads issued together), then lanes and
// warps are added in a fixed order, so every CTA of the row block gets the
// same bits.  LN: (A, B) = (sum g / H, sum g xhat / H); RMS: (rstd,
// rstd^3 * sum g x / H).
template <int OP>
__device__ __forceinline__ void merge_rows_bwd(const DynArgs& a, const float* __restrict__ part,
                                               int64_t r0, int nrow, int nc, float2* sh_stat,
                                               float* red) {
    const float2* p2 = reinterpret_cast<const float2*>(part);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float2 acc[kSpMergeRows];
#pragma unroll
    for (int i = 0; i < kSpMergeRows; ++i) acc[i] = make_float2(0.f, 0.f);
    for (int c = threadIdx.x; c < nc; c += kSpT) {
#pragma unroll
        for (int i = 0; i < kSpMergeRows; ++i) {
            if (i < nrow) {
                const float2 p = __ldcg(p2 + (r0 + i) * nc + c);
                acc[i].x += p.x;
                acc[i].y += p.y;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kSpMergeRows; ++i) {
        if (i < nrow) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                acc[i].x += __shfl_xor_sync(0xFFFFFFFFu, acc[i].x, off);
                acc[i].y += __shfl_xor_sync(0xFFFFFFFFu, acc[i].y, off);
            }
            if (lane == 0) {
                red[(warp * kSpMergeRows + i) * 2] = acc[i].x;
                red[(warp * kSpMergeRows + i) * 2 + 1] = acc[i].y;
            }
        }
    }
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < nrow) {
        const int i = threadIdx.x;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int w = 0; w < kSpT / 32; ++w) {
            s0 += red[(w * kSpMergeRows + i) * 2];
            s1 += red[(w * kSpMergeRows + i) * 2 + 1];
        }
        const float invH = 1.0f / static_cast<float>(a.hidden);
        if constexpr (OP == 3) {
            sh_stat[i] = make_float2(s0 * invH, s1 * invH);
        } else {
            const float rs = rsqrtf(s0 * invH + a.eps);
            sh_stat[i] = make_float2(rs, rs * rs * rs * s1 * invH);
        }
    }
    __syncthreads();
}

// Grid (chunks, row blocks): dx for the block's rows, and the block's column
// sums of its chunk -> ws[block][plane][H].  With `stat` null the block
// (at most kSpMergeRows rows) merges its rows' partials itself.
template <int OP>
__global__ void __launch_bounds__(kSpT) split_apply_bwd(DynArgs a, const float2* __restrict__ stat,
                                                        const float* __restrict__ part, int nc) {
    constexpr int NP = OP == 3 ? 2 : 1;
    __shared__ float2 sh_stat[kSpMergeRows];
    __shared__ float red[(kSpT / 32) * kSpMergeRows * 2];
    // CTAs take the grid last to first (see kSplitApplyLastFirst); row block
    // `blk` always feeds column-partial slot `blk`
    const int c = kSplitApplyLastFirst ? gridDim.x - 1 - blockIdx.x : blockIdx.x, H = a.hidden;
    const int NV = H / kVec;
    const int64_t nb = gridDim.y;
    const int64_t blk = kSplitApplyLastFirst ? nb - 1 - blockIdx.y : blockIdx.y;
    const int64_t r0 = a.rows * blk / nb, r1 = a.rows * (blk + 1) / nb;
    if (r0 < r1) {
        prefetch_chunk(a.in0, r0, c, H);
        prefetch_chunk(a.in1, r0, c, H);
    }
    pdl_wait();
    if (!stat) merge_rows_bwd<OP>(a, part, r0, static_cast<int>(r1 - r0), nc, sh_stat, red);
    float acc0[kSpV][8], acc1[NP == 2 ? kSpV : 1][8];
#pragma unroll
    for (int k = 0; k < kSpV; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            acc0[k][e] = 0.f;
            if constexpr (NP == 2) acc1[k][e] = 0.f;
        }
    for (int64_t r = r0; r < r1; ++r) {
        const float2 st = stat ? __ldcg(stat + r) : sh_stat[r - r0];
        float x[kSpV][8], dy[kSpV][8];
        load_chunk(a.in0, r, c, H, x);
        load_chunk(a.in1, r, c, H, dy);
        const float mu = OP == 3 ? __ldg(a.mean + r) : 0.f;
        const float rs = OP == 3 ? __ldg(a.rstd + r) : st.x;
#pragma unroll
        for (int k = 0; k < kSpV; ++k) {
            const int v = c * kSpVecs + k * kSpT + threadIdx.x;
            if (v >= NV) continue;
            const int64_t off = r * H + static_cast<int64_t>(v) * kVec;
            float w[8], o[8];
            unpack8(ld_param(a.p0 + static_cast<int64_t>(v) * kVec), w);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if constexpr (OP == 3) {
                    const float xh = (x[k][e] - mu) * rs;
                    o[e] = rs * (dy[k][e] * w[e] - st.x - xh * st.y);
                    acc0[k][e] = fmaf(dy[k][e], xh, acc0[k][e]);
                    acc1[k][e] += dy[k][e];
                } else {
                    o[e] = rs * dy[k][e] * w[e] - x[k][e] * st.y;
                    acc0[k][e] = fmaf(dy[k][e] * x[k][e], rs, acc0[k][e]);
                }
            }
            if (OP == 4 && a.add) {  // fused-add backward: + the residual-stream gradient
                float d[8];
                unpack8(ld_stream(a.add + off), d);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] += d[e];
            }
            st_stream(a.out0 + off, pack8(o));
        }
    }
    // one row block: the column sums are final and go straight to the outputs
    float* wp = a.ws + blk * NP * H;
    float* w0 = a.cols0 ? a.cols0 : wp;
    float* w1 = a.cols0 ? a.cols1 : wp + H;
#pragma unroll
    for (int k = 0; k < kSpV; ++k) {
        const int v = c * kSpVecs + k * kSpT + threadIdx.x;
        if (v >= NV) continue;
        float4* q0 = reinterpret_cast<float4*>(w0 + static_cast<int64_t>(v) * kVec);
        q0[0] = make_float4(acc0[k][0], acc0[k][1], acc0[k][2], acc0[k][3]);
        q0[1] = make_float4(acc0[k][4], acc0[k][5], acc0[k][6], acc0[k][7]);
        if constexpr (NP == 2) {
            float4* q1 = reinterpret_cast<float4*>(w1 + static_cast<int64_t>(v) * kVec);
            q1[0] = make_float4(acc1[k][0], acc1[k][1], acc1[k][2], acc1[k][3]);
            q1[1] = make_float4(acc1[k][4], acc1[k][5], acc1[k][6], acc1[k][7]);
        }
    }
}

// Backward apply ring: each thread copies its own vectors of the block's
// next row (x, dy and, for the fused-add backward, the residual-stream
// gradient) into a two-stage ring of dynamic shared memory with 16-byte
// cp.async, layout [stage][tensor][vector][thread], while it computes the
// current row.  A thread only reads what it copied, so
// cp.async.wait_group is the only synchronization.  The first row's copies
// are issued before the row merge, so they overlap it.
constexpr int kSpBwdStages = 2;

__device__ __forceinline__ void sp_cp16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void sp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void sp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <bool ADD>
constexpr int sp_bwd_ring_bytes() { return kSpBwdStages * (ADD ? 3 : 2) * kSpVecs * 16; }

// RMSNorm backward apply pass (ADD: the fused-add backward, whose
// residual-stream gradient is added to dx), the rows streamed through the
// copy ring above.  Grid and outputs as split_apply_bwd.  Against
// split_apply_bwd at 4 x 4194304: fused-add 47.9 -> 39.4 us, RMSNorm 36.9 ->
// 35.8 us; the LayerNorm backward, with more arithmetic per element, was
// slower through the ring (42.6 -> 45.8 us) and keeps split_apply_bwd.
template <bool ADD>
__global__ void __launch_bounds__(kSpT) split_apply_bwd_ring(DynArgs a, const float2* __restrict__ stat,
                                                             const float* __restrict__ part, int nc) {
    constexpr int OP = 4;
    constexpr int NP = OP == 3 ? 2 : 1;
    constexpr int NT = ADD ? 3 : 2;
    constexpr int S = kSpBwdStages;
    extern __shared__ __align__(16) uint4 sp_ring[];  // [S][NT][kSpV][kSpT]
    __shared__ float2 sh_stat[kSpMergeRows];
    __shared__ float red[(kSpT / 32) * kSpMergeRows * 2];
    // CTAs take the grid last to first (see kSplitApplyLastFirst); row block
    // `blk` always feeds column-partial slot `blk`
    const int c = kSplitApplyLastFirst ? gridDim.x - 1 - blockIdx.x : blockIdx.x, H = a.hidden;
    const int NV = H / kVec;
    const int64_t nb = gridDim.y;
    const int64_t blk = kSplitApplyLastFirst ? nb - 1 - blockIdx.y : blockIdx.y;
    const int64_t r0 = a.rows * blk / nb, r1 = a.rows * (blk + 1) / nb;
    if (r0 < r1) {
        prefetch_chunk(a.in0, r0, c, H);
        prefetch_chunk(a.in1, r0, c, H);
    }
    const auto slot = [&](int st, int tsr, int k) {
        return sp_ring + ((st * NT + tsr) * kSpV + k) * kSpT + threadIdx.x;
    };
    // one commit group per row (empty past the block)
    const auto issue = [&](int64_t r, int st) {
        if (r < r1) {
#pragma unroll
            for (int k = 0; k < kSpV; ++k) {
                const int v = c * kSpVecs + k * kSpT + threadIdx.x;
                if (v < NV) {
                    const int64_t off = r * H + static_cast<int64_t>(v) * kVec;
                    sp_cp16(slot(st, 0, k), a.in0 + off);
                    sp_cp16(slot(st, 1, k), a.in1 + off);
                    if constexpr (ADD) sp_cp16(slot(st, 2, k), a.add + off);
                }
            }
        }
        sp_commit();
    };
    pdl_wait();
    issue(r0, 0);
    if (!stat) merge_rows_bwd<OP>(a, part, r0, static_cast<int>(r1 - r0), nc, sh_stat, red);
    uint4 wv[kSpV];
    float acc0[kSpV][8], acc1[NP == 2 ? kSpV : 1][8];
#pragma unroll
    for (int k = 0; k < kSpV; ++k) {
        const int v = c * kSpVecs + k * kSpT + threadIdx.x;
        wv[k] = v < NV ? ld_param(a.p0 + static_cast<int64_t>(v) * kVec) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            acc0[k][e] = 0.f;
            if constexpr (NP == 2) acc1[k][e] = 0.f;
        }
    }
    // LayerNorm's saved statistics, fetched one row ahead
    float mu_n = 0.f, rs_n = 0.f;
    if (OP == 3 && r0 < r1) {
        mu_n = __ldg(a.mean + r0);
        rs_n = __ldg(a.rstd + r0);
    }
    int it = 0;
    for (int64_t r = r0; r < r1; ++r, ++it) {
        uint4 xv[kSpV], dv[kSpV];
        issue(r + 1, (it + 1) % S);  // into the stage the previous row used
        const float mu = mu_n, rs_saved = rs_n;
        if (OP == 3 && r + 1 < r1) {
            mu_n = __ldg(a.mean + r + 1);
            rs_n = __ldg(a.rstd + r + 1);
        }
        const int st_i = it % S;
        sp_wait<S - 1>();
#pragma unroll
        for (int k = 0; k < kSpV; ++k) {
            xv[k] = *slot(st_i, 0, k);
            dv[k] = *slot(st_i, 1, k);
        }
        const float2 st = stat ? __ldcg(stat + r) : sh_stat[r - r0];
        const float rs = OP == 3 ? rs_saved : st.x;
#pragma unroll
        for (int k = 0; k < kSpV; ++k) {
            const int v = c * kSpVecs + k * kSpT + threadIdx.x;
            if (v >= NV) continue;
            const int64_t off = r * H + static_cast<int64_t>(v) * kVec;
            float x[8], dy[8], w[8], o[8];
            unpack8(xv[k], x);
            unpack8(dv[k], dy);
            unpack8(wv[k], w);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if constexpr (OP == 3) {
                    const float xh = (x[e] - mu) * rs;
                    o[e] = rs * (dy[e] * w[e] - st.x - xh * st.y);
                    acc0[k][e] = fmaf(dy[e], xh, acc0[k][e]);
                    acc1[k][e] += dy[e];
                } else {
                    o[e] = rs * dy[e] * w[e] - x[e] * st.y;
                    acc0[k][e] = fmaf(dy[e] * x[e], rs, acc0[k][e]);
                }
            }
            if constexpr (ADD) {  // fused-add backward: + the residual-stream gradient
                float d[8];
                unpack8(*slot(st_i, 2, k), d);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] += d[e];
            }
            st_stream(a.out0 + off, pack8(o));
        }
    }
    sp_wait<0>();  // only empty groups remain
    // one row block: the column sums are final and go straight to the outputs
    float* wp = a.ws + blk * NP * H;
    float* w0 = a.cols0 ? a.cols0 : wp;
    float* w1 = a.cols0 ? a.cols1 : wp + H;
#pragma unroll
    for (int k = 0; k < kSpV; ++k) {
        const int v = c * kSpVecs + k * kSpT + threadIdx.x;
        if (v >= NV) continue;
        float4* q0 = reinterpret_cast<float4*>(w0 + static_cast<int64_t>(v) * kVec);
        q0[0] = make_float4(acc0[k][0], acc0[k][1], acc0[k][2], acc0[k][3]);
        q0[1] = make_float4(acc0[k][4], acc0[k][5], acc0[k][6], acc0[k][7]);
        if constexpr (NP == 2) {
            float4* q1 = reinterpret_cast<float4*>(w1 + static_cast<int64_t>(v) * kVec);
            q1[0] = make_float4(acc1[k][0], acc1[k][1], acc1[k][2], acc1[k][3]);
            q1[1] = make_float4(acc1[k][4], acc1[k][5], acc1[k][6], acc1[k][7]);
        }
    }
}

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel k, dim3 grid, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kSpT);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

// The RMSNorm backward apply pass: its copy ring in dynamic shared memory
// (set once per kernel), launched as a programmatic dependent.
template <bool ADD>
cudaError_t launch_apply_bwd_ring(const DynArgs& a, const float2* stat, const float* part, int nc, int rb,
                                  cudaStream_t st) {
    constexpr int smem = sp_bwd_ring_bytes<ADD>();
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaError_t e = cudaFuncSetAttribute(split_apply_bwd_ring<ADD>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem))
            return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nc, rb);
    cfg.blockDim = dim3(kSpT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_apply_bwd_ring<ADD>, a, stat, part, nc);
}

size_t align16(size_t b) { return (b + 15) / 16 * 16; }

// Workspace layout: [column partials (backward)] [part rows x nc x 2] [stat rows x 2].
struct SplitLayout {
    size_t cols, part, stat, total;
};

SplitLayout split_layout(int op, int64_t rows, int64_t hidden, int sms) {
    int nc = 0, rb = 0;
    split_shape(op, rows, hidden, sms, &nc, &rb);
    const bool bwd = op == 3 || op == 4;
    SplitLayout l{};
    l.cols = bwd ? align16(static_cast<size_t>(rb) * (op == 3 ? 2 : 1) * hidden * sizeof(float)) : 0;
    l.part = align16(static_cast<size_t>(rows) * nc * 2 * sizeof(float));
    l.stat = align16(static_cast<size_t>(rows) * 2 * sizeof(float));
    l.total = l.cols + l.part + l.stat;
    return l;
}

template <int OP>
cudaError_t fwd_t(const DynArgs& a, char* ws, int sms, cudaStream_t st) {
    int nc, rb;
    split_shape(OP, a.rows, a.hidden, sms, &nc, &rb);
    const SplitLayout l = split_layout(OP, a.rows, a.hidden, sms);
    float* part = reinterpret_cast<float*>(ws + l.cols);
    float2* stat = reinterpret_cast<float2*>(ws + l.cols + l.part);
    const unsigned gy = static_cast<unsigned>(a.rows < kSpMaxGridY ? a.rows : kSpMaxGridY);
    const unsigned gr = static_cast<unsigned>(a.rows < 0x7FFFFFFF ? a.rows : 0x7FFFFFFF);
    if (cudaError_t e = launch_pdl(split_stats<OP>, dim3(nc, gy), st, a, part, nc)) return e;
    if constexpr (OP == 2) {
        if (cudaError_t e = launch_pdl(split_merge_fwd<OP>, dim3(gr), st, a,
                                       static_cast<const float*>(part), stat, nc))
            return e;
        return launch_pdl(split_apply_fwd<OP>, dim3(nc, gy), st, a, static_cast<const float*>(part),
                          static_cast<const float2*>(stat), nc);
    }
    return launch_pdl(split_apply_fwd<OP>, dim3(nc, gy), st, a, static_cast<const float*>(part),
                      static_cast<const float2*>(nullptr), nc);
}

template <int OP>
cudaError_t bwd_t(DynArgs a, char* ws, int sms, cudaStream_t st) {
    int nc, rb;
    split_shape(OP, a.rows, a.hidden, sms, &nc, &rb);
    const SplitLayout l = split_layout(OP, a.rows, a.hidden, sms);
    a.ws = reinterpret_cast<float*>(ws);
    float* part = reinterpret_cast<float*>(ws + l.cols);
    float2* stat = reinterpret_cast<float2*>(ws + l.cols + l.part);
    const unsigned gy = static_cast<unsigned>(a.rows < kSpMaxGridY ? a.rows : kSpMaxGridY);
    const unsigned gr = static_cast<unsigned>(a.rows < 0x7FFFFFFF ? a.rows : 0x7FFFFFFF);
    if (cudaError_t e = launch_pdl(split_stats_bwd<OP>, dim3(nc, gy), st, a, part, nc)) return e;
    // row blocks short enough merge their rows' statistics themselves
    const bool merge_in_apply = (a.rows + rb - 1) / rb <= kSpMergeRows;
    if (!merge_in_apply) {
        if (cudaError_t e = launch_pdl(split_merge_bwd<OP>, dim3(gr), st, a,
                                       static_cast<const float*>(part), stat, nc))
            return e;
    }
    const float2* sv = merge_in_apply ? nullptr : static_cast<const float2*>(stat);
    if constexpr (OP == 4) {
        return a.add ? launch_apply_bwd_ring<true>(a, sv, part, nc, rb, st)
                     : launch_apply_bwd_ring<false>(a, sv, part, nc, rb, st);
    } else {
        return launch_pdl(split_apply_bwd<OP>, dim3(nc, rb), st, a, sv, static_cast<const float*>(part), nc);
    }
}

}  // namespace

bool split_shape(int op, int64_t rows, int64_t hidden, int sms, int* nchunks, int* rblocks) {
    if (hidden < kVec || hidden % kVec != 0 || hidden > kSplitMaxHidden) return false;
    const int64_t nc = (hidden + kSpChunk - 1) / kSpChunk;
    int64_t rb = 0;
    if (op == 3 || op == 4) {
        // about two CTAs per SM over (chunk, row block); every row block
        // adds a column-partial slot of planes x hidden fp32, so no more
        // blocks than that
        rb = (2LL * sms + nc - 1) / nc;
        if (rb > rows) rb = rows;
        if (rb > kSpMaxGridY) rb = kSpMaxGridY;
        if (rb < 1) rb = 1;
    }
    *nchunks = static_cast<int>(nc);
    *rblocks = static_cast<int>(rb);
    return true;
}

size_t split_workspace_bytes(int op, int64_t rows, int64_t hidden, int sms) {
    if (rows <= 0 || hidden < kVec || hidden % kVec != 0 || hidden > kSplitMaxHidden) return 0;
    return split_layout(op, rows, hidden, sms).total;
}

// a.out0 / out1 / in0 / in1 / p0 / p1 / add / mean / rstd / rows / hidden /
// eps as for the other families; `workspace` holds split_workspace_bytes.
cudaError_t launch_split(int op, const DynArgs& a, void* workspace, int sms, cudaStream_t st) {
    char* ws = static_cast<char*>(workspace);
    switch (op) {
        case 0: return fwd_t<0>(a, ws, sms, st);
        case 1: return fwd_t<1>(a, ws, sms, st);
        case 2: return fwd_t<2>(a, ws, sms, st);
        case 3: return bwd_t<3>(a, ws, sms, st);
        case 4: return bwd_t<4>(a, ws, sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nf
