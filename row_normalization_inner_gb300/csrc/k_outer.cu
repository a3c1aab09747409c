// Outer normalization: statistics per column, over the rows (the block- and
// grid-parallel outer normalization that the "Llu/ln bwd" discussion lists
// beside the inner variants; batch normalization of a [rows, hidden] matrix
// in training mode).
//
// A column's rows are far apart in memory, so a whole column cannot stay in
// one CTA: each direction is a statistics pass over (column tile, row
// stripe) CTAs, a small merge kernel per column, and an elementwise apply
// pass.  The forward reads x twice and the backward reads x and dy twice.
// (Walking the matrix in column chunks so that the apply pass re-reads its
// chunk from L2 was measured on GB300 and lost to the plain two passes: the
// extra launches and merge bubbles cost more than the saved HBM reads.)
//
// Tiles are OX x 8 columns (OX column lanes, 16-byte copies; 128 lanes from
// hidden 1024 up, 32 below) by a row stripe walked by 256 / OX row lanes,
// so a row's tile is read as OX * 16 contiguous bytes.  A thread streams its
// rows through a private cp.async ring in shared memory (several rows in
// flight, no registers held), the grid is one wave of resident CTAs, and the
// arithmetic runs on packed fp32 pairs (add / mul / fma .f32x2).
//
// Forward statistics: each thread keeps shifted sums (shift = its first
// value) per column and turns them into (count, mean, M2); row lanes and
// then stripes are merged in a fixed order with Chan's pairwise formula --
// numerically stable and deterministic.  The merge kernel writes mean, rstd
// and the per-column affine pair a = rstd * gamma, b = beta - mean * a, so
// the apply pass is one fma per element.  Backward: per-stripe column sums
// of dy * xhat and dy, merged in a fixed order into dgamma / dbeta, and the
// apply pass forms dx = c1 * dy - k2 - (x - mean) * k3 with per-column
// c1 = rstd * gamma, k2 = c1 * dbeta / R, k3 = c1 * rstd * dgamma / R.
//
// The statistics passes stream x (and dy) with an L2 evict-last hint and
// the apply passes read them evict-first, so whatever part of the input L2
// can hold is read from DRAM once (forward 16384 x 4096: 70.4 -> 65.9 us).
//
// Every kernel is launched as a programmatic dependent of the one before it
// and starts with griddepcontrol.wait, so launch latency overlaps the tail
// of the previous kernel while every read still follows its producer.
#include "common.cuh"
#include "pairs.cuh"
#include "launch.h"

namespace nf {
namespace {

constexpr int kOT = 256;  // threads per streaming CTA
constexpr int kMW = 8;    // merge kernels: warps (columns) per CTA
constexpr int kMU = 8;    // merge kernels: partials in flight per lane

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

// Row stripes: `ns` stripes of `base` rows, the first `rem` of them one row
// longer (base = rows / ns, rem = rows % ns).
struct Stripes {
    int64_t base;
    int rem;
    __device__ __forceinline__ int64_t begin(int s) const { return s * base + (s < rem ? s : rem); }
    __device__ __forceinline__ int64_t size(int s) const { return base + (s < rem ? 1 : 0); }
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- per-thread copy ring ---------------------------------------------------
// Each thread streams its own rows through a private ring of S stages in
// dynamic shared memory, U rows of A arrays per stage, filled by 16-byte
// cp.async copies: S - 1 stages are in flight while one is computed, and no
// registers are held by the loads.  A thread only reads what it copied, so
// cp.async.wait_group is the only synchronization.  Layout
// [stage][array][row][thread] keeps a warp's 16-byte reads conflict-free.
// 16-byte copy with an L2 eviction-priority policy: the statistics passes
// ask L2 to keep x (and dy), which their apply pass reads again; the apply
// passes mark them evict-first (their last use).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;"
                 ::"r"(smem_addr(smem)), "l"(gmem), "l"(pol) : "memory");
}
__device__ __forceinline__ uint64_t policy_keep() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_last_use() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The apply passes walk each thread's rows last to first: the statistics
// pass streamed them first to last, so the rows it read last are the ones
// still in L2 when the apply pass starts.
constexpr bool kApplyLastFirst = true;

template <int S, int U, int A, int OY>
struct RowRing {
    static constexpr int kBytes = S * A * U * kOT * 16;
    uint4* base;
    int64_t row0;  // this thread's first row; its rows are row0 + i * OY
    int cnt;       // number of rows of this thread
    uint64_t pol;  // L2 policy of the copies
    bool rev;      // walk the rows last to first
    // row of this thread's i-th step
    __device__ __forceinline__ int64_t row(int i) const {
        return row0 + static_cast<int64_t>(rev ? cnt - 1 - i : i) * OY;
    }
    __device__ __forceinline__ uint4* at(int st, int a, int u) const {
        return base + (((st % S) * A + a) * U + u) * kOT + threadIdx.x;
    }
    // One commit group with rows st*U .. st*U+U-1 (empty past the end).
    __device__ __forceinline__ void issue(int st, const uint16_t* const (&src)[A], int hidden,
                                          int64_t c0) const {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = st * U + u;
            if (i < cnt) {
#pragma unroll
                for (int a = 0; a < A; ++a)
                    cp_async16(at(st, a, u), src[a] + row(i) * hidden + c0, pol);
            }
        }
        cp_commit();
    }
    __device__ __forceinline__ int stages() const { return (cnt + U - 1) / U; }
    __device__ __forceinline__ void prologue(const uint16_t* const (&src)[A], int hidden, int64_t c0) const {
#pragma unroll
        for (int st = 0; st < S - 1; ++st) issue(st, src, hidden, c0);
    }
    // Start stage st + S - 1 and wait for stage st.
    __device__ __forceinline__ void advance(int st, const uint16_t* const (&src)[A], int hidden,
                                            int64_t c0) const {
        issue(st + S - 1, src, hidden, c0);
        cp_wait<S - 1>();
    }
};

// Rows of this thread in a stripe of `len` rows: ty, ty + OY, ...
template <int OY>
__device__ __forceinline__ int thread_rows(int64_t len, int ty) {
    return len > ty ? static_cast<int>((len - ty + OY - 1) / OY) : 0;
}

// ---- packed fp32 pairs ------------------------------------------------------
__device__ __forceinline__ float2 neg2(float2 v) { return make_float2(-v.x, -v.y); }
__device__ __forceinline__ void load8x2(const float* p, float2 (&f)[4]) {  // p 4-byte aligned
#pragma unroll
    for (int q = 0; q < 4; ++q) f[q] = make_float2(__ldcg(p + 2 * q), __ldcg(p + 2 * q + 1));
}

constexpr int kFS = 4, kFU = 4;  // forward rings: 4 stages of 4 rows (64 KB per CTA)
constexpr int kBS = 3, kBU = 4;  // backward rings: 3 stages of 4 rows of x and dy (96 KB)
template <int OY> using FwdRing = RowRing<kFS, kFU, 1, OY>;
template <int OY> using BwdRing = RowRing<kBS, kBU, 2, OY>;
constexpr int kFwdBytes = kFS * kFU * kOT * 16;
constexpr int kBwdBytes = kBS * 2 * kBU * kOT * 16;
constexpr int kFwdCtasPerSm = 3;
constexpr int kBwdCtasPerSm = 2;

// Forward pass 1: per (stripe, column) mean and M2 -> part[stripe][H]
// (float2).  Grid: (column tiles, stripes).
template <int OX>
__global__ void __launch_bounds__(kOT, kFwdCtasPerSm)
outer_stats(const uint16_t* __restrict__ x, float2* __restrict__ part, Stripes sp, int hidden,
            int col0, int col1) {
    constexpr int OY = kOT / OX;
    extern __shared__ __align__(16) uint4 dsm[];
    pdl_wait();
    const int tx = threadIdx.x % OX, ty = threadIdx.x / OX, stripe = blockIdx.y;
    const int64_t c0 = col0 + (static_cast<int64_t>(blockIdx.x) * OX + tx) * kVec;
    const bool ok = c0 < col1;
    const FwdRing<OY> ring{dsm, sp.begin(stripe) + ty, ok ? thread_rows<OY>(sp.size(stripe), ty) : 0,
                           policy_keep(), false};
    const uint16_t* const src[1] = {x};
    float2 nk[4], s1[4], s2[4];  // nk = -shift
#pragma unroll
    for (int q = 0; q < 4; ++q) { nk[q] = make_float2(0.f, 0.f); s1[q] = nk[q]; s2[q] = nk[q]; }
    ring.prologue(src, hidden, c0);
    const int nst = ring.stages();
    for (int st = 0; st < nst; ++st) {
        ring.advance(st, src, hidden, c0);
#pragma unroll
        for (int u = 0; u < kFU; ++u) {
            const int i = st * kFU + u;
            if (i < ring.cnt) {
                float2 f[4];
                unpack8x2(*ring.at(st, 0, u), f);
                if (i == 0) {  // the shift is the thread's first value
#pragma unroll
                    for (int q = 0; q < 4; ++q) nk[q] = neg2(f[q]);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 d = __fadd2_rn(f[q], nk[q]);
                    s1[q] = __fadd2_rn(s1[q], d);
                    s2[q] = __ffma2_rn(d, d, s2[q]);
                }
            }
        }
    }
    cp_wait<0>();
    __syncthreads();  // the ring is reused below
    Chan(*sh)[OX][kVec] = reinterpret_cast<Chan(*)[OX][kVec]>(dsm);
    const float n = static_cast<float>(ring.cnt);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        Chan c{n, 0.f, 0.f};
        if (n > 0.f) {
            const float a1 = e & 1 ? s1[e / 2].y : s1[e / 2].x;
            const float a2 = e & 1 ? s2[e / 2].y : s2[e / 2].x;
            const float sh_k = e & 1 ? -nk[e / 2].y : -nk[e / 2].x;
            const float m = a1 / n;
            c.mean = sh_k + m;
            c.m2 = fmaxf(a2 - a1 * m, 0.f);
        }
        sh[ty][tx][e] = c;
    }
    __syncthreads();
    if (ty == 0 && ok) {
        float2 out[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            Chan acc = sh[0][tx][e];
#pragma unroll
            for (int y = 1; y < OY; ++y) acc = chan_merge(acc, sh[y][tx][e]);
            out[e] = make_float2(acc.mean, acc.m2);
        }
        float4* dst = reinterpret_cast<float4*>(part + static_cast<int64_t>(stripe) * hidden + c0);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            dst[e] = make_float4(out[2 * e].x, out[2 * e].y, out[2 * e + 1].x, out[2 * e + 1].y);
    }
}

// Forward pass 2: y = x * a + b with (a, b) = coef[0][j], coef[1][j].
template <int OX>
__global__ void __launch_bounds__(kOT, kFwdCtasPerSm)
outer_apply(uint16_t* y, const uint16_t* x, const float* __restrict__ coef, Stripes sp, int hidden,
            int col0, int col1) {
    constexpr int OY = kOT / OX;
    extern __shared__ __align__(16) uint4 dsm[];
    pdl_wait();
    const int tx = threadIdx.x % OX, ty = threadIdx.x / OX, stripe = blockIdx.y;
    const int64_t c0 = col0 + (static_cast<int64_t>(blockIdx.x) * OX + tx) * kVec;
    if (c0 >= col1) return;
    const FwdRing<OY> ring{dsm, sp.begin(stripe) + ty, thread_rows<OY>(sp.size(stripe), ty),
                           policy_last_use(), kApplyLastFirst};
    const uint16_t* const src[1] = {x};
    ring.prologue(src, hidden, c0);
    float2 a[4], b[4];
    load8x2(coef + c0, a);
    load8x2(coef + hidden + c0, b);
    const int nst = ring.stages();
    for (int st = 0; st < nst; ++st) {
        ring.advance(st, src, hidden, c0);
#pragma unroll
        for (int u = 0; u < kFU; ++u) {
            const int i = st * kFU + u;
            if (i < ring.cnt) {
                float2 f[4], o[4];
                unpack8x2(*ring.at(st, 0, u), f);
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = __ffma2_rn(f[q], a[q], b[q]);
                st_stream(y + ring.row(i) * hidden + c0, pack8x2(o));
            }
        }
    }
    cp_wait<0>();
}

// Backward pass 1: per (stripe, column) sums of dy * xhat and dy ->
// ws[stripe][0][H], ws[stripe][1][H].
template <int OX>
__global__ void __launch_bounds__(kOT, kBwdCtasPerSm)
outer_bwd_sums(const uint16_t* __restrict__ dy, const uint16_t* __restrict__ x,
               const float* __restrict__ mean, const float* __restrict__ rstd,
               float* __restrict__ ws, Stripes sp, int hidden, int col0, int col1) {
    constexpr int OY = kOT / OX;
    extern __shared__ __align__(16) uint4 dsm[];
    pdl_wait();
    const int tx = threadIdx.x % OX, ty = threadIdx.x / OX, stripe = blockIdx.y;
    const int64_t c0 = col0 + (static_cast<int64_t>(blockIdx.x) * OX + tx) * kVec;
    const bool ok = c0 < col1;
    const BwdRing<OY> ring{dsm, sp.begin(stripe) + ty, ok ? thread_rows<OY>(sp.size(stripe), ty) : 0,
                           policy_keep(), false};
    const uint16_t* const src[2] = {x, dy};
    ring.prologue(src, hidden, c0);
    float2 sg[4], sb[4], nmu[4], rs[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        sg[q] = make_float2(0.f, 0.f); sb[q] = sg[q]; nmu[q] = sg[q]; rs[q] = sg[q];
    }
    if (ok) {
        load8x2(mean + c0, nmu);
        load8x2(rstd + c0, rs);
#pragma unroll
        for (int q = 0; q < 4; ++q) nmu[q] = neg2(nmu[q]);
    }
    const int nst = ring.stages();
    for (int st = 0; st < nst; ++st) {
        ring.advance(st, src, hidden, c0);
#pragma unroll
        for (int u = 0; u < kBU; ++u) {
            const int i = st * kBU + u;
            if (i < ring.cnt) {
                float2 xf[4], df[4];
                unpack8x2(*ring.at(st, 0, u), xf);
                unpack8x2(*ring.at(st, 1, u), df);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 xh = __fmul2_rn(__fadd2_rn(xf[q], nmu[q]), rs[q]);
                    sg[q] = __ffma2_rn(df[q], xh, sg[q]);
                    sb[q] = __fadd2_rn(sb[q], df[q]);
                }
            }
        }
    }
    cp_wait<0>();
    __syncthreads();  // the ring is reused below
    float4(*sh)[OX][4] = reinterpret_cast<float4(*)[OX][4]>(dsm);
    sh[ty][tx][0] = make_float4(sg[0].x, sg[0].y, sg[1].x, sg[1].y);
    sh[ty][tx][1] = make_float4(sg[2].x, sg[2].y, sg[3].x, sg[3].y);
    sh[ty][tx][2] = make_float4(sb[0].x, sb[0].y, sb[1].x, sb[1].y);
    sh[ty][tx][3] = make_float4(sb[2].x, sb[2].y, sb[3].x, sb[3].y);
    __syncthreads();
    if (ty == 0 && ok) {
        float4 t[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) t[q] = sh[0][tx][q];
#pragma unroll
        for (int yy = 1; yy < OY; ++yy)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = sh[yy][tx][q];
                t[q].x += v.x; t[q].y += v.y; t[q].z += v.z; t[q].w += v.w;
            }
        float* slot = ws + static_cast<int64_t>(stripe) * 2 * hidden;
        reinterpret_cast<float4*>(slot + c0)[0] = t[0];
        reinterpret_cast<float4*>(slot + c0)[1] = t[1];
        reinterpret_cast<float4*>(slot + hidden + c0)[0] = t[2];
        reinterpret_cast<float4*>(slot + hidden + c0)[1] = t[3];
    }
}

// Backward pass 2: dx = c1 * dy - k2 - (x - mean) * k3.
template <int OX>
__global__ void __launch_bounds__(kOT, kBwdCtasPerSm)
outer_bwd_apply(uint16_t* dx, const uint16_t* dy, const uint16_t* x, const float* __restrict__ mean,
                const float* __restrict__ rstd, const uint16_t* __restrict__ gamma,
                const float* __restrict__ dgamma, const float* __restrict__ dbeta, float invR,
                Stripes sp, int hidden, int col0, int col1) {
    constexpr int OY = kOT / OX;
    extern __shared__ __align__(16) uint4 dsm[];
    pdl_wait();
    const int tx = threadIdx.x % OX, ty = threadIdx.x / OX, stripe = blockIdx.y;
    const int64_t c0 = col0 + (static_cast<int64_t>(blockIdx.x) * OX + tx) * kVec;
    if (c0 >= col1) return;
    const BwdRing<OY> ring{dsm, sp.begin(stripe) + ty, thread_rows<OY>(sp.size(stripe), ty),
                           policy_last_use(), kApplyLastFirst};
    const uint16_t* const src[2] = {x, dy};
    ring.prologue(src, hidden, c0);
    float2 nmu[4], c1[4], nk2[4], nk3[4];  // -mean, c1, -k2, -k3
    {
        float2 g[4], rs[4], dg[4], db[4];
        unpack8x2(ld_param(gamma + c0), g);
        load8x2(mean + c0, nmu);
        load8x2(rstd + c0, rs);
        load8x2(dgamma + c0, dg);
        load8x2(dbeta + c0, db);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            nmu[q] = neg2(nmu[q]);
            c1[q] = make_float2(rs[q].x * g[q].x, rs[q].y * g[q].y);
            nk2[q] = make_float2(-(c1[q].x * db[q].x * invR), -(c1[q].y * db[q].y * invR));
            nk3[q] = make_float2(-(c1[q].x * rs[q].x * dg[q].x * invR),
                                 -(c1[q].y * rs[q].y * dg[q].y * invR));
        }
    }
    const int nst = ring.stages();
    for (int st = 0; st < nst; ++st) {
        ring.advance(st, src, hidden, c0);
#pragma unroll
        for (int u = 0; u < kBU; ++u) {
            const int i = st * kBU + u;
            if (i < ring.cnt) {
                float2 xf[4], df[4], o[4];
                unpack8x2(*ring.at(st, 0, u), xf);
                unpack8x2(*ring.at(st, 1, u), df);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    o[q] = __ffma2_rn(__fadd2_rn(xf[q], nmu[q]), nk3[q], __ffma2_rn(c1[q], df[q], nk2[q]));
                st_stream(dx + ring.row(i) * hidden + c0, pack8x2(o));
            }
        }
    }
    cp_wait<0>();
}

__device__ __forceinline__ Chan chan_shfl_down(Chan c, int off) {
    return {__shfl_down_sync(0xffffffffu, c.n, off), __shfl_down_sync(0xffffffffu, c.mean, off),
            __shfl_down_sync(0xffffffffu, c.m2, off)};
}

// One warp per column: lane L merges stripes L, L + 32, ... in order, then
// the lanes merge in a fixed tree (lane 0 ends with the column).  Writes
// mean / rstd and the affine pair (a, b) -> coef[0][H], coef[1][H].
__global__ void __launch_bounds__(kMW * 32)
outer_finalize(const float2* __restrict__ part, const uint16_t* __restrict__ gamma,
               const uint16_t* __restrict__ beta, float* __restrict__ mean_out,
               float* __restrict__ rstd_out, float* __restrict__ coef, int64_t rows, int hidden,
               int col0, int col1, int nstripe, Stripes sp, float eps) {
    pdl_wait();
    const int lane = threadIdx.x % 32;
    const int64_t j = col0 + static_cast<int64_t>(blockIdx.x) * kMW + threadIdx.x / 32;
    if (j >= col1) return;  // whole warps
    // gamma / beta are loaded before the merge so their latency overlaps it
    const uint16_t gj = gamma[j], bj = beta[j];
    Chan acc{0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < nstripe; s0 += 32 * kMU) {
        float2 p[kMU];
#pragma unroll
        for (int u = 0; u < kMU; ++u) {
            const int s = s0 + u * 32 + lane;
            p[u] = s < nstripe ? __ldcg(part + static_cast<int64_t>(s) * hidden + j) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kMU; ++u) {
            const int s = s0 + u * 32 + lane;
            if (s < nstripe) acc = chan_merge(acc, Chan{static_cast<float>(sp.size(s)), p[u].x, p[u].y});
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const Chan o = chan_shfl_down(acc, off);
        if (lane < off) acc = chan_merge(acc, o);
    }
    if (lane != 0) return;
    const float var = acc.m2 / static_cast<float>(rows);
    const float rstd = rsqrtf(var + eps);
    const float g = __uint_as_float(static_cast<uint32_t>(gj) << 16);
    const float b = __uint_as_float(static_cast<uint32_t>(bj) << 16);
    const float a = rstd * g;
    if (mean_out) mean_out[j] = acc.mean;
    if (rstd_out) rstd_out[j] = rstd;
    coef[j] = a;
    coef[hidden + j] = fmaf(-acc.mean, a, b);
}

// Sum the stripes of each column in the fixed order of outer_finalize ->
// dgamma[j], dbeta[j].
__global__ void __launch_bounds__(kMW * 32)
outer_bwd_reduce(const float* __restrict__ ws, float* __restrict__ dgamma,
                 float* __restrict__ dbeta, int hidden, int col0, int col1, int nstripe) {
    pdl_wait();
    const int lane = threadIdx.x % 32;
    const int64_t j = col0 + static_cast<int64_t>(blockIdx.x) * kMW + threadIdx.x / 32;
    if (j >= col1) return;  // whole warps
    float sg = 0.f, sb = 0.f;
    for (int s0 = 0; s0 < nstripe; s0 += 32 * kMU) {
        float pg[kMU], pb[kMU];
#pragma unroll
        for (int u = 0; u < kMU; ++u) {
            const int s = s0 + u * 32 + lane;
            const float* slot = ws + static_cast<int64_t>(s) * 2 * hidden;
            pg[u] = s < nstripe ? __ldcg(slot + j) : 0.f;
            pb[u] = s < nstripe ? __ldcg(slot + hidden + j) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kMU; ++u) {
            sg += pg[u];
            sb += pb[u];
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float og = __shfl_down_sync(0xffffffffu, sg, off);
        const float ob = __shfl_down_sync(0xffffffffu, sb, off);
        if (lane < off) {
            sg += og;
            sb += ob;
        }
    }
    if (lane != 0) return;
    dgamma[j] = sg;
    dbeta[j] = sb;
}

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel k, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

Stripes make_stripes(int64_t rows, int ns) { return Stripes{rows / ns, static_cast<int>(rows % ns)}; }

// Column lanes per tile: 128 (1024 columns) from hidden 1024 up, else 32.
int lanes_for(int64_t hidden) { return hidden >= 1024 ? 128 : 32; }

template <int OX>
cudaError_t set_smem_attrs() {
    cudaError_t e = cudaFuncSetAttribute(outer_stats<OX>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdBytes);
    if (!e) e = cudaFuncSetAttribute(outer_apply<OX>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdBytes);
    if (!e) e = cudaFuncSetAttribute(outer_bwd_sums<OX>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdBytes);
    if (!e) e = cudaFuncSetAttribute(outer_bwd_apply<OX>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdBytes);
    return e;
}

// Opt the streaming kernels into their dynamic shared memory, once per device.
cudaError_t ensure_smem_attrs() {
    constexpr int kMaxDev = 64;
    static bool done[kMaxDev] = {};
    int dev;
    if (cudaError_t e = cudaGetDevice(&dev)) return e;
    if (dev >= 0 && dev < kMaxDev && done[dev]) return cudaSuccess;
    cudaError_t e = set_smem_attrs<32>();
    if (!e) e = set_smem_attrs<128>();
    if (!e && dev >= 0 && dev < kMaxDev) done[dev] = true;
    return e;
}
static_assert(sizeof(Chan) * kOT * kVec <= kFwdBytes, "stats epilogue fits the ring");
static_assert(sizeof(float4) * kOT * 4 <= kBwdBytes, "sums epilogue fits the ring");

// Row stripes: about one CTA per SM over the column tiles (measured faster
// than a full wave of 2-3 resident CTAs per SM: fewer stripe partials to
// merge and longer streams per thread), and at least 4 rows per row lane.
int stripes_for(int64_t rows, int64_t cols, int sms) {
    const int64_t r = rows > 0 ? rows : 1;
    const int ox = lanes_for(cols);
    const int64_t nt = (cols + ox * kVec - 1) / (ox * kVec);
    int64_t ns = sms / nt;
    const int64_t rows_min = 4LL * (kOT / ox);
    const int64_t most = (r + rows_min - 1) / rows_min;
    if (ns > most) ns = most;
    if (ns > 65535) ns = 65535;
    if (ns < 1) ns = 1;
    return static_cast<int>(ns);
}

template <int OX>
cudaError_t fwd_pass(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                      const void* beta, int64_t rows, int64_t hidden, float eps, float2* part,
                      float* coef, int64_t c0, int64_t c1, int stripes, cudaStream_t st) {
    const Stripes sp = make_stripes(rows, stripes);
    const int h = static_cast<int>(hidden), a = static_cast<int>(c0), b = static_cast<int>(c1);
    const dim3 grid(static_cast<unsigned>((c1 - c0 + OX * kVec - 1) / (OX * kVec)), stripes);
    if (cudaError_t e = launch_pdl(outer_stats<OX>, grid, dim3(kOT), kFwdBytes, st,
                                   static_cast<const uint16_t*>(x), part, sp, h, a, b))
        return e;
    if (cudaError_t e = launch_pdl(outer_finalize, dim3(static_cast<unsigned>((c1 - c0 + kMW - 1) / kMW)),
                                   dim3(kMW * 32), 0, st, static_cast<const float2*>(part),
                                   static_cast<const uint16_t*>(gamma),
                                   static_cast<const uint16_t*>(beta), mean, rstd, coef, rows, h, a,
                                   b, stripes, sp, eps))
        return e;
    return launch_pdl(outer_apply<OX>, grid, dim3(kOT), kFwdBytes, st, static_cast<uint16_t*>(y),
                      static_cast<const uint16_t*>(x), static_cast<const float*>(coef), sp, h, a, b);
}

template <int OX>
cudaError_t bwd_pass(void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                      const float* mean, const float* rstd, const void* gamma, int64_t rows,
                      int64_t hidden, float* ws, int64_t c0, int64_t c1, int stripes,
                      cudaStream_t st) {
    const Stripes sp = make_stripes(rows, stripes);
    const int h = static_cast<int>(hidden), a = static_cast<int>(c0), b = static_cast<int>(c1);
    const dim3 grid(static_cast<unsigned>((c1 - c0 + OX * kVec - 1) / (OX * kVec)), stripes);
    if (cudaError_t e = launch_pdl(outer_bwd_sums<OX>, grid, dim3(kOT), kBwdBytes, st,
                                   static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(x),
                                   mean, rstd, ws, sp, h, a, b))
        return e;
    if (cudaError_t e = launch_pdl(outer_bwd_reduce, dim3(static_cast<unsigned>((c1 - c0 + kMW - 1) / kMW)),
                                   dim3(kMW * 32), 0, st, static_cast<const float*>(ws), dgamma,
                                   dbeta, h, a, b, stripes))
        return e;
    return launch_pdl(outer_bwd_apply<OX>, grid, dim3(kOT), kBwdBytes, st,
                      static_cast<uint16_t*>(dx), static_cast<const uint16_t*>(dy),
                      static_cast<const uint16_t*>(x), mean, rstd,
                      static_cast<const uint16_t*>(gamma), static_cast<const float*>(dgamma),
                      static_cast<const float*>(dbeta), 1.0f / static_cast<float>(rows), sp, h, a, b);
}

}  // namespace

int outer_stripes(int64_t rows, int64_t hidden, int sms) { return stripes_for(rows, hidden, sms); }

size_t outer_workspace_bytes(int64_t rows, int64_t hidden, int sms) {
    const size_t ns = static_cast<size_t>(outer_stripes(rows, hidden, sms));
    const size_t fwd = ns * hidden * sizeof(float2) + 2 * hidden * sizeof(float);
    const size_t bwd = ns * 2 * hidden * sizeof(float);
    const size_t grid = outer_grid_workspace_bytes(rows, hidden, sms);  // the on-chip form
    const size_t most = fwd > bwd ? fwd : bwd;
    return most > grid ? most : grid;
}

// One pass over all columns.  (Walking the columns in chunks sized for L2,
// so that each chunk's apply pass would re-read it from there, was measured
// slower at every size, even with the eviction hints: each chunk adds three
// launches and a merge bubble, and a chunk has fewer column tiles to spread
// over the SMs.)
cudaError_t launch_outer_fwd(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                             const void* beta, int64_t rows, int64_t hidden, float eps,
                             void* workspace, int sms, cudaStream_t st) {
    if (cudaError_t e = ensure_smem_attrs()) return e;
    const int ns = outer_stripes(rows, hidden, sms);
    float2* part = static_cast<float2*>(workspace);
    float* coef = reinterpret_cast<float*>(part + static_cast<int64_t>(ns) * hidden);
    return lanes_for(hidden) == 128
               ? fwd_pass<128>(y, mean, rstd, x, gamma, beta, rows, hidden, eps, part, coef, 0, hidden, ns, st)
               : fwd_pass<32>(y, mean, rstd, x, gamma, beta, rows, hidden, eps, part, coef, 0, hidden, ns, st);
}

cudaError_t launch_outer_bwd(void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                             const float* mean, const float* rstd, const void* gamma, int64_t rows,
                             int64_t hidden, void* workspace, int sms, cudaStream_t st) {
    if (cudaError_t e = ensure_smem_attrs()) return e;
    const int ns = outer_stripes(rows, hidden, sms);
    float* ws = static_cast<float*>(workspace);
    return lanes_for(hidden) == 128
               ? bwd_pass<128>(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows, hidden, ws, 0, hidden, ns, st)
               : bwd_pass<32>(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows, hidden, ws, 0, hidden, ns, st);
}

}  // namespace nf
