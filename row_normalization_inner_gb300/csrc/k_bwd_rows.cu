// Row-block backward kernels for short rows (hidden 1024 and 2048): the
// LayerNorm backward, the RMSNorm backward and the fused residual-add
// RMSNorm backward, with the combined inner (per-row dx) and outer
// (across-rows dgamma / dbeta or dw) reductions of "Llu/ln bwd" (NVIDIA/Fuser
// PR #207, discussion of the layer norm backward as a normalization that
// reduces within rows and across them) and the column partials kept in a
// workspace ("TMA inner persistent scheduler", NVIDIA/Fuser PR #5587,
// description: the RMS norm and layer norm workspace support).
//
// Layout.  One persistent CTA per SM owns a contiguous stripe of rows and
// cuts it into blocks of R consecutive rows.  The CTA's threads form NG
// groups of GT threads; a group covers a whole row, thread t owning the
// 16-byte column slices v*GT + t (v < VPT), and the same columns in every
// row.  Group g takes the stripe's blocks g, g + NG, g + 2 NG, ...
//
// Data movement.  Each group has a private ring of SG stages in shared
// memory.  One thread of the group issues, per block, one 1-D bulk
// asynchronous copy (cp.async.bulk, global -> shared) per input tensor:
// the block's R rows are contiguous in memory, so each copy is R * H * 2
// bytes.  The copies complete on the stage's mbarrier; SG - 1 blocks are
// in flight while the group computes one.
//
// Per block.  Every thread reads its slices of the R rows from shared
// memory (128-bit loads), forms its share of the 2R row sums, and folds
// them across the warp with a recursive-halving shuffle (each lane ends
// with one of the 2R warp totals, log2(32) exchange steps in all instead
// of 5 per value), then across the group's warps through shared memory
// behind one named barrier.  The barrier also tells the issuing thread
// that every thread has read the stage, so it refills the stage with the
// group's block SG ahead.  dx is then formed from the row sums and stored
// with 128-bit streaming stores.
//
// Column sums.  Because a thread owns the same columns in every row, its
// share of the across-rows sums (sum dy * xhat and sum dy for LayerNorm,
// sum dy * x * rstd for RMSNorm) is 2 or 1 register pairs per 8 columns,
// independent of the hidden size.  At the end the NG groups fold their
// sums through shared memory in group order into the CTA's one workspace
// slot, and the column reduction (stage 2) adds the slots in slot order,
// so dgamma / dbeta / dw are bit-identical from run to run.
//
// Every mbarrier wait is bounded (2 s on the global timer).  A group whose
// wait gives up learns it at the named barrier (a reduction of the
// failure flags over the group), records NF_ERR_TIMEOUT, waits (bounded)
// for the copies it already issued, and leaves with the rest of the CTA.
#include "common.cuh"
#include "pairs.cuh"
#include "pdl.cuh"
#include "launch.h"

namespace nf {

enum RowsOp { kRowsLn = 0, kRowsRms = 1, kRowsFused = 2 };

// [kernel-span norm_rows_bwd_kernel] (with its shape table)
// Per hidden size: VPT vectors per thread, R rows per block, NG groups;
// IL = 0 gives each CTA a contiguous stripe of rows, IL = q >= 1 deals the
// blocks out to the CTAs in chunks of q consecutive blocks, round robin;
// CPS CTAs are resident per SM and the grid is GM x SMs CTAs (GM > CPS
// runs several waves, and the hardware hands the later CTAs to whichever
// SMs finish first).  Either mapping is a fixed function of (rows, grid),
// so which rows feed which partial slot never depends on timing.
template <int OP, int H> struct RowsShape;
template <int OP> struct RowsShape<OP, 1024> {
    static constexpr int VPT = 1, R = 4, NG = 3, IL = 0, CPS = 1, GM = 1;
};
// LayerNorm at 1024: four groups (16384 x 1024: 19.6 against 20.3 us with
// three; RMSNorm was slower with four: 23.0 against 19.0 us).
template <> struct RowsShape<kRowsLn, 1024> {
    static constexpr int VPT = 1, R = 4, NG = 4, IL = 0, CPS = 1, GM = 1;
};
template <int OP> struct RowsShape<OP, 2048> {
    static constexpr int VPT = 2, R = 2, NG = 3, IL = 0, CPS = 1, GM = 1;
};

constexpr int kRowsSmemBudget = 200 * 1024;  // per SM
constexpr int kRowsMaxStages = 8;

template <int OP, int H>
struct RGeo {
    static constexpr int VPT = RowsShape<OP, H>::VPT;
    static constexpr int R = RowsShape<OP, H>::R;
    static constexpr int NG = RowsShape<OP, H>::NG;
    static constexpr int IL = RowsShape<OP, H>::IL;
    static constexpr int CPS = RowsShape<OP, H>::CPS;
    static constexpr int GM = RowsShape<OP, H>::GM;
    static_assert(CPS >= 1 && GM >= CPS, "at least one wave");
    static constexpr int NV = H / kVec;
    static constexpr int GT = NV / VPT;       // threads per group: one row's width
    static constexpr int GW = GT / 32;
    static constexpr int THREADS = NG * GT;
    static_assert(NV % VPT == 0 && GT % 32 == 0, "whole warps per row");
    static_assert(GW >= 2 && GW <= 32, "the cross-warp step expects 2..32 warps per group");
    static_assert(THREADS <= 1024 && NG <= 15, "CTA size; named barriers 1..NG");
    static constexpr int NIN = OP == kRowsFused ? 3 : 2;   // staged tensors
    static constexpr int ROW_BYTES = H * 2;
    static_assert(ROW_BYTES % 128 == 0, "rows are whole 128-byte lines");
    static constexpr int TBYTES = R * ROW_BYTES;          // one tensor's block
    static constexpr int STAGE_BYTES = NIN * TBYTES;
    static constexpr int SG0 = kRowsSmemBudget / CPS / STAGE_BYTES / NG;
    static constexpr int SG = SG0 > kRowsMaxStages ? kRowsMaxStages : SG0;
    static_assert(SG >= 2, "at least two stages per group");
    static constexpr int NSUM = 2 * R;                    // row sums per block
    static_assert((NSUM & (NSUM - 1)) == 0 && NSUM >= 4 && NSUM <= 32,
                  "a power of two of row sums, read back as float4");
    static constexpr int PLANES = OP == kRowsLn ? 2 : 1;
    static_assert(SG * STAGE_BYTES >= PLANES * H * 4, "a group's ring holds its column sums");
    static constexpr int RED_FLOATS = 2 * GW * NSUM;       // two parities
    static constexpr int RING = NG * SG * STAGE_BYTES;
    static constexpr int BAR_OFF = RING;
    static constexpr int RED_OFF = (BAR_OFF + NG * SG * 8 + 15) / 16 * 16;  // float4 reads
    static constexpr int SMEM = RED_OFF + NG * RED_FLOATS * 4;
};

struct RowsArgs {
    uint16_t* dx;
    const uint16_t* x;       // LayerNorm / RMSNorm input (fused: the saved residual sum)
    const uint16_t* dy;
    const uint16_t* dres;    // fused: the residual-stream gradient
    const uint16_t* w;       // gamma / weight
    const float* mean;
    const float* rstd;
    float* ws;               // [grid][PLANES][H]
    int* status;
    int64_t rows;
    float eps;
};

__device__ __forceinline__ void rows_bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint4 rows_lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Named barrier over `nthreads` threads that also returns whether any of
// them passed `pred` = true.
__device__ __forceinline__ bool bar_any(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 q, %1, 0;\n\t"
                 "bar.red.or.pred p, %2, %3, q;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r) : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads) : "memory");
    return r != 0;
}

// Recursive halving over the 32 lanes of a warp: N values in, and lane l
// leaves with the warp total of value l >> (5 - log2 N) in v[0].  At the
// exchange with offset o the lane whose bit o is set keeps the upper half of
// its remaining values and sends the lower half (its partner the reverse),
// so the values left halve each step; once one is left the remaining
// offsets are a plain butterfly.  Each total is formed in an order that
// depends only on lane numbers, and in the butterfly partners add the same
// two operands, so every lane holding a total holds the same bits.
template <int N>
__device__ __forceinline__ void warp_halving_sum(float (&v)[N], int lane) {
    int o = 16;
#pragma unroll
    for (int n = N; n > 1; n >>= 1, o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
    }
#pragma unroll
    for (; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], o);
}

// The blocks of R rows a CTA owns, in the order its groups take them
// (group g takes the CTA's blocks g, g + NG, ...).
template <int R, int IL>
struct BlockMap {
    int64_t rows, r0;  // contiguous: the CTA's stripe [r0, r0 + n)
    int n;
    int64_t c, grid, nblocks;  // interleaved: CTA c of `grid`, nblocks in all
    int count;         // blocks of this CTA

    __device__ __forceinline__ BlockMap(int64_t rows_, int64_t c_, int64_t grid_)
        : rows(rows_), c(c_), grid(grid_) {
        if constexpr (IL == 0) {
            r0 = rows * c / grid;
            n = static_cast<int>(rows * (c + 1) / grid - r0);
            count = (n + R - 1) / R;
            nblocks = 0;
        } else {
            r0 = 0;
            n = 0;
            nblocks = (rows + R - 1) / R;
            const int64_t nchunks = (nblocks + IL - 1) / IL;
            int64_t k = 0;
            if (c < nchunks) {
                const int64_t mc = (nchunks - 1 - c) / grid + 1;  // chunks of this CTA
                k = mc * IL;
                const int64_t rem = nblocks % IL;
                if (rem != 0 && (nchunks - 1 - c) % grid == 0) k -= IL - rem;  // owns the short last chunk
            }
            count = static_cast<int>(k);
        }
    }
    // first row and row count of this CTA's k-th block (k < count)
    __device__ __forceinline__ void block(int k, int64_t* row0, int* nr) const {
        if constexpr (IL == 0) {
            *row0 = r0 + static_cast<int64_t>(k) * R;
            *nr = min(R, n - k * R);
        } else {
            const int64_t b = (c + static_cast<int64_t>(k / IL) * grid) * IL + k % IL;
            *row0 = b * R;
            *nr = static_cast<int>(min(static_cast<int64_t>(R), rows - b * R));
        }
    }
};

template <int N> struct Log2 { static constexpr int v = 1 + Log2<N / 2>::v; };
template <> struct Log2<1> { static constexpr int v = 0; };

template <int OP, int H>
__global__ void __launch_bounds__(RGeo<OP, H>::THREADS, RGeo<OP, H>::CPS)
norm_rows_bwd_kernel(RowsArgs a) {
    using G = RGeo<OP, H>;
    constexpr int R = G::R, VPT = G::VPT, NSUM = G::NSUM;
    extern __shared__ __align__(128) uint8_t smem[];

    const int g = threadIdx.x / G::GT;
    const int gt = threadIdx.x % G::GT;
    const int warp = gt >> 5, lane = gt & 31;
    const BlockMap<R, G::IL> map(a.rows, blockIdx.x, gridDim.x);
    const int nb = map.count;                                       // blocks of this CTA
    const int mine = nb > g ? (nb - g + G::NG - 1) / G::NG : 0;     // blocks of this group
    // Warm L2 with the group's first SG blocks before waiting for the kernel
    // ahead in the stream (a hint; the bulk copies below then find them there).
    for (int j = 0; j < G::SG && j < mine; ++j) {
        int64_t row;
        int nr;
        map.block(g + j * G::NG, &row, &nr);
        const int lines = nr * (G::ROW_BYTES / 128);
        for (int i = gt; i < lines; i += G::GT) {
            prefetch_l2(reinterpret_cast<const uint8_t*>(a.x + row * H) + i * 128);
            prefetch_l2(reinterpret_cast<const uint8_t*>(a.dy + row * H) + i * 128);
            if constexpr (OP == kRowsFused)
                prefetch_l2(reinterpret_cast<const uint8_t*>(a.dres + row * H) + i * 128);
        }
    }
    grid_dep_wait();

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::BAR_OFF) + g * G::SG;
    uint8_t* slice = smem + g * G::SG * G::STAGE_BYTES;
    float* red = reinterpret_cast<float*>(smem + G::RED_OFF) + g * G::RED_FLOATS;
    if (threadIdx.x == 0) {
        uint64_t* all = reinterpret_cast<uint64_t*>(smem + G::BAR_OFF);
        for (int s = 0; s < G::NG * G::SG; ++s) mbar_init(&all[s], 1);
        fence_barrier_init();
    }
    __syncthreads();

    // block j of this group is the CTA's block g + j NG; it uses stage j % SG
    const auto issue = [&](int j) {
        int64_t row;
        int nr;
        map.block(g + j * G::NG, &row, &nr);
        const int s = j % G::SG;
        const uint32_t bytes = static_cast<uint32_t>(nr) * G::ROW_BYTES;
        mbar_arrive_expect_tx(&full[s], G::NIN * bytes);
        const uint32_t st = smem_addr(slice + s * G::STAGE_BYTES);
        if constexpr (OP == kRowsLn || OP == kRowsRms) {
            rows_bulk_g2s(st, a.x + row * H, bytes, &full[s]);
            rows_bulk_g2s(st + G::TBYTES, a.dy + row * H, bytes, &full[s]);
        } else {
            rows_bulk_g2s(st, a.x + row * H, bytes, &full[s]);
            rows_bulk_g2s(st + G::TBYTES, a.dy + row * H, bytes, &full[s]);
            rows_bulk_g2s(st + 2 * G::TBYTES, a.dres + row * H, bytes, &full[s]);
        }
    };
    if (gt == 0) {
        for (int j = 0; j < G::SG && j < mine; ++j) issue(j);
    }

    // gamma / w for this thread's columns, widened once
    float2 wf[VPT][4];
#pragma unroll
    for (int v = 0; v < VPT; ++v) unpack8x2(ld_param(a.w + (v * G::GT + gt) * kVec), wf[v]);
    float2 acc0[VPT][4], acc1[OP == kRowsLn ? VPT : 1][4];
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc0[v][q] = make_float2(0.f, 0.f);
            if constexpr (OP == kRowsLn) acc1[v][q] = make_float2(0.f, 0.f);
        }

    // LayerNorm: the saved statistics of the group's blocks.  Lane l < R of
    // each warp holds the mean of row l of the block, lane R + l its rstd;
    // the next block's are fetched one block ahead and broadcast with
    // shuffles when used.
    static_assert(2 * R <= 32, "one lane per saved statistic");
    const auto fetch_stat = [&](int j) {
        float v = 0.f;
        if constexpr (OP == kRowsLn) {
            if (j < mine && lane < 2 * R) {
                int64_t row;
                int nr;
                map.block(g + j * G::NG, &row, &nr);
                const int r = lane % R;
                if (r < nr) v = __ldg((lane < R ? a.mean : a.rstd) + row + r);
            }
        }
        return v;
    };
    float stat = fetch_stat(0);
    float mu[R], rsv[R];

    bool failed = false;
    int j = 0;
    for (; j < mine; ++j) {
        int64_t row0;
        int nr;
        map.block(g + j * G::NG, &row0, &nr);
        const int s = j % G::SG;
        const uint32_t par = (j / G::SG) & 1;
        const float stat_next = fetch_stat(j + 1);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            mu[r] = __shfl_sync(0xFFFFFFFFu, stat, r);
            rsv[r] = __shfl_sync(0xFFFFFFFFu, stat, R + r);
        }
        const bool ok = mbar_wait(&full[s], par, kWaitLimitNs);
        const uint32_t st = smem_addr(slice + s * G::STAGE_BYTES);

        // this thread's slices of the block's rows, widened (rows past the
        // stripe's end read as zeros and are neither summed nor stored)
        float2 xa[R][VPT][4], da[R][VPT][4];
        uint4 ra[OP == kRowsFused ? R : 1][VPT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const uint32_t off = r * G::ROW_BYTES + (v * G::GT + gt) * 16;
                uint4 xv = make_uint4(0, 0, 0, 0), dv = make_uint4(0, 0, 0, 0);
                if (ok && r < nr) {
                    xv = rows_lds128(st + off);
                    dv = rows_lds128(st + G::TBYTES + off);
                    if constexpr (OP == kRowsFused) ra[r][v] = rows_lds128(st + 2 * G::TBYTES + off);
                }
                unpack8x2(xv, xa[r][v]);
                unpack8x2(dv, da[r][v]);
            }

        // pass 1: the row sums (and, for LayerNorm, the column sums)
        float sums[NSUM];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
            if constexpr (OP == kRowsLn) {
                // xhat = x * rstd - mean * rstd, g = dy * gamma: sums of g and g * xhat
                const float2 rs2 = make_float2(rsv[r], rsv[r]);
                const float nmr = -mu[r] * rsv[r];
                const float2 nmr2 = make_float2(nmr, nmr);
#pragma unroll
                for (int v = 0; v < VPT; ++v)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 xh = __ffma2_rn(xa[r][v][q], rs2, nmr2);
                        const float2 gg = __fmul2_rn(da[r][v][q], wf[v][q]);
                        s0 = __fadd2_rn(s0, gg);
                        s1 = __ffma2_rn(gg, xh, s1);
                        acc0[v][q] = __ffma2_rn(da[r][v][q], xh, acc0[v][q]);
                        acc1[v][q] = __fadd2_rn(acc1[v][q], da[r][v][q]);
                        xa[r][v][q] = xh;   // kept for pass 2
                        da[r][v][q] = gg;
                    }
            } else {
                // sums of x^2 and g * x with g = dy * w
#pragma unroll
                for (int v = 0; v < VPT; ++v)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        s0 = __ffma2_rn(xa[r][v][q], xa[r][v][q], s0);
                        s1 = __ffma2_rn(__fmul2_rn(da[r][v][q], wf[v][q]), xa[r][v][q], s1);
                    }
            }
            sums[2 * r] = s0.x + s0.y;
            sums[2 * r + 1] = s1.x + s1.y;
        }

        // fold the row sums over the group: lanes, then warps
        warp_halving_sum<NSUM>(sums, lane);
        float* rb = red + (j & 1) * G::GW * NSUM;
        constexpr int kLog = Log2<NSUM>::v;
        if ((lane & ((1 << (5 - kLog)) - 1)) == 0) rb[warp * NSUM + (lane >> (5 - kLog))] = sums[0];
        // every thread of the group has read the stage and written its warp
        // totals; a failed wait anywhere in the group stops the whole group
        if (bar_any(1 + g, G::GT, !ok)) { failed = true; break; }
        if (gt == 0 && j + G::SG < mine) issue(j + G::SG);
        float tot[NSUM];
#pragma unroll
        for (int i = 0; i < NSUM; ++i) tot[i] = 0.f;
#pragma unroll
        for (int w = 0; w < G::GW; ++w)
#pragma unroll
            for (int i4 = 0; i4 < NSUM / 4; ++i4) {
                const float4 p = reinterpret_cast<const float4*>(rb + w * NSUM)[i4];
                tot[4 * i4] += p.x;
                tot[4 * i4 + 1] += p.y;
                tot[4 * i4 + 2] += p.z;
                tot[4 * i4 + 3] += p.w;
            }

        // pass 2: dx, and for RMSNorm the column sums
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float2 c0, c1;
            float rsr = 0.f;
            if constexpr (OP == kRowsLn) {
                // dx = rstd * g - rstd * A - xhat * (rstd * B), A, B = row means of g, g * xhat
                const float rsA = rsv[r] * tot[2 * r] * (1.0f / H);
                const float rsB = rsv[r] * tot[2 * r + 1] * (1.0f / H);
                c0 = make_float2(-rsA, -rsA);
                c1 = make_float2(-rsB, -rsB);
                rsr = rsv[r];
            } else {
                // rstd = rsqrt(sum x^2 / H + eps); dx = rstd * g - x * rstd^3 * sum(g x) / H
                rsr = rsqrtf(tot[2 * r] * (1.0f / H) + a.eps);
                const float c = rsr * rsr * rsr * tot[2 * r + 1] * (1.0f / H);
                c0 = make_float2(0.f, 0.f);
                c1 = make_float2(-c, -c);
            }
            const float2 rs2 = make_float2(rsr, rsr);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                float2 o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (OP == kRowsLn) {
                        o[q] = __ffma2_rn(xa[r][v][q], c1, __ffma2_rn(rs2, da[r][v][q], c0));
                    } else {
                        const float2 gg = __fmul2_rn(da[r][v][q], wf[v][q]);
                        o[q] = __ffma2_rn(xa[r][v][q], c1, __fmul2_rn(rs2, gg));
                        if (r < nr)
                            acc0[v][q] = __ffma2_rn(__fmul2_rn(da[r][v][q], xa[r][v][q]), rs2, acc0[v][q]);
                    }
                }
                if constexpr (OP == kRowsFused) {
                    float2 af[4];
                    unpack8x2(ra[r][v], af);
#pragma unroll
                    for (int q = 0; q < 4; ++q) o[q] = __fadd2_rn(o[q], af[q]);
                }
                if (r < nr) st_stream(a.dx + (row0 + r) * H + (v * G::GT + gt) * kVec, pack8x2(o));
            }
        }
        stat = stat_next;
    }
    grid_dep_release();

    if (failed) {
        // let the copies this group issued land before the CTA can exit:
        // blocks j .. min(mine, j + SG) - 1 were issued and not consumed
        if (gt == 0) {
            record_status(a.status, kStatusTimeout);
            const int last = min(mine, j + G::SG);
            for (int jj = j; jj < last; ++jj)
                mbar_wait(&full[jj % G::SG], (jj / G::SG) & 1, kWaitLimitNs / 4);
        }
        __syncwarp();
    }

    // fold the groups' column sums in group order into this CTA's slot
    float* mine_f = reinterpret_cast<float*>(slice);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int jj = (v * G::GT + gt) * kVec;
        reinterpret_cast<float4*>(mine_f + jj)[0] =
            make_float4(acc0[v][0].x, acc0[v][0].y, acc0[v][1].x, acc0[v][1].y);
        reinterpret_cast<float4*>(mine_f + jj)[1] =
            make_float4(acc0[v][2].x, acc0[v][2].y, acc0[v][3].x, acc0[v][3].y);
        if constexpr (OP == kRowsLn) {
            reinterpret_cast<float4*>(mine_f + H + jj)[0] =
                make_float4(acc1[v][0].x, acc1[v][0].y, acc1[v][1].x, acc1[v][1].y);
            reinterpret_cast<float4*>(mine_f + H + jj)[1] =
                make_float4(acc1[v][2].x, acc1[v][2].y, acc1[v][3].x, acc1[v][3].y);
        }
    }
    __syncthreads();
    float4* out = reinterpret_cast<float4*>(a.ws + static_cast<int64_t>(blockIdx.x) * G::PLANES * H);
    for (int c4 = threadIdx.x; c4 < G::PLANES * H / 4; c4 += G::THREADS) {
        float4 s = reinterpret_cast<const float4*>(smem)[c4];
#pragma unroll
        for (int gg = 1; gg < G::NG; ++gg) {
            const float4 v = reinterpret_cast<const float4*>(smem + gg * G::SG * G::STAGE_BYTES)[c4];
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
        out[c4] = s;
    }
}

// [end kernel-span norm_rows_bwd_kernel]

namespace {

template <int OP, int H>
cudaError_t launch_rows_t(const RowsArgs& a, int grid, cudaStream_t st) {
    using G = RGeo<OP, H>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(norm_rows_bwd_kernel<OP, H>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    return launch_with_pdl(norm_rows_bwd_kernel<OP, H>, dim3(grid), dim3(G::THREADS), G::SMEM,
                           st, a);
}

template <int OP>
cudaError_t launch_rows_op(int64_t hidden, const RowsArgs& a, int grid, cudaStream_t st) {
    switch (hidden) {
        case 1024: return launch_rows_t<OP, 1024>(a, grid, st);
        case 2048: return launch_rows_t<OP, 2048>(a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

template <int OP>
bool rows_shape_of(int64_t hidden, int* threads, int* stages, int* smem, int* groups, int* grid_per_sm) {
    switch (hidden) {
#define NF_ROWS_CASE(HV)                                                                 \
        case HV: *threads = RGeo<OP, HV>::THREADS; *stages = RGeo<OP, HV>::NG * RGeo<OP, HV>::SG; \
                 *smem = RGeo<OP, HV>::SMEM; *groups = RGeo<OP, HV>::NG;                  \
                 *grid_per_sm = RGeo<OP, HV>::GM; return true;
        NF_ROWS_CASE(1024) NF_ROWS_CASE(2048)
#undef NF_ROWS_CASE
        default: return false;
    }
}

}  // namespace

bool rows_bwd_shape(int op, int64_t hidden, int* threads, int* stages, int* smem_bytes, int* groups,
                    int* grid_per_sm) {
    // op numbering of the bulk family: 3 LayerNorm backward, 4 RMSNorm backward
    if (op == 3) return rows_shape_of<kRowsLn>(hidden, threads, stages, smem_bytes, groups, grid_per_sm);
    if (op == 4) return rows_shape_of<kRowsRms>(hidden, threads, stages, smem_bytes, groups, grid_per_sm);
    return false;
}

cudaError_t launch_ln_bwd_rows(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                               const float* mean, const float* rstd, const void* gamma,
                               int64_t rows, int grid, int* status, cudaStream_t st) {
    RowsArgs a{};
    a.dx = static_cast<uint16_t*>(dx);
    a.x = static_cast<const uint16_t*>(x);
    a.dy = static_cast<const uint16_t*>(dy);
    a.w = static_cast<const uint16_t*>(gamma);
    a.mean = mean;
    a.rstd = rstd;
    a.ws = ws;
    a.status = status;
    a.rows = rows;
    return launch_rows_op<kRowsLn>(hidden, a, grid, st);
}

cudaError_t launch_rms_bwd_rows(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                                const void* dres, const void* w, int64_t rows, float eps, int grid,
                                int* status, cudaStream_t st) {
    RowsArgs a{};
    a.dx = static_cast<uint16_t*>(dx);
    a.x = static_cast<const uint16_t*>(x);
    a.dy = static_cast<const uint16_t*>(dy);
    a.dres = static_cast<const uint16_t*>(dres);
    a.w = static_cast<const uint16_t*>(w);
    a.ws = ws;
    a.status = status;
    a.rows = rows;
    a.eps = eps;
    return dres ? launch_rows_op<kRowsFused>(hidden, a, grid, st)
                : launch_rows_op<kRowsRms>(hidden, a, grid, st);
}

}  // namespace nf
