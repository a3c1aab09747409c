// Bulk-copy staged kernels ("TMA inner persistent scheduler", NVIDIA/Fuser
// PR #5587: a TMA path beside the non-TMA one, vectorized smem-to-register
// loads, and register sharing between the copy branch and the compute
// branch).
//
// One persistent CTA per SM walks a contiguous stripe of rows.  Warp group 0
// is the producer: one elected thread issues, per row, one 1-D bulk
// asynchronous copy (cp.async.bulk, global -> this CTA's shared memory) per
// input tensor into a ring of S stages, each completing on the stage's
// "full" mbarrier (one issuing thread per producer warp, each serving its
// own row groups).  The consumers are NG independent row groups of GW warps
// each; row i of the stripe belongs to group i % NG, and every group owns a
// private slice of SG ring stages which it consumes strictly in order (so a
// stage's barrier phases and the group's row sequence move in lockstep and
// a parity wait can never match a phase from an earlier use).  A group
// waits on its row's "full" barrier, reads the row from shared memory with
// 128-bit loads into registers (2 to 5 vectors of 8 bf16 per thread),
// releases the stage on its "empty" mbarrier at once (so the next copy
// starts while it computes), reduces the row within the group (warp
// shuffles, then a named barrier private to the group), normalizes in
// registers and stores with 128-bit streaming stores.  Up to S rows per SM are in flight in the ring and NG
// rows are being computed at once, independent of the register budget.
//
// Register sharing: with SHARE the producer warp group drops to 40
// registers per thread (setmaxnreg.dec) and the consumer warps rise to
// CONS_REGS.  The host only launches the SHARE variant after checking that
// the kernel's launch register count covers the split; otherwise it
// launches the variant without setmaxnreg (same results).
//
// Every mbarrier wait is bounded (2 s on the global timer).  A consumer
// warp that gives up contributes a failure count to its group's reduction
// (a one-warp group needs no count: its lanes vote on the wait), so the
// whole group sees the same outcome and leaves together; the producer,
// on giving up, waits (bounded) for the copies it already issued and
// leaves.  Either records NF_ERR_TIMEOUT in the device status word.
#include "common.cuh"
#include "pairs.cuh"
#include "pdl.cuh"
#include "launch.h"

namespace nf {

// kFusedBwd: the RMSNorm backward of the fused residual add, which also
// stages the residual-stream gradient and adds it to dx.
enum BulkOp { kFused = 0, kRms = 1, kLnFwd = 2, kLnBwd = 3, kRmsBwd = 4, kFusedBwd = 5 };

// Row-group shape: GW warps per row and NG concurrent row groups per CTA.
// Every shape makes the consumer warps a whole number of warp groups (the
// CTA is then 128 * k threads), which setmaxnreg requires: it is executed
// by all four warps of a warp group together, so a partial warp group
// would wait forever.
// Forward: GW warps per row, NGF groups; backward: GWB warps per row, NGB
// groups (backward rows carry column accumulators, so most backward CTAs
// stay at 384 threads, where consumers get 232 registers); the fused-add
// backward (three staged rows) may differ: GWFB, NGFB.  From hidden 2048 up
// the LayerNorm / RMSNorm backward spreads a row over enough warps that
// each thread holds 2 vectors (4 warps at 2048, 8 at 4096, 16 at 8192): a
// row is reduced in fewer serial steps, and at 4096 / 8192 one wide group
// per CTA measured faster than two narrow ones (LayerNorm 0.81 -> 0.89 and
// 0.81 -> 0.92 of the copy peak).  The fused-add backward measured faster
// with its narrower groups, and at 1024 wider groups were slower.
template <int H> struct BulkRow;
template <> struct BulkRow<1024>  { static constexpr int GW = 1,  NGF = 16, GWB = 1,  NGB = 8, GWFB = 1,  NGFB = 8; };
template <> struct BulkRow<2048>  { static constexpr int GW = 2,  NGF = 8,  GWB = 4,  NGB = 2, GWFB = 2,  NGFB = 4; };
template <> struct BulkRow<4096>  { static constexpr int GW = 4,  NGF = 4,  GWB = 8,  NGB = 1, GWFB = 4,  NGFB = 2; };
template <> struct BulkRow<5120>  { static constexpr int GW = 4,  NGF = 4,  GWB = 4,  NGB = 2, GWFB = 4,  NGFB = 2; };  // 5 vectors/thread
template <> struct BulkRow<8192>  { static constexpr int GW = 8,  NGF = 2,  GWB = 16, NGB = 1, GWFB = 8,  NGFB = 1; };
template <> struct BulkRow<12288> { static constexpr int GW = 12, NGF = 1,  GWB = 12, NGB = 1, GWFB = 12, NGFB = 1; };

template <int OP, int H>
struct BulkShape {
    static constexpr bool BWD = OP == 3 || OP == 4 || OP == 5;
    static constexpr int GW = OP == 5 ? BulkRow<H>::GWFB : BWD ? BulkRow<H>::GWB : BulkRow<H>::GW;
    static constexpr int NG = OP == 5 ? BulkRow<H>::NGFB : BWD ? BulkRow<H>::NGB : BulkRow<H>::NGF;
};

constexpr int kSmemBudget = 200 * 1024;  // ring + barriers + reduction scratch
constexpr int kMaxStagesPerGroup = 8;
constexpr int kProducerRegs = 40;
constexpr int kConsumersBarrier = 15;  // named barrier of all consumer threads (groups use 1..NG)

template <int OP> struct OpIO {
    static constexpr int NIN = OP == kFusedBwd ? 3
                               : (OP == kFused || OP == kLnBwd || OP == kRmsBwd) ? 2 : 1;  // staged tensors per row
};

template <int OP, int H>
struct BGeo {
    static constexpr int GW = BulkShape<OP, H>::GW;
    static constexpr int NG = BulkShape<OP, H>::NG;
    static constexpr int GT = GW * 32;                // threads per row group
    static constexpr int NCT = NG * GT;               // consumer threads
    static constexpr int THREADS = 128 + NCT;
    static constexpr int NV = H / kVec;
    static constexpr int VPT = NV / GT;
    static_assert(NV % GT == 0 && VPT >= 1, "whole vectors per consumer thread");
    static_assert(THREADS <= 1024, "CTA size");
    static_assert(THREADS % 128 == 0, "whole warp groups (setmaxnreg)");
    static_assert(GW == 1 || NG <= 15, "named barriers 1..NG");
    static constexpr int ROW_BYTES = H * 2;
    static constexpr int STAGE_BYTES = ROW_BYTES * OpIO<OP>::NIN;
    static constexpr int SG0 = kSmemBudget / STAGE_BYTES / NG;
    static constexpr int SG = SG0 > kMaxStagesPerGroup ? kMaxStagesPerGroup : SG0;  // stages per group
    static_assert(SG >= 2, "need at least two stages per row group");
    static constexpr int S = SG * NG;                  // ring stages
    // registers: the launch allocation, and what consumers get after the
    // producer group drops to kProducerRegs
    static constexpr int LAUNCH_REGS0 = (65536 / THREADS) / 8 * 8;
    static constexpr int LAUNCH_REGS = LAUNCH_REGS0 > 248 ? 248 : LAUNCH_REGS0;
    static constexpr int CONS_REGS0 = (LAUNCH_REGS * THREADS - 128 * kProducerRegs) / NCT / 8 * 8;
    static constexpr int CONS_REGS = CONS_REGS0 > 248 ? 248 : CONS_REGS0;
    // reduction scratch per group: one buffer per row parity, GW x 3 floats each
    static constexpr int RED_PER_GROUP = 2 * GW * 3;
    // dynamic shared memory layout
    static constexpr int RING = S * STAGE_BYTES;
    static constexpr int BAR_OFF = RING;                     // full[S], empty[S]
    static constexpr int RED_OFF = BAR_OFF + 2 * S * 8;
    static constexpr int SMEM = RED_OFF + NG * RED_PER_GROUP * 4;
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_addr(p)));
    return v;
}

// Sum N values over the GW warps of one row group; every thread of the
// group gets the same totals (warps summed in a fixed order).  `rb` is this
// reduction's private GW*N-float buffer.
template <int GW, int N>
__device__ __forceinline__ void group_reduce(float (&v)[N], float* rb, int gwarp, int lane, int gid) {
    warp_sum<N>(v);
    if constexpr (GW > 1) {
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < N; ++i) rb[gwarp * N + i] = v[i];
        }
        named_sync(1 + gid, GW * 32);
#pragma unroll
        for (int i = 0; i < N; ++i) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < GW; ++w) s += rb[w * N + i];
            v[i] = s;
        }
    }
}

// Whether a row group gave up waiting for its row: the summed failure count
// in the last reduced value when the group spans several warps, else the
// warp's own vote.
template <int NF, int N>
__device__ __forceinline__ bool group_failed(const float (&v)[N], bool ok) {
    if constexpr (NF > 0) return v[N - 1] != 0.f;
    else return !ok;
}

struct BulkArgs {
    uint16_t* out0;          // fused: x (in place); rms/ln fwd: y; ln bwd: dx
    uint16_t* out1;          // fused: residual (in place)
    const uint16_t* in0;     // fused: x; rms/ln: x; ln bwd: x
    const uint16_t* in1;     // fused: residual; ln/rms bwd: dy
    const uint16_t* p0;      // weight / gamma
    const uint16_t* p1;      // beta
    const uint16_t* add;     // rms bwd: gradient added to dx (fused-add backward), or null
    float* mean;             // ln fwd out / ln bwd in
    float* rstd;
    float* ws;               // bwd column partials [grid][planes][H], one slot per CTA
    int* status;
    int64_t rows;
    float eps;
};

template <int OP, int H, bool SHARE>
__global__ void __launch_bounds__(BGeo<OP, H>::THREADS, 1)
norm_bulk_kernel(BulkArgs a) {
    using G = BGeo<OP, H>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::BAR_OFF);
    uint64_t* empty = full + G::S;
    const int64_t nct = gridDim.x;
    const int64_t r0 = a.rows * blockIdx.x / nct;
    const int64_t r1 = a.rows * (blockIdx.x + 1) / nct;
    const int n = static_cast<int>(r1 - r0);
    // Launched as a programmatic dependent: nothing is read before the
    // previous grid in the stream has finished.  Only L2 is warmed first
    // with the stripe's first ring-full of rows (a hint; the bulk copies
    // then find them there).
    {
        static_assert(G::ROW_BYTES % 128 == 0, "rows are whole 128-byte lines");
        const int lines = (n < G::S ? n : G::S) * (G::ROW_BYTES / 128);
        const uint8_t* t0 = reinterpret_cast<const uint8_t*>(a.in0 + r0 * H);
        const uint8_t* t1 = OpIO<OP>::NIN >= 2 ? reinterpret_cast<const uint8_t*>(a.in1 + r0 * H) : nullptr;
        const uint8_t* t2 = OpIO<OP>::NIN == 3 ? reinterpret_cast<const uint8_t*>(a.add + r0 * H) : nullptr;
        for (int i = threadIdx.x; i < lines; i += G::THREADS) {
            prefetch_l2(t0 + i * 128);
            if (t1) prefetch_l2(t1 + i * 128);
            if (t2) prefetch_l2(t2 + i * 128);
        }
    }
    grid_dep_wait();

    if (threadIdx.x == 0) {
        for (int s = 0; s < G::S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], G::GW);  // the GW warps of the group that consumed it
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (threadIdx.x < 128) {
        // ---------------- producer warp group
        if constexpr (SHARE) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
        // One producer thread per producer warp (lane 0 of warps
        // 0..NPROD-1); warp w serves the row groups g with g % NPROD == w.
        // Groups own private ring slices, so two producers never touch the
        // same stage, and each group's rows are issued in order.
        constexpr int NPROD = G::NG < 4 ? G::NG : 4;
        constexpr int GPP = G::NG / NPROD;  // groups per producer
        const int pw = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0 && pw < NPROD) {
            int issued[GPP];
#pragma unroll
            for (int k = 0; k < GPP; ++k) issued[k] = 0;
            bool ok = true;
            const int qmax = (n + G::NG - 1) / G::NG;
            for (int q = 0; q < qmax && ok; ++q) {
#pragma unroll
                for (int k = 0; k < GPP; ++k) {
                    const int g = pw + k * NPROD;
                    const int i = g + q * G::NG;
                    if (!ok || i >= n) continue;
                    const int s = g * G::SG + q % G::SG;
                    const uint32_t par = ((q / G::SG) & 1) ^ 1;
                    if (!mbar_wait(&empty[s], par, kWaitLimitNs)) { ok = false; continue; }
                    mbar_arrive_expect_tx(&full[s], G::STAGE_BYTES);
                    const int64_t row = r0 + i;
                    uint8_t* st = smem + s * G::STAGE_BYTES;
                    bulk_g2s(smem_addr(st), a.in0 + row * H, G::ROW_BYTES, &full[s]);
                    if constexpr (OpIO<OP>::NIN >= 2)
                        bulk_g2s(smem_addr(st + G::ROW_BYTES), a.in1 + row * H, G::ROW_BYTES, &full[s]);
                    if constexpr (OpIO<OP>::NIN == 3)
                        bulk_g2s(smem_addr(st + 2 * G::ROW_BYTES), a.add + row * H, G::ROW_BYTES, &full[s]);
                    issued[k] = q + 1;
                }
            }
            if (!ok) {
                record_status(a.status, kStatusTimeout);
                // let the copies already issued land before the CTA can exit
                // (a group's last SG issued rows cover each of its stages once)
#pragma unroll
                for (int k = 0; k < GPP; ++k) {
                    const int g = pw + k * NPROD;
                    const int first = issued[k] > G::SG ? issued[k] - G::SG : 0;
                    for (int q = first; q < issued[k]; ++q)
                        mbar_wait(&full[g * G::SG + q % G::SG], (q / G::SG) & 1, kWaitLimitNs / 4);
                }
            }
        }
        return;
    }

    // ---------------- consumer row groups
    if constexpr (SHARE) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(G::CONS_REGS));
    const int ct = threadIdx.x - 128;
    const int gid = ct / G::GT;          // row group
    const int gt = ct % G::GT;           // thread within the group
    const int gwarp = gt >> 5, lane = gt & 31;
    float* red = reinterpret_cast<float*>(smem + G::RED_OFF) + gid * G::RED_PER_GROUP;

    uint4 prm0[G::VPT];  // weight / gamma, loaded once (beta is re-read from L1 per row)
#pragma unroll
    for (int k = 0; k < G::VPT; ++k) {
        prm0[k] = ld_param(a.p0 + (k * G::GT + gt) * kVec);
    }
    constexpr bool kRmsB = OP == kRmsBwd || OP == kFusedBwd;
    constexpr bool kBwd = OP == kLnBwd || kRmsB;
    // Backward consumers with a large register share keep gamma / w widened
    // to fp32 for the whole stripe, so no row re-widens it; with a smaller
    // share (the 512-thread hidden-12288 shape) it stays packed.  All the
    // elementwise arithmetic runs on fp32 pairs (add / mul / fma .f32x2).
    constexpr bool kCacheW = kBwd && G::CONS_REGS >= 200;
    float2 wf[kCacheW ? G::VPT : 1][4];
    if constexpr (kCacheW) {
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) unpack8x2(prm0[k], wf[k]);
    }
    float2 acc_g[kBwd ? G::VPT : 1][4], acc_b[OP == kLnBwd ? G::VPT : 1][4];
    if constexpr (kBwd) {
#pragma unroll
        for (int k = 0; k < G::VPT; ++k)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc_g[k][q] = make_float2(0.f, 0.f);
    }
    if constexpr (OP == kLnBwd) {
#pragma unroll
        for (int k = 0; k < G::VPT; ++k)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc_b[k][q] = make_float2(0.f, 0.f);
    }
    // saved statistics of the group's next rows, fetched ahead
    // (a queue kStatAhead rows deep, shifted by one each row: no dynamic
    // indexing, and the loads have several rows of work to land; at hidden
    // 1024, 8 rows deep measured 0.687 of the copy peak against 0.681 for 4
    // and 0.666 for 1)
    constexpr int kStatAhead = OP == kLnBwd ? 8 : 1;
    float qmu[kStatAhead], qrs[kStatAhead];
#pragma unroll
    for (int d = 0; d < kStatAhead; ++d) {
        qmu[d] = 0.f;
        qrs[d] = 0.f;
        if constexpr (OP == kLnBwd) {
            const int ii = gid + d * G::NG;
            if (ii < n) { qmu[d] = __ldg(a.mean + r0 + ii); qrs[d] = __ldg(a.rstd + r0 + ii); }
        }
    }

    bool failed = false;
    int j = 0;  // this group's row counter (selects the reduction buffers)
    for (int i = gid; i < n; i += G::NG, ++j) {
        const int s = gid * G::SG + j % G::SG;   // j == i / NG
        const uint32_t par = (j / G::SG) & 1;
        const int64_t row = r0 + i;
        const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&full[s], par, kWaitLimitNs));
        const float fail = ok ? 0.f : 1.f;
        // A one-warp group already agrees on `ok` (the vote above); wider
        // groups sum the failures with the row's reduction.
        constexpr int NF = G::GW > 1 ? 1 : 0;
        const uint8_t* st = smem + s * G::STAGE_BYTES;
        uint4 v0[G::VPT], v1[G::VPT], v2[OpIO<OP>::NIN == 3 ? G::VPT : 1];
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            v0[k] = lds128(st + (k * G::GT + gt) * 16);
            if constexpr (OpIO<OP>::NIN >= 2) v1[k] = lds128(st + G::ROW_BYTES + (k * G::GT + gt) * 16);
            if constexpr (OpIO<OP>::NIN == 3) v2[k] = lds128(st + 2 * G::ROW_BYTES + (k * G::GT + gt) * 16);
        }
        // LayerNorm shift: the row's first element, read before the stage is released
        float c = 0.f;
        if constexpr (OP == kLnFwd) c = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(st));
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the stage may be refilled now
        float* rb0 = red + (j & 1) * G::GW * 3;

        if constexpr (OP == kFused || OP == kRms) {
            float2 f[G::VPT][4];
            float2 ss = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                unpack8x2(v0[k], f[k]);
                if constexpr (OP == kFused) {
                    float2 b[4];
                    unpack8x2(v1[k], b);
#pragma unroll
                    for (int q = 0; q < 4; ++q) f[k][q] = __fadd2_rn(f[k][q], b[q]);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) ss = __ffma2_rn(f[k][q], f[k][q], ss);
            }
            float v[1 + NF] = {ss.x + ss.y};
            if constexpr (NF) v[1] = fail;
            group_reduce<G::GW, 1 + NF>(v, rb0, gwarp, lane, gid);
            if (group_failed<NF>(v, ok)) { failed = true; break; }
            if constexpr (OP == kFused) {
#pragma unroll
                for (int k = 0; k < G::VPT; ++k)
                    st_stream(a.out1 + row * H + (k * G::GT + gt) * kVec, pack8x2(f[k]));
            }
            const float rstd = rsqrtf(v[0] * (1.0f / H) + a.eps);
            const float2 rstd2 = make_float2(rstd, rstd);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float2 w[4], o[4];
                unpack8x2(prm0[k], w);
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = __fmul2_rn(__fmul2_rn(f[k][q], rstd2), w[q]);
                st_stream(a.out0 + row * H + (k * G::GT + gt) * kVec, pack8x2(o));
            }
        } else if constexpr (OP == kLnFwd) {
            // one reduction of the shifted sums: with d = x - c,
            // mean = c + sum d / H and var = sum d^2 / H - (sum d / H)^2
            float2 f[G::VPT][4];
            const float2 nc2 = make_float2(-c, -c);
            float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                unpack8x2(v0[k], f[k]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 d = __fadd2_rn(f[k][q], nc2);
                    s1 = __fadd2_rn(s1, d);
                    s2 = __ffma2_rn(d, d, s2);
                }
            }
            float v[2 + NF] = {s1.x + s1.y, s2.x + s2.y};
            if constexpr (NF) v[2] = fail;
            group_reduce<G::GW, 2 + NF>(v, rb0, gwarp, lane, gid);
            if (group_failed<NF>(v, ok)) { failed = true; break; }
            const float dm = v[0] * (1.0f / H);
            const float mean = c + dm;
            const float var = fmaxf(v[1] * (1.0f / H) - dm * dm, 0.f);
            const float rstd = rsqrtf(var + a.eps);
            const float2 nmean2 = make_float2(-mean, -mean);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k)
#pragma unroll
                for (int q = 0; q < 4; ++q) f[k][q] = __fadd2_rn(f[k][q], nmean2);  // the row, centered
            const float2 rstd2 = make_float2(rstd, rstd);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float2 g[4], b[4], o[4];
                unpack8x2(prm0[k], g);
                unpack8x2(ld_param(a.p1 + (k * G::GT + gt) * kVec), b);
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = __ffma2_rn(f[k][q], __fmul2_rn(rstd2, g[q]), b[q]);
                st_stream(a.out0 + row * H + (k * G::GT + gt) * kVec, pack8x2(o));
            }
            if (gt == 0) {
                if (a.mean) a.mean[row] = mean;
                if (a.rstd) a.rstd[row] = rstd;
            }
        } else if constexpr (kRmsB) {
            // rstd recomputed from the row: rs = rsqrt(sum x^2 / H + eps),
            // dx = rs * g - x * (rs^3 * sum(g x) / H) with g = dy * w
            // the row is widened once when the register share allows,
            // otherwise vector by vector on each pass
            float2 xf[kCacheW ? G::VPT : 1][4], df[kCacheW ? G::VPT : 1][4];
            float2 sxx = make_float2(0.f, 0.f), sgx = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float2 xk[4], dk[4], wk[4];
                unpack8x2(v0[k], xk);
                unpack8x2(v1[k], dk);
                if constexpr (kCacheW) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) { xf[k][q] = xk[q]; df[k][q] = dk[q]; wk[q] = wf[k][q]; }
                } else {
                    unpack8x2(prm0[k], wk);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    sxx = __ffma2_rn(xk[q], xk[q], sxx);
                    sgx = __ffma2_rn(__fmul2_rn(dk[q], wk[q]), xk[q], sgx);
                }
            }
            float v[2 + NF] = {sxx.x + sxx.y, sgx.x + sgx.y};
            if constexpr (NF) v[2] = fail;
            group_reduce<G::GW, 2 + NF>(v, rb0, gwarp, lane, gid);
            if (group_failed<NF>(v, ok)) { failed = true; break; }
            const float rs = rsqrtf(v[0] * (1.0f / H) + a.eps);
            const float c = rs * rs * rs * v[1] * (1.0f / H);
            const float2 rs2 = make_float2(rs, rs), nc2 = make_float2(-c, -c);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float2 xk[4], dk[4], wk[4], o[4];
                if constexpr (kCacheW) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) { xk[q] = xf[k][q]; dk[q] = df[k][q]; wk[q] = wf[k][q]; }
                } else {
                    unpack8x2(v0[k], xk);
                    unpack8x2(v1[k], dk);
                    unpack8x2(prm0[k], wk);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    o[q] = __ffma2_rn(xk[q], nc2, __fmul2_rn(rs2, __fmul2_rn(dk[q], wk[q])));
                    acc_g[k][q] = __ffma2_rn(__fmul2_rn(dk[q], xk[q]), rs2, acc_g[k][q]);
                }
                if constexpr (OP == kFusedBwd) {  // + the residual-stream gradient
                    float2 af[4];
                    unpack8x2(v2[k], af);
#pragma unroll
                    for (int q = 0; q < 4; ++q) o[q] = __fadd2_rn(o[q], af[q]);
                }
                st_stream(a.out0 + row * H + (k * G::GT + gt) * kVec, pack8x2(o));
            }
        } else {  // kLnBwd
            // xhat = x * rstd - mean * rstd (one fma), g = dy * gamma;
            // dx = rstd * g - rstd * A - xhat * (rstd * B)
            const float mu = qmu[0], rs = qrs[0];
#pragma unroll
            for (int d = 0; d + 1 < kStatAhead; ++d) {
                qmu[d] = qmu[d + 1];
                qrs[d] = qrs[d + 1];
            }
            if (i + kStatAhead * G::NG < n) {
                qmu[kStatAhead - 1] = __ldg(a.mean + row + kStatAhead * G::NG);
                qrs[kStatAhead - 1] = __ldg(a.rstd + row + kStatAhead * G::NG);
            }
            const float nmr = -mu * rs;
            const float2 rs2 = make_float2(rs, rs), nmr2 = make_float2(nmr, nmr);
            float2 xf[kCacheW ? G::VPT : 1][4], df[kCacheW ? G::VPT : 1][4];
            float2 sg = make_float2(0.f, 0.f), sgx = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float2 xk[4], dk[4], wk[4];
                unpack8x2(v0[k], xk);
                unpack8x2(v1[k], dk);
                if constexpr (kCacheW) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) { xf[k][q] = xk[q]; df[k][q] = dk[q]; wk[q] = wf[k][q]; }
                } else {
                    unpack8x2(prm0[k], wk);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 xh = __ffma2_rn(xk[q], rs2, nmr2);
                    const float2 g = __fmul2_rn(dk[q], wk[q]);
                    sg = __fadd2_rn(sg, g);
                    sgx = __ffma2_rn(g, xh, sgx);
                    acc_g[k][q] = __ffma2_rn(dk[q], xh, acc_g[k][q]);
                    acc_b[k][q] = __fadd2_rn(acc_b[k][q], dk[q]);
                }
            }
            float v[2 + NF] = {sg.x + sg.y, sgx.x + sgx.y};
            if constexpr (NF) v[2] = fail;
            group_reduce<G::GW, 2 + NF>(v, rb0, gwarp, lane, gid);
            if (group_failed<NF>(v, ok)) { failed = true; break; }
            const float rsA = rs * v[0] * (1.0f / H), rsB = rs * v[1] * (1.0f / H);
            const float2 nrsA2 = make_float2(-rsA, -rsA), nrsB2 = make_float2(-rsB, -rsB);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float2 xk[4], dk[4], wk[4], o[4];
                if constexpr (kCacheW) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) { xk[q] = xf[k][q]; dk[q] = df[k][q]; wk[q] = wf[k][q]; }
                } else {
                    unpack8x2(v0[k], xk);
                    unpack8x2(v1[k], dk);
                    unpack8x2(prm0[k], wk);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 xh = __ffma2_rn(xk[q], rs2, nmr2);
                    o[q] = __ffma2_rn(xh, nrsB2, __ffma2_rn(rs2, __fmul2_rn(dk[q], wk[q]), nrsA2));
                }
                st_stream(a.out0 + row * H + (k * G::GT + gt) * kVec, pack8x2(o));
            }
        }
    }
    // This CTA's rows are done: let a programmatically dependent launch
    // (the column reduction of the backward ops) start scheduling.  It still
    // waits for this grid to finish before it reads anything.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if constexpr (kBwd) {
        // Fold the NG groups' column partials into one slot per CTA, in
        // group order: each group parks its partials in its own ring slice
        // (all of its rows are consumed, so no copy targets that slice any
        // more), every consumer thread meets at a consumer-wide barrier --
        // failed groups too, so nobody waits on a missing warp -- and the
        // consumers then sum the slices column by column.
        constexpr int NP = OP == kLnBwd ? 2 : 1;
        static_assert(G::SG * G::STAGE_BYTES >= NP * H * 4, "ring slice holds a group's partials");
        float* mine = reinterpret_cast<float*>(smem + gid * G::SG * G::STAGE_BYTES);
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            const int jj = (k * G::GT + gt) * kVec;
            reinterpret_cast<float4*>(mine + jj)[0] = make_float4(acc_g[k][0].x, acc_g[k][0].y, acc_g[k][1].x, acc_g[k][1].y);
            reinterpret_cast<float4*>(mine + jj)[1] = make_float4(acc_g[k][2].x, acc_g[k][2].y, acc_g[k][3].x, acc_g[k][3].y);
            if constexpr (NP == 2) {
                reinterpret_cast<float4*>(mine + H + jj)[0] = make_float4(acc_b[k][0].x, acc_b[k][0].y, acc_b[k][1].x, acc_b[k][1].y);
                reinterpret_cast<float4*>(mine + H + jj)[1] = make_float4(acc_b[k][2].x, acc_b[k][2].y, acc_b[k][3].x, acc_b[k][3].y);
            }
        }
        named_sync(kConsumersBarrier, G::NCT);
        float4* out = reinterpret_cast<float4*>(a.ws + static_cast<int64_t>(blockIdx.x) * NP * H);
        for (int c4 = ct; c4 < NP * H / 4; c4 += G::NCT) {
            float4 acc = reinterpret_cast<const float4*>(smem)[c4];
#pragma unroll
            for (int g = 1; g < G::NG; ++g) {
                const float4 v = reinterpret_cast<const float4*>(smem + g * G::SG * G::STAGE_BYTES)[c4];
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
            out[c4] = acc;
        }
    }
    if (failed && gt == 0) record_status(a.status, kStatusTimeout);
}

namespace {

template <int OP, int H>
cudaError_t launch_bulk_t(const BulkArgs& a, int grid, cudaStream_t st) {
    using G = BGeo<OP, H>;
    // Pick the register-sharing variant only when the launch allocation
    // covers the split (otherwise setmaxnreg.inc could wait forever) and
    // the consumers really gain registers.  Per process (the binary is the
    // same on every device); a benign race at worst repeats the query.
    static int share_ok = -1;
    static bool attr_set[2] = {false, false};
    if (share_ok < 0) {
        cudaFuncAttributes fa;
        int ok = 0;
        if (cudaFuncGetAttributes(&fa, norm_bulk_kernel<OP, H, true>) == cudaSuccess) {
            const long pool = static_cast<long>(fa.numRegs) * G::THREADS;
            const long need = 128L * kProducerRegs + static_cast<long>(G::NCT) * G::CONS_REGS;
            ok = (G::THREADS % 128 == 0 && fa.numRegs >= kProducerRegs &&
                  fa.numRegs < G::CONS_REGS && pool >= need) ? 1 : 0;
        }
        share_ok = ok;
    }
    if (share_ok) {
        if (!attr_set[1]) {
            cudaError_t e = cudaFuncSetAttribute(norm_bulk_kernel<OP, H, true>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
            if (e != cudaSuccess) return e;
            attr_set[1] = true;
        }
        return launch_with_pdl(norm_bulk_kernel<OP, H, true>, dim3(grid), dim3(G::THREADS), G::SMEM,
                               st, a);
    } else {
        if (!attr_set[0]) {
            cudaError_t e = cudaFuncSetAttribute(norm_bulk_kernel<OP, H, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
            if (e != cudaSuccess) return e;
            attr_set[0] = true;
        }
        return launch_with_pdl(norm_bulk_kernel<OP, H, false>, dim3(grid), dim3(G::THREADS), G::SMEM,
                               st, a);
    }
    return cudaGetLastError();
}

template <int OP>
cudaError_t launch_bulk_op(int64_t hidden, const BulkArgs& a, int grid, cudaStream_t st) {
    NF_HIDDEN_SWITCH(hidden, { return launch_bulk_t<OP, H>(a, grid, st); })
}

template <int OP>
bool shape_of(int64_t hidden, int* threads, int* stages, int* smem, int* groups) {
    switch (hidden) {
#define NF_BULK_CASE(HV)                                                                \
        case HV: *threads = BGeo<OP, HV>::THREADS; *stages = BGeo<OP, HV>::S;           \
                 *smem = BGeo<OP, HV>::SMEM; *groups = BGeo<OP, HV>::NG; return true;
        NF_BULK_CASE(1024) NF_BULK_CASE(2048) NF_BULK_CASE(4096)
        NF_BULK_CASE(5120) NF_BULK_CASE(8192) NF_BULK_CASE(12288)
#undef NF_BULK_CASE
        default: return false;
    }
}

}  // namespace

bool bulk_shape(int op, int64_t hidden, int* threads, int* stages, int* smem_bytes, int* groups) {
    int gm;
    if ((op == kLnBwd || op == kRmsBwd) &&
        rows_bwd_shape(op, hidden, threads, stages, smem_bytes, groups, &gm))
        return true;
    switch (op) {
        case kFused: return shape_of<kFused>(hidden, threads, stages, smem_bytes, groups);
        case kRms: return shape_of<kRms>(hidden, threads, stages, smem_bytes, groups);
        case kLnFwd: return shape_of<kLnFwd>(hidden, threads, stages, smem_bytes, groups);
        case kLnBwd: return shape_of<kLnBwd>(hidden, threads, stages, smem_bytes, groups);
        case kRmsBwd: return shape_of<kRmsBwd>(hidden, threads, stages, smem_bytes, groups);
        default: return false;
    }
}

cudaError_t launch_fused_bulk(int64_t hidden, void* x, void* res, const void* w, int64_t rows,
                              float eps, int grid, int* status, cudaStream_t st) {
    BulkArgs a{};
    a.out0 = static_cast<uint16_t*>(x);
    a.out1 = static_cast<uint16_t*>(res);
    a.in0 = static_cast<const uint16_t*>(x);
    a.in1 = static_cast<const uint16_t*>(res);
    a.p0 = static_cast<const uint16_t*>(w);
    a.status = status;
    a.rows = rows;
    a.eps = eps;
    return launch_bulk_op<kFused>(hidden, a, grid, st);
}

cudaError_t launch_rms_bulk(int64_t hidden, void* y, const void* x, const void* w, int64_t rows,
                            float eps, int grid, int* status, cudaStream_t st) {
    BulkArgs a{};
    a.out0 = static_cast<uint16_t*>(y);
    a.in0 = static_cast<const uint16_t*>(x);
    a.p0 = static_cast<const uint16_t*>(w);
    a.status = status;
    a.rows = rows;
    a.eps = eps;
    return launch_bulk_op<kRms>(hidden, a, grid, st);
}

cudaError_t launch_ln_fwd_bulk(int64_t hidden, void* y, float* mean, float* rstd, const void* x,
                               const void* gamma, const void* beta, int64_t rows, float eps,
                               int grid, int* status, cudaStream_t st) {
    BulkArgs a{};
    a.out0 = static_cast<uint16_t*>(y);
    a.in0 = static_cast<const uint16_t*>(x);
    a.p0 = static_cast<const uint16_t*>(gamma);
    a.p1 = static_cast<const uint16_t*>(beta);
    a.mean = mean;
    a.rstd = rstd;
    a.status = status;
    a.rows = rows;
    a.eps = eps;
    return launch_bulk_op<kLnFwd>(hidden, a, grid, st);
}

cudaError_t launch_ln_bwd_bulk(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                               const float* mean, const float* rstd, const void* gamma,
                               int64_t rows, int grid, int* status, cudaStream_t st) {
    int t, sg, sm, ng, gm;
    if (rows_bwd_shape(kLnBwd, hidden, &t, &sg, &sm, &ng, &gm))
        return launch_ln_bwd_rows(hidden, dx, ws, dy, x, mean, rstd, gamma, rows, grid, status, st);
    BulkArgs a{};
    a.out0 = static_cast<uint16_t*>(dx);
    a.in0 = static_cast<const uint16_t*>(x);
    a.in1 = static_cast<const uint16_t*>(dy);
    a.p0 = static_cast<const uint16_t*>(gamma);
    a.mean = const_cast<float*>(mean);
    a.rstd = const_cast<float*>(rstd);
    a.ws = ws;
    a.status = status;
    a.rows = rows;
    return launch_bulk_op<kLnBwd>(hidden, a, grid, st);
}

cudaError_t launch_rms_bwd_bulk(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                                const void* dres, const void* w, int64_t rows, float eps, int grid,
                                int* status, cudaStream_t st) {
    int t, sg, sm, ng, gm;
    if (rows_bwd_shape(kRmsBwd, hidden, &t, &sg, &sm, &ng, &gm))
        return launch_rms_bwd_rows(hidden, dx, ws, dy, x, dres, w, rows, eps, grid, status, st);
    BulkArgs a{};
    a.out0 = static_cast<uint16_t*>(dx);
    a.in0 = static_cast<const uint16_t*>(x);
    a.in1 = static_cast<const uint16_t*>(dy);
    a.add = static_cast<const uint16_t*>(dres);
    a.p0 = static_cast<const uint16_t*>(w);
    a.ws = ws;
    a.status = status;
    a.rows = rows;
    a.eps = eps;
    return dres ? launch_bulk_op<kFusedBwd>(hidden, a, grid, st)
                : launch_bulk_op<kRmsBwd>(hidden, a, grid, st);
}

}  // namespace nf
