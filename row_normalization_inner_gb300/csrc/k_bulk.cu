// Bulk-copy staged kernels ("TMA inner persistent scheduler", NVIDIA/Fuser
// PR #5587: a TMA path beside the non-TMA one, vectorized smem-to-register
// loads, and register sharing between the copy branch and the compute
// branch).
//
// One persistent CTA per SM walks a contiguous stripe of rows.  Warp group 0
// is the producer: one elected thread issues, per row, one 1-D bulk
// asynchronous copy (cp.async.bulk, global -> this CTA's shared memory) per
// input tensor into a ring of S stages, each completing on the stage's
// "full" mbarrier.  The remaining NCWG warp groups are consumers: they wait
// on "full", read the row from shared memory with 128-bit loads into
// registers, release the stage on its "empty" mbarrier at once (so the next
// copy starts while they still compute), reduce and normalize the row in
// registers and store the results with 128-bit streaming stores.  So up to
// S rows per SM are in flight regardless of the register budget.
//
// Register sharing: with SHARE the producer warp group drops to 40
// registers per thread (setmaxnreg.dec) and the consumer groups rise to
// CONS_REGS.  The host only launches the SHARE variant after checking that
// the kernel's launch register count covers the split; otherwise it
// launches the variant without setmaxnreg (same results).
//
// Every mbarrier wait is bounded (2 s on the global timer).  A consumer
// that gives up raises a CTA-wide flag that all consumer warps read after
// the next consumer barrier, so they leave together; the producer, on
// giving up, waits (bounded) for the copies it already issued and leaves.
// Either records NF_ERR_TIMEOUT in the device status word.
#include "common.cuh"
#include "launch.h"

namespace nf {

enum BulkOp { kFused = 0, kRms = 1, kLnFwd = 2, kLnBwd = 3 };

template <int H> struct BulkShape;
// NCWG consumer warp groups per CTA (so 128 * NCWG consumer threads).
template <> struct BulkShape<1024>  { static constexpr int NCWG = 1; };
template <> struct BulkShape<2048>  { static constexpr int NCWG = 1; };
template <> struct BulkShape<4096>  { static constexpr int NCWG = 1; };
template <> struct BulkShape<5120>  { static constexpr int NCWG = 1; };
template <> struct BulkShape<8192>  { static constexpr int NCWG = 2; };
template <> struct BulkShape<12288> { static constexpr int NCWG = 2; };

constexpr int kSmemBudget = 200 * 1024;  // ring + barriers + reduction scratch
constexpr int kMaxStages = 16;
constexpr int kProducerRegs = 40;

template <int OP> struct OpIO {
    static constexpr int NIN = (OP == kFused || OP == kLnBwd) ? 2 : 1;  // staged tensors per row
};

template <int OP, int H>
struct BGeo {
    static constexpr int NCWG = BulkShape<H>::NCWG;
    static constexpr int NCT = 128 * NCWG;            // consumer threads
    static constexpr int NCW = NCT / 32;              // consumer warps
    static constexpr int THREADS = 128 + NCT;
    static constexpr int NV = H / kVec;
    static constexpr int VPT = NV / NCT;
    static_assert(NV % NCT == 0, "row must split evenly over the consumer threads");
    static constexpr int ROW_BYTES = H * 2;
    static constexpr int STAGE_BYTES = ROW_BYTES * OpIO<OP>::NIN;
    static constexpr int S0 = kSmemBudget / STAGE_BYTES;
    static constexpr int S = S0 > kMaxStages ? kMaxStages : S0;
    static_assert(S >= 2, "need at least two stages");
    // consumer register target: what the launch allocation leaves after the producer drops to 40
    static constexpr int LAUNCH_REGS = (65536 / THREADS) / 8 * 8 > 255 ? 248 : (65536 / THREADS) / 8 * 8;
    static constexpr int CONS_REGS_RAW = (LAUNCH_REGS * THREADS - 128 * kProducerRegs) / NCT / 8 * 8;
    static constexpr int CONS_REGS = CONS_REGS_RAW > 248 ? 248 : CONS_REGS_RAW;
    // dynamic shared memory layout
    static constexpr int RING = S * STAGE_BYTES;
    static constexpr int BAR_OFF = RING;                    // full[S], empty[S]
    static constexpr int RED_OFF = BAR_OFF + 2 * S * 8;     // 2 buffers x NCW x 2 floats
    static constexpr int FLAG_OFF = RED_OFF + 2 * NCW * 2 * 4;
    static constexpr int SMEM = FLAG_OFF + 16;
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void consumer_sync(int nct) {
    asm volatile("bar.sync 1, %0;" ::"r"(nct) : "memory");
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_addr(p)));
    return v;
}

template <int N>
__device__ __forceinline__ void consumer_sum(float (&v)[N], float* red, int ct, int ncw, int nct) {
    warp_sum<N>(v);
    const int warp = ct >> 5, lane = ct & 31;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i) red[warp * N + i] = v[i];
    }
    consumer_sync(nct);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        float s = 0.f;
        for (int w = 0; w < ncw; ++w) s += red[w * N + i];
        v[i] = s;
    }
}

struct BulkArgs {
    uint16_t* out0;          // fused: x (in place); rms/ln fwd: y; ln bwd: dx
    uint16_t* out1;          // fused: residual (in place)
    const uint16_t* in0;     // fused: x; rms/ln: x; ln bwd: x
    const uint16_t* in1;     // fused: residual; ln bwd: dy
    const uint16_t* p0;      // weight / gamma
    const uint16_t* p1;      // beta
    float* mean;             // ln fwd out / ln bwd in
    float* rstd;
    float* ws;               // ln bwd column partials [grid][2][H]
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
    float* red = reinterpret_cast<float*>(smem + G::RED_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::FLAG_OFF);

    const int64_t nct = gridDim.x;
    const int64_t r0 = a.rows * blockIdx.x / nct;
    const int64_t r1 = a.rows * (blockIdx.x + 1) / nct;
    const int n = static_cast<int>(r1 - r0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < G::S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], G::NCW);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (threadIdx.x < 128) {
        // ---------------- producer warp group
        if constexpr (SHARE) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
        if (threadIdx.x == 0) {
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < n; ++i) {
                const int s = i % G::S;
                const uint32_t par = ((i / G::S) & 1) ^ 1;
                if (!mbar_wait(&empty[s], par, kWaitLimitNs)) { ok = false; break; }
                mbar_arrive_expect_tx(&full[s], G::STAGE_BYTES);
                const int64_t row = r0 + i;
                uint8_t* st = smem + s * G::STAGE_BYTES;
                bulk_g2s(smem_addr(st), a.in0 + row * H, G::ROW_BYTES, &full[s]);
                if constexpr (OpIO<OP>::NIN == 2)
                    bulk_g2s(smem_addr(st + G::ROW_BYTES), a.in1 + row * H, G::ROW_BYTES, &full[s]);
                issued = i + 1;
            }
            if (!ok) {
                record_status(a.status, kStatusTimeout);
                // let the copies already issued land before the CTA can exit
                const int first = issued > G::S ? issued - G::S : 0;
                for (int i = first; i < issued; ++i)
                    mbar_wait(&full[i % G::S], (i / G::S) & 1, kWaitLimitNs / 4);
            }
        }
        return;
    }

    // ---------------- consumer warp groups
    if constexpr (SHARE) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(G::CONS_REGS));
    const int ct = threadIdx.x - 128;
    const int lane = ct & 31;

    uint4 prm0[G::VPT], prm1[G::VPT];  // weight/gamma and beta, loaded once
#pragma unroll
    for (int k = 0; k < G::VPT; ++k) {
        prm0[k] = ld_param(a.p0 + (k * G::NCT + ct) * kVec);
        if constexpr (OP == kLnFwd) prm1[k] = ld_param(a.p1 + (k * G::NCT + ct) * kVec);
        else prm1[k] = make_uint4(0, 0, 0, 0);
    }
    float acc_g[OP == kLnBwd ? G::VPT : 1][8], acc_b[OP == kLnBwd ? G::VPT : 1][8];
    if constexpr (OP == kLnBwd) {
#pragma unroll
        for (int k = 0; k < G::VPT; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) { acc_g[k][e] = 0.f; acc_b[k][e] = 0.f; }
    }
    // saved statistics of the next row, fetched one row ahead
    float nmu = 0.f, nrs = 0.f;
    if constexpr (OP == kLnBwd) {
        if (n > 0) { nmu = __ldg(a.mean + r0); nrs = __ldg(a.rstd + r0); }
    }

    for (int i = 0; i < n; ++i) {
        const int s = i % G::S;
        const uint32_t par = (i / G::S) & 1;
        const int64_t row = r0 + i;
        if (!mbar_wait(&full[s], par, kWaitLimitNs)) *abort_flag = 1;
        const uint8_t* st = smem + s * G::STAGE_BYTES;
        uint4 v0[G::VPT], v1[G::VPT];
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            v0[k] = lds128(st + (k * G::NCT + ct) * 16);
            if constexpr (OpIO<OP>::NIN == 2) v1[k] = lds128(st + G::ROW_BYTES + (k * G::NCT + ct) * 16);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the stage may be refilled now
        float* rb = red + (i & 1) * G::NCW * 2;

        if constexpr (OP == kFused || OP == kRms) {
            float f[G::VPT][8];
            float ss[1] = {0.f};
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                unpack8(v0[k], f[k]);
                if constexpr (OP == kFused) {
                    float b[8];
                    unpack8(v1[k], b);
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[k][e] += b[e];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) ss[0] += f[k][e] * f[k][e];
            }
            consumer_sum<1>(ss, rb, ct, G::NCW, G::NCT);
            if (*abort_flag) break;
            if constexpr (OP == kFused) {
#pragma unroll
                for (int k = 0; k < G::VPT; ++k)
                    st_stream(a.out1 + row * H + (k * G::NCT + ct) * kVec, pack8(f[k]));
            }
            const float rstd = rsqrtf(ss[0] * (1.0f / H) + a.eps);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float w[8], o[8];
                unpack8(prm0[k], w);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = f[k][e] * rstd * w[e];
                st_stream(a.out0 + row * H + (k * G::NCT + ct) * kVec, pack8(o));
            }
        } else if constexpr (OP == kLnFwd) {
            float f[G::VPT][8];
            float sm[1] = {0.f};
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                unpack8(v0[k], f[k]);
#pragma unroll
                for (int e = 0; e < 8; ++e) sm[0] += f[k][e];
            }
            consumer_sum<1>(sm, rb, ct, G::NCW, G::NCT);
            if (*abort_flag) break;
            const float mean = sm[0] * (1.0f / H);
            float sq[1] = {0.f};
#pragma unroll
            for (int k = 0; k < G::VPT; ++k)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float d = f[k][e] - mean;
                    sq[0] += d * d;
                }
            consumer_sum<1>(sq, rb + G::NCW, ct, G::NCW, G::NCT);
            const float rstd = rsqrtf(sq[0] * (1.0f / H) + a.eps);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float g[8], b[8], o[8];
                unpack8(prm0[k], g);
                unpack8(prm1[k], b);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = (f[k][e] - mean) * rstd * g[e] + b[e];
                st_stream(a.out0 + row * H + (k * G::NCT + ct) * kVec, pack8(o));
            }
            if (ct == 0) {
                if (a.mean) a.mean[row] = mean;
                if (a.rstd) a.rstd[row] = rstd;
            }
        } else {  // kLnBwd
            const float mu = nmu, rs = nrs;
            if (i + 1 < n) { nmu = __ldg(a.mean + row + 1); nrs = __ldg(a.rstd + row + 1); }
            float v[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float xf[8], df[8], gf[8];
                unpack8(v0[k], xf);
                unpack8(v1[k], df);
                unpack8(prm0[k], gf);
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
            consumer_sum<2>(v, rb, ct, G::NCW, G::NCT);
            if (*abort_flag) break;
            const float A = v[0] * (1.0f / H), B = v[1] * (1.0f / H);
#pragma unroll
            for (int k = 0; k < G::VPT; ++k) {
                float xf[8], df[8], gf[8], o[8];
                unpack8(v0[k], xf);
                unpack8(v1[k], df);
                unpack8(prm0[k], gf);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = rs * (df[e] * gf[e] - A - (xf[e] - mu) * rs * B);
                st_stream(a.out0 + row * H + (k * G::NCT + ct) * kVec, pack8(o));
            }
        }
    }
    if (*abort_flag) {
        if (ct == 0) record_status(a.status, kStatusTimeout);
        return;
    }
    if constexpr (OP == kLnBwd) {
        float* wg = a.ws + static_cast<int64_t>(blockIdx.x) * 2 * H;
        float* wb = wg + H;
#pragma unroll
        for (int k = 0; k < G::VPT; ++k) {
            const int j = (k * G::NCT + ct) * kVec;
            reinterpret_cast<float4*>(wg + j)[0] = make_float4(acc_g[k][0], acc_g[k][1], acc_g[k][2], acc_g[k][3]);
            reinterpret_cast<float4*>(wg + j)[1] = make_float4(acc_g[k][4], acc_g[k][5], acc_g[k][6], acc_g[k][7]);
            reinterpret_cast<float4*>(wb + j)[0] = make_float4(acc_b[k][0], acc_b[k][1], acc_b[k][2], acc_b[k][3]);
            reinterpret_cast<float4*>(wb + j)[1] = make_float4(acc_b[k][4], acc_b[k][5], acc_b[k][6], acc_b[k][7]);
        }
    }
}

namespace {

template <int OP, int H>
cudaError_t launch_bulk_t(const BulkArgs& a, int grid, cudaStream_t st) {
    using G = BGeo<OP, H>;
    // Pick the register-sharing variant only when the launch allocation
    // covers the split (otherwise setmaxnreg.inc could wait forever).
    // Per process (the binary is the same on every device); a benign race
    // at worst repeats the query.  -1 unknown, 0 plain variant, 1 sharing.
    static int share_ok = -1;
    static bool attr_set[2] = {false, false};
    if (share_ok < 0) {
        cudaFuncAttributes fa;
        int ok = 0;
        if (cudaFuncGetAttributes(&fa, norm_bulk_kernel<OP, H, true>) == cudaSuccess) {
            const long pool = static_cast<long>(fa.numRegs) * G::THREADS;
            const long need = 128L * kProducerRegs + static_cast<long>(G::NCT) * G::CONS_REGS;
            // only worth it (and only well-formed) when consumers really gain registers
            ok = (fa.numRegs >= kProducerRegs && fa.numRegs < G::CONS_REGS && pool >= need) ? 1 : 0;
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
        norm_bulk_kernel<OP, H, true><<<grid, G::THREADS, G::SMEM, st>>>(a);
    } else {
        if (!attr_set[0]) {
            cudaError_t e = cudaFuncSetAttribute(norm_bulk_kernel<OP, H, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
            if (e != cudaSuccess) return e;
            attr_set[0] = true;
        }
        norm_bulk_kernel<OP, H, false><<<grid, G::THREADS, G::SMEM, st>>>(a);
    }
    return cudaGetLastError();
}

template <int OP>
cudaError_t launch_bulk_op(int64_t hidden, const BulkArgs& a, int grid, cudaStream_t st) {
    NF_HIDDEN_SWITCH(hidden, { return launch_bulk_t<OP, H>(a, grid, st); })
}

template <int OP>
bool shape_of(int64_t hidden, int* threads, int* stages, int* smem) {
    switch (hidden) {
#define NF_BULK_CASE(HV) \
        case HV: *threads = BGeo<OP, HV>::THREADS; *stages = BGeo<OP, HV>::S; *smem = BGeo<OP, HV>::SMEM; return true;
        NF_BULK_CASE(1024) NF_BULK_CASE(2048) NF_BULK_CASE(4096)
        NF_BULK_CASE(5120) NF_BULK_CASE(8192) NF_BULK_CASE(12288)
#undef NF_BULK_CASE
        default: return false;
    }
}

}  // namespace

bool bulk_shape(int op, int64_t hidden, int* threads, int* stages, int* smem_bytes) {
    switch (op) {
        case kFused: return shape_of<kFused>(hidden, threads, stages, smem_bytes);
        case kRms: return shape_of<kRms>(hidden, threads, stages, smem_bytes);
        case kLnFwd: return shape_of<kLnFwd>(hidden, threads, stages, smem_bytes);
        case kLnBwd: return shape_of<kLnBwd>(hidden, threads, stages, smem_bytes);
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

}  // namespace nf
