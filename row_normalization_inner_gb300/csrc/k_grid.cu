// Grid-resident inner normalization: a call's rows stay on chip across one
// grid-wide exchange of the row statistics.  The "Llu/ln bwd" discussion
// names grid-parallel inner normalization (a row over more CTAs than one
// block or cluster) as the missing variant; the split family does it with a
// launch per phase and reads every row twice.  When the rows of a call fit
// in the shared memory of one CTA per SM, this family reads them once:
//
//   CTA c (one per SM, all co-resident: cooperative launch) owns the column
//   slice [c * vc, (c + 1) * vc) of 8-element vectors of EVERY row.
//   Phase 1 copies its slice of every row into shared memory (per-thread
//   16-byte cp.async, one row ahead of the row being summed) and sums the
//   per-row partials as the rows land (RMS: sum x^2;
//   LayerNorm: sums of x - c and its square, c the row's first element;
//   backward: the two row sums of the gradient formula).  It writes them to
//   the workspace and arrives at a grid barrier (a bounded wait: if it runs
//   out the kernel records NF_ERR_TIMEOUT in the device status word and
//   returns).  Every CTA then adds the rows' partials in the same fixed
//   order (same bits everywhere) and phase 2 writes the outputs from shared
//   memory.
//
// A column's every row sits in one CTA, so the backward column sums
// (dgamma / dbeta, dw) are complete in that CTA and written directly from
// phase 2, in a fixed row order: deterministic without a column-reduction
// pass.  The backward keeps x on chip and reads dy a second time after the
// barrier, from L2 (a grid's rows fit there: the whole family holds at most
// the SMs' shared memory, about 34 MB).
//
// The fused op stores residual = bf16(x + residual) and normalizes that
// stored value (its statistics and its output both come from the bf16
// residual held on chip), the literal reading of the in-place statement
// "residual += x; x = norm(residual) * w" with bf16 storage.
#include "common.cuh"
#include "launch.h"
#include "pairs.cuh"
#include "pdl.cuh"

namespace nf {

// [kernel-span grid_norm] (with its barrier and copy helpers)
// Arrivals at the grid barrier on this device, over all launches.  Every CTA
// of a grid_norm launch adds 1 exactly once, and a launch occupies every SM
// (one CTA per SM, the whole register file), so two launches never arrive
// at the same time and the count is a multiple of the grid size between
// launches: a CTA's target is the next multiple of the grid size above its
// ticket.  No per-call reset is needed.
__device__ unsigned long long g_grid_arrivals;

namespace {

constexpr int kGrT = 512;                // threads per CTA (one CTA per SM)
constexpr int kGrWarps = kGrT / 32;
constexpr int kGrBatch = 8;              // second-tensor vectors a thread loads at once in phase 1

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// The arrival: an acquire-release add, so the CTA's writes (ordered before
// it by the CTA barrier) are published by it, and the last CTA to arrive
// sees every other CTA's writes through the chain of adds.
__device__ __forceinline__ unsigned long long atom_add_acq_rel(unsigned long long* p, unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}
__device__ __forceinline__ void gr_cp16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void gr_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's newest copy groups are pending.
template <int N>
__device__ __forceinline__ void gr_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Grid barrier, called by every thread of every CTA once its writes are
// done: thread 0 publishes the CTA's writes with its arrival (a ticket) and
// waits until the arrivals reach the next multiple of `grid` above it, or
// until `limit_ns` has passed; in the second case it records NF_ERR_TIMEOUT
// in the device status word.  The last CTA to arrive completes the count
// itself and does not wait.  Returns false in every thread of a CTA that
// gave up (it must then return without further work).  Only valid when all
// `grid` CTAs are resident (a cooperative launch).
__device__ __forceinline__ bool grid_barrier(unsigned long long* arrivals, unsigned long long grid,
                                             uint64_t limit_ns, int* status, int* give_up) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned long long ticket = atom_add_acq_rel(arrivals, 1ull);
        const unsigned long long target = (ticket / grid + 1) * grid;
        int fail = 0;
        if (ticket + 1 != target) {
            const uint64_t t0 = global_ns();
            while (ld_acquire_u64(arrivals) < target) {
                if (global_ns() - t0 > limit_ns) {
                    fail = 1;
                    break;
                }
            }
            __threadfence();
        }
        if (fail) record_status(status, kStatusTimeout);
        *give_up = fail;
    }
    __syncthreads();
    return !*give_up;
}

// Test kernel for the bounded wait above: the CTAs wait for one CTA more
// than the grid has (on a counter the launcher zeroes), so every wait runs
// out.
__global__ void grid_barrier_selftest(unsigned long long* arrivals, uint64_t limit_ns, int* status) {
    __shared__ int give_up;
    grid_barrier(arrivals, gridDim.x + 1ull, limit_ns, status, &give_up);
}

// OP: 0 fused add + RMSNorm, 1 RMSNorm, 2 LayerNorm forward, 3 LayerNorm
// backward (saved mean / rstd), 4 RMSNorm backward (ADD: + the fused-add
// residual-stream gradient a.add).  RM: the row bound the per-row sums are
// unrolled for (rows <= RM); U: vectors a thread handles at once per row in
// phase 2 (RM * U = 8).
template <int OP, int RM, int U, bool ADD>
__global__ void __launch_bounds__(kGrT, 1)
grid_norm(DynArgs a, float2* __restrict__ part, int vc, int* status) {
    extern __shared__ __align__(16) uint4 gr_rows[];  // [rows][vc]: this CTA's slice of every row
    __shared__ float red[kGrWarps * RM * 2];
    __shared__ float2 stat[RM];
    __shared__ int give_up;
    constexpr bool kBwd = OP >= 3;
    constexpr bool kTwo = OP == 0 || kBwd;  // phase 1 reads a second tensor (residual / dy)
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int R = static_cast<int>(a.rows), H = a.hidden, G = gridDim.x;
    const int NV = H / kVec;
    const int vbeg = blockIdx.x * vc;
    const int nv = NV - vbeg < vc ? (NV - vbeg > 0 ? NV - vbeg : 0) : vc;
    const float invH = 1.0f / static_cast<float>(H);
    const uint16_t* p0 = a.p0 + static_cast<int64_t>(vbeg) * kVec;

    // forward: warm L2 with this CTA's weights (read in phase 2), one
    // 128-byte line (8 vectors) per thread; a hint, so it may run before
    // the wait for the kernel ahead
    if constexpr (!kBwd) {
        for (int i = t * 8; i < nv; i += kGrT * 8) {
            prefetch_l2(p0 + static_cast<int64_t>(i) * kVec);
            if (OP == 2) prefetch_l2(a.p1 + static_cast<int64_t>(vbeg + i) * kVec);
        }
    }
    grid_dep_wait();

    // ---- phase 1: the slice of every row into shared memory, row by row ----
    // (the copies of row r + 1 go out while row r is summed; all rows at
    // once measured slower: the second tensor's loads queued behind them)
    {
        const uint16_t* src = a.in0 + static_cast<int64_t>(vbeg) * kVec;
        for (int i = t; i < nv; i += kGrT) gr_cp16(&gr_rows[i], src + static_cast<int64_t>(i) * kVec);
        gr_commit();
    }
    // per-row constants: LN forward: the shift (the row's first element);
    // LN backward: the saved mean and rstd
    float rc0[RM], rc1[RM], acc[RM][2];
#pragma unroll
    for (int r = 0; r < RM; ++r) {
        rc0[r] = rc1[r] = 0.f;
        acc[r][0] = acc[r][1] = 0.f;
        if (r < R) {
            if constexpr (OP == 2)
                rc0[r] = __uint_as_float(static_cast<uint32_t>(__ldg(a.in0 + static_cast<int64_t>(r) * H)) << 16);
            if constexpr (OP == 3) {
                rc0[r] = __ldg(a.mean + r);
                rc1[r] = __ldg(a.rstd + r);
            }
        }
    }
    // one batch of the second tensor (and the weight): `sb` holds row r's
    // vectors i0, i0 + kGrT, ... (kGrBatch of them), `wb` the weight's
    auto consume = [&](int r, int i0, const uint4 (&sb)[kGrBatch], const uint4 (&wb)[kGrBatch]) {
        const int64_t roff = static_cast<int64_t>(r) * H + static_cast<int64_t>(vbeg) * kVec;
#pragma unroll
        for (int k = 0; k < kGrBatch; ++k) {
            const int i = i0 + k * kGrT;
            if (i >= nv) break;
            float f[8];
            unpack8(gr_rows[r * vc + i], f);
            if constexpr (OP == 0) {
                float b[8];
                unpack8(sb[k], b);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] += b[e];
                const uint4 h = pack8(f);  // the stored residual, normalized in phase 2
                gr_rows[r * vc + i] = h;
                st_stream(a.out1 + roff + static_cast<int64_t>(i) * kVec, h);
                unpack8(h, f);
            }
            if constexpr (OP <= 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r][0] = fmaf(f[e], f[e], acc[r][0]);
            } else if constexpr (OP == 2) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float d = f[e] - rc0[r];
                    acc[r][0] += d;
                    acc[r][1] = fmaf(d, d, acc[r][1]);
                }
            } else {
                float dy[8], w[8];
                unpack8(sb[k], dy);
                unpack8(wb[k], w);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float g = dy[e] * w[e];
                    if constexpr (OP == 3) {
                        acc[r][0] += g;
                        acc[r][1] = fmaf(g, (f[e] - rc0[r]) * rc1[r], acc[r][1]);
                    } else {
                        acc[r][0] = fmaf(f[e], f[e], acc[r][0]);
                        acc[r][1] = fmaf(g, f[e], acc[r][1]);
                    }
                }
            }
        }
    };
    // the second tensor's batch of row r at vectors i0, i0 + kGrT, ...
    auto load_row = [&](int r, int i0, uint4 (&sb)[kGrBatch]) {
        const int64_t roff = static_cast<int64_t>(r) * H + static_cast<int64_t>(vbeg) * kVec;
#pragma unroll
        for (int k = 0; k < kGrBatch; ++k) {
            const int i = i0 + k * kGrT;
            if (i < nv) sb[k] = ld_stream(a.in1 + roff + static_cast<int64_t>(i) * kVec);
        }
    };
    auto load_w1 = [&](int i0, uint4 (&wb)[kGrBatch]) {
#pragma unroll
        for (int k = 0; k < kGrBatch; ++k) {
            const int i = i0 + k * kGrT;
            if (i < nv) wb[k] = ld_param(p0 + static_cast<int64_t>(i) * kVec);
        }
    };
    // The fused op, when a row is one batch per thread, loads row r + 1's
    // residual while row r is summed (two register buffers).  Longer rows,
    // and the backward (a second dy buffer, or the weight held across rows,
    // spills), take their batches one at a time.
    const bool one = OP == 0 && nv <= kGrBatch * kGrT;
    uint4 sbA[kGrBatch], sbB[kGrBatch];  // unused (and dropped) by the other ops
    if constexpr (OP == 0) {
        if (one) load_row(0, t, sbA);
    }
#pragma unroll
    for (int r = 0; r < RM; ++r) {
        if (r >= R) break;
        if (r + 1 < R) {
            const uint16_t* src = a.in0 + static_cast<int64_t>(r + 1) * H + static_cast<int64_t>(vbeg) * kVec;
            for (int i = t; i < nv; i += kGrT) gr_cp16(&gr_rows[(r + 1) * vc + i], src + static_cast<int64_t>(i) * kVec);
        }
        gr_commit();
        if constexpr (OP == 0) {
            if (one) {
                uint4 (&cur)[kGrBatch] = (r & 1) ? sbB : sbA;
                uint4 (&nxt)[kGrBatch] = (r & 1) ? sbA : sbB;
                if (r + 1 < R) load_row(r + 1, t, nxt);
                gr_wait<1>();  // this thread's copies of row r have landed (only row r + 1's may be pending)
                consume(r, t, cur, cur);  // (no weight in the fused op's first phase)
                continue;
            }
        }
        for (int i0 = t; i0 < nv; i0 += kGrBatch * kGrT) {
            uint4 sb[kGrBatch], wb[kGrBatch];
            if constexpr (kTwo) load_row(r, i0, sb);
            if constexpr (kBwd) load_w1(i0, wb);
            gr_wait<1>();  // this thread's copies of row r have landed (only row r + 1's may be pending)
            consume(r, i0, sb, wb);
        }
    }
    gr_wait<0>();  // nothing left in flight (the last row committed an empty group)
    // the CTA's partial of each row: lanes, then warps in order
#pragma unroll
    for (int r = 0; r < RM; ++r) {
        if (r < R) {
            warp_sum<2>(acc[r]);
            if (lane == 0) {
                red[(warp * RM + r) * 2] = acc[r][0];
                red[(warp * RM + r) * 2 + 1] = acc[r][1];
            }
        }
    }
    __syncthreads();
    if (t < R) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int w = 0; w < kGrWarps; ++w) {
            s0 += red[(w * RM + t) * 2];
            s1 += red[(w * RM + t) * 2 + 1];
        }
        part[static_cast<int64_t>(t) * G + blockIdx.x] = make_float2(s0, s1);
    }

    // phase 2's first weights go out before the barrier (inputs only); each
    // iteration then loads the next one's before computing its own
    uint4 wn[U], bn[OP == 2 ? U : 1];
    auto load_w = [&](int i0n) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0n + u * kGrT + t;
            if (i < nv) {
                wn[u] = ld_param(p0 + static_cast<int64_t>(i) * kVec);
                if constexpr (OP == 2) bn[u] = ld_param(a.p1 + static_cast<int64_t>(vbeg + i) * kVec);
            }
        }
    };
    load_w(0);

    // ---- grid barrier (every CTA is resident: cooperative launch) ----
    if (!grid_barrier(&g_grid_arrivals, static_cast<unsigned long long>(G), kWaitLimitNs, status, &give_up))
        return;

    // ---- every CTA adds the partials of every row in the same order ----
    if (warp < R) {
        float q[2] = {0.f, 0.f};
        for (int c = lane; c < G; c += 32) {
            const float2 p = __ldcg(part + static_cast<int64_t>(warp) * G + c);
            q[0] += p.x;
            q[1] += p.y;
        }
        warp_sum<2>(q);
        if (lane == 0) {
            const int r = warp;
            if constexpr (OP <= 1) {
                stat[r] = make_float2(0.f, rsqrtf(q[0] * invH + a.eps));
            } else if constexpr (OP == 2) {
                // the shift read before the barrier (x may be y, already being overwritten)
                float c = 0.f;
#pragma unroll
                for (int q2 = 0; q2 < RM; ++q2)
                    if (q2 == r) c = rc0[q2];
                const float dm = q[0] * invH;
                const float mean = c + dm;
                const float rstd = rsqrtf(fmaxf(q[1] * invH - dm * dm, 0.f) + a.eps);
                stat[r] = make_float2(mean, rstd);
                if (blockIdx.x == 0) {
                    if (a.mean) a.mean[r] = mean;
                    if (a.rstd) a.rstd[r] = rstd;
                }
            } else if constexpr (OP == 3) {
                stat[r] = make_float2(q[0] * invH, q[1] * invH);  // (A, B)
            } else {
                const float rs = rsqrtf(q[0] * invH + a.eps);
                stat[r] = make_float2(rs, rs * rs * rs * q[1] * invH);
            }
        }
    }
    __syncthreads();
    float2 st[RM];
#pragma unroll
    for (int r = 0; r < RM; ++r) st[r] = r < R ? stat[r] : make_float2(0.f, 0.f);

    // ---- phase 2: the outputs from the slice held on chip ----
    for (int i0 = 0; i0 < nv; i0 += U * kGrT) {
        uint4 wc[U], bc[OP == 2 ? U : 1];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            wc[u] = wn[u];
            if constexpr (OP == 2) bc[u] = bn[u];
        }
        if (i0 + U * kGrT < nv) load_w(i0 + U * kGrT);
        uint4 dyv[kBwd ? U : 1][kBwd ? RM : 1], adv[ADD ? U : 1][ADD ? RM : 1];
        if constexpr (kBwd) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = i0 + u * kGrT + t;
#pragma unroll
                for (int r = 0; r < RM; ++r) {
                    if (r < R && i < nv) {
                        const int64_t off = static_cast<int64_t>(r) * H + static_cast<int64_t>(vbeg + i) * kVec;
                        dyv[u][r] = ld_stream(a.in1 + off);
                        if constexpr (ADD) adv[u][r] = ld_stream(a.add + off);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * kGrT + t;
            if (i >= nv) continue;
            const int64_t vo = static_cast<int64_t>(vbeg + i) * kVec;
            float w[8], b[8], c0[8], c1[8];
            unpack8(wc[u], w);
            if constexpr (OP == 2) unpack8(bc[u], b);
#pragma unroll
            for (int e = 0; e < 8; ++e) c0[e] = c1[e] = 0.f;
#pragma unroll
            for (int r = 0; r < RM; ++r) {
                if (r >= R) continue;
                float f[8], o[8];
                unpack8(gr_rows[r * vc + i], f);
                if constexpr (OP <= 1) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = f[e] * st[r].y * w[e];
                } else if constexpr (OP == 2) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = fmaf(f[e] - st[r].x, st[r].y * w[e], b[e]);
                } else {
                    float dy[8];
                    unpack8(dyv[u][r], dy);
                    if constexpr (OP == 3) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float xh = (f[e] - rc0[r]) * rc1[r];
                            o[e] = rc1[r] * (dy[e] * w[e] - st[r].x - xh * st[r].y);
                            c0[e] = fmaf(dy[e], xh, c0[e]);
                            c1[e] += dy[e];
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            o[e] = st[r].x * dy[e] * w[e] - f[e] * st[r].y;
                            c0[e] = fmaf(dy[e] * f[e], st[r].x, c0[e]);
                        }
                        if constexpr (ADD) {
                            float d[8];
                            unpack8(adv[u][r], d);
#pragma unroll
                            for (int e = 0; e < 8; ++e) o[e] += d[e];
                        }
                    }
                }
                st_stream(a.out0 + static_cast<int64_t>(r) * H + vo, pack8(o));
            }
            if constexpr (kBwd) {  // every row of these columns is here: the column sums are final
                float4* q0 = reinterpret_cast<float4*>(a.cols0 + vo);
                q0[0] = make_float4(c0[0], c0[1], c0[2], c0[3]);
                q0[1] = make_float4(c0[4], c0[5], c0[6], c0[7]);
                if constexpr (OP == 3) {
                    float4* q1 = reinterpret_cast<float4*>(a.cols1 + vo);
                    q1[0] = make_float4(c1[0], c1[1], c1[2], c1[3]);
                    q1[1] = make_float4(c1[4], c1[5], c1[6], c1[7]);
                }
            }
        }
    }
}

// [end kernel-span grid_norm]

// Static shared memory of grid_norm (the reduction scratch, bounded by the
// largest RM), left out of the dynamic budget below.
constexpr int kGrStaticSmem = kGrWarps * kGridMaxRows * 2 * 4 + kGridMaxRows * 8 + 16;
constexpr int kGrDynMax = 227 * 1024 - kGrStaticSmem;
// Every launch asks for at least this much dynamic shared memory, more than
// half an SM's 228 KB, so no two grid_norm CTAs ever share an SM whatever
// their register count: a launch holds every SM, as the arrival count needs.
constexpr int kGrExclusiveSmem = 116 * 1024;

// One cooperative launch of grid_norm<OP, RM, U, ADD>, a programmatic
// dependent of the work ahead in the stream.
template <int OP, int RM, int U, bool ADD>
cudaError_t launch_coop(int sms, size_t smem, cudaStream_t st, const DynArgs& a, float2* part, int vc,
                        int* status) {
    auto kernel = grid_norm<OP, RM, U, ADD>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGrDynMax))
            return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kGrT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, a, part, vc, status);
}

template <int OP, bool ADD = false>
cudaError_t launch_op(const DynArgs& a, float2* part, int vc, int sms, size_t smem, int* status,
                      cudaStream_t st) {
    if (a.rows <= 2) return launch_coop<OP, 2, 4, ADD>(sms, smem, st, a, part, vc, status);
    if (a.rows <= 4) return launch_coop<OP, 4, 2, ADD>(sms, smem, st, a, part, vc, status);
    return launch_coop<OP, 8, 1, ADD>(sms, smem, st, a, part, vc, status);
}

// ---- outer normalization with the matrix on chip, in column bands ----------
// Per-column statistics over the rows, one read of x.  One cooperative launch
// of one CTA per SM; CTA c owns the row stripe [r0, r0 + n) (rows / SMs,
// the first rows % SMs stripes one row longer).  The columns are walked in
// bands of `bvec` 16-byte vectors (bvec * 8 columns); each band of the
// stripe is copied into one of two shared-memory buffers (row pitch bvec + 1
// vectors, so reads down a column hit distinct banks) two bands ahead.  Per
// band:
//   statistics: thread t takes vector t / tpv of the band (tpv = 512 / bvec
//     threads per vector) and rows t % tpv, t % tpv + tpv, ...; shifted sums
//     per column (shift = its first value) give (count, mean, M2), merged
//     across the tpv lanes with Chan's pairwise formula in a fixed tree; the
//     CTA's partial per column goes to the workspace, then the CTA arrives
//     at the first grid barrier;
//   merge (after the first barrier): one warp per column over all warps of
//     the grid (lanes take CTAs lane, lane + 32, ..., then a fixed shuffle
//     tree) into mean, rstd and the affine pair a = rstd * gamma,
//     b = beta - mean * a; second grid barrier;
//   apply: every CTA reads the band's (a, b) and writes y = x * a + b from
//     shared memory, in coalesced row segments.
// The loop computes band k + 1's statistics and arrives before it applies
// band k, so band k's stores drain while the grid gathers at the barrier.
// Partials and pairs alternate between two workspace slots by band parity.

constexpr int kOgMaxGrid = 256;  // CTAs (SMs) the column merge handles

struct OuterGridArgs {
    uint16_t* y;
    const uint16_t* x;
    const uint16_t* gamma;
    const uint16_t* beta;
    float* mean;        // per-column outputs, may be null
    float* rstd;
    float2* part;       // [2][SMs][bvec * 8]: the CTAs' (mean, M2) of a band
    float2* ab;         // [2][bvec * 8]: a band's (a, b)
    int64_t rows;
    int hidden;
    float eps;
    int bvec;           // vectors per band (a power of two, 16 .. 512)
};

__device__ __forceinline__ void chan2(float& n, float& m, float& q, float nb, float mb, float qb) {
    if (nb == 0.f) return;
    if (n == 0.f) {
        n = nb;
        m = mb;
        q = qb;
        return;
    }
    const float nn = n + nb;
    const float d = mb - m;
    const float wb = nb / nn;
    m += d * wb;
    q += qb + d * d * n * wb;
    n = nn;
}

// The grid barrier in two halves: every thread calls grid_arrive once its
// writes are done (thread 0 publishes them and takes the ticket); later
// every thread calls grid_wait, which returns false in every thread of a
// CTA whose bounded wait ran out.  A CTA arrives at its next barrier only
// after its wait on this one, so the arrival count still steps by whole
// grids.
__device__ __forceinline__ void grid_arrive(unsigned long long* arrivals, unsigned long long grid,
                                            unsigned long long* target) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned long long ticket = atom_add_acq_rel(arrivals, 1ull);
        const unsigned long long tg = (ticket / grid + 1) * grid;
        *target = ticket + 1 == tg ? 0ull : tg;  // 0: this CTA completed the count
    }
}
__device__ __forceinline__ bool grid_wait(unsigned long long* arrivals, const unsigned long long* target,
                                          uint64_t limit_ns, int* status, int* give_up) {
    if (threadIdx.x == 0) {
        int fail = 0;
        if (*target != 0ull) {
            const uint64_t t0 = global_ns();
            while (ld_acquire_u64(arrivals) < *target) {
                if (global_ns() - t0 > limit_ns) {
                    fail = 1;
                    break;
                }
            }
            __threadfence();
        }
        if (fail) record_status(status, kStatusTimeout);
        *give_up = fail;
    }
    __syncthreads();
    return !*give_up;
}

__global__ void __launch_bounds__(kGrT, 1) outer_grid_fwd(OuterGridArgs g, int* status) {
    extern __shared__ __align__(16) uint4 ob[];  // [2][stripe rows][bvec + 1], then (a, b) of a band
    __shared__ int give_up;
    __shared__ unsigned long long target;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int G = gridDim.x, c = blockIdx.x, H = g.hidden, NV = H / kVec;
    const int bvec = g.bvec, pitch = bvec + 1, tpv = kGrT / bvec;
    const int64_t base = g.rows / G;
    const int rem = static_cast<int>(g.rows % G);
    const int64_t r0 = c * base + (c < rem ? c : rem);
    const int n = static_cast<int>(base + (c < rem ? 1 : 0));
    const int rs = static_cast<int>(base + (rem ? 1 : 0));   // the longest stripe: buffer rows
    uint4* const buf0 = ob;
    uint4* const buf1 = ob + static_cast<int64_t>(rs) * pitch;
    auto bufk = [&](int k) { return (k & 1) ? buf1 : buf0; };
    float2* sab = reinterpret_cast<float2*>(ob + 2 * static_cast<int64_t>(rs) * pitch);
    const int nb = (NV + bvec - 1) / bvec;                    // bands
    const int BC = bvec * kVec;                               // columns per band
    unsigned long long* arrivals = &g_grid_arrivals;
    const unsigned long long grid = static_cast<unsigned long long>(G);
    auto nvec = [&](int k) { return NV - k * bvec < bvec ? NV - k * bvec : bvec; };  // vectors of band k

    // copy band k of the stripe into its buffer (thread t: vector t % bvec,
    // rows t / bvec + (kGrT / bvec) * m: coalesced row segments)
    auto issue = [&](int k) {
        if (k < nb) {
            const int vb = k * bvec, v = t % bvec;
            if (vb + v < NV) {
                uint4* dst = bufk(k);
                const uint16_t* src = g.x + r0 * H + static_cast<int64_t>(vb + v) * kVec;
                for (int i = t / bvec; i < n; i += tpv) gr_cp16(&dst[i * pitch + v], src + static_cast<int64_t>(i) * H);
            }
        }
        gr_commit();
    };
    // the CTA's statistics of each column of band k -> its partial slot
    auto stats = [&](int k) {
        const uint4* buf = bufk(k);
        const int nvb = nvec(k);
        const int v = t / tpv, ro = t % tpv;
        float cn = 0.f, cm[8], cq[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) cm[e] = cq[e] = 0.f;
        if (v < nvb && ro < n) {
            float sh[8], s1[8], s2[8];
            unpack8(buf[ro * pitch + v], sh);
#pragma unroll
            for (int e = 0; e < 8; ++e) s1[e] = s2[e] = 0.f;
            int cnt = 0;
#pragma unroll 4
            for (int i = ro; i < n; i += tpv, ++cnt) {
                float f[8];
                unpack8(buf[i * pitch + v], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float d = f[e] - sh[e];
                    s1[e] += d;
                    s2[e] = fmaf(d, d, s2[e]);
                }
            }
            cn = static_cast<float>(cnt);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float dm = s1[e] / cn;
                cm[e] = sh[e] + dm;
                cq[e] = fmaxf(s2[e] - s1[e] * dm, 0.f);
            }
        }
        // the tpv lanes of the vector, in a fixed tree (lane ro takes ro + off)
        for (int off = tpv >> 1; off > 0; off >>= 1) {
            const float on = __shfl_down_sync(0xFFFFFFFFu, cn, off);
            float om[8], oq[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                om[e] = __shfl_down_sync(0xFFFFFFFFu, cm[e], off);
                oq[e] = __shfl_down_sync(0xFFFFFFFFu, cq[e], off);
            }
            if (ro < off) {
                float nn = cn;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    nn = cn;
                    chan2(nn, cm[e], cq[e], on, om[e], oq[e]);
                }
                cn = nn;
            }
        }
        if (ro == 0 && v < nvb) {
            float4* q = reinterpret_cast<float4*>(g.part + (static_cast<int64_t>(k & 1) * G + c) * BC + v * kVec);
#pragma unroll
            for (int e = 0; e < 8; e += 2) q[e / 2] = make_float4(cm[e], cq[e], cm[e + 1], cq[e + 1]);
        }
    };
    // band k's columns merged across the CTAs, one warp per column over the grid
    auto merge = [&](int k) {
        const float2* part = g.part + static_cast<int64_t>(k & 1) * G * BC;
        float2* ab = g.ab + static_cast<int64_t>(k & 1) * BC;
        for (int j = c * kGrWarps + warp; j < nvec(k) * kVec; j += G * kGrWarps) {
            const int col = k * BC + j;
            const float ga = __uint_as_float(static_cast<uint32_t>(__ldg(g.gamma + col)) << 16);
            const float be = __uint_as_float(static_cast<uint32_t>(__ldg(g.beta + col)) << 16);
            float2 p[kOgMaxGrid / 32];  // every load in flight before the first merge
#pragma unroll
            for (int q = 0; q < kOgMaxGrid / 32; ++q) {
                const int s = lane + 32 * q;
                if (s < G) p[q] = __ldcg(part + static_cast<int64_t>(s) * BC + j);
            }
            float cn = 0.f, cm = 0.f, cq = 0.f;
#pragma unroll
            for (int q = 0; q < kOgMaxGrid / 32; ++q) {
                const int s = lane + 32 * q;
                if (s < G) chan2(cn, cm, cq, static_cast<float>(base + (s < rem ? 1 : 0)), p[q].x, p[q].y);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float on = __shfl_down_sync(0xFFFFFFFFu, cn, off);
                const float om = __shfl_down_sync(0xFFFFFFFFu, cm, off);
                const float oq = __shfl_down_sync(0xFFFFFFFFu, cq, off);
                if (lane < off) chan2(cn, cm, cq, on, om, oq);
            }
            if (lane == 0) {
                const float rstd = rsqrtf(cq / static_cast<float>(g.rows) + g.eps);
                const float aa = rstd * ga;
                ab[j] = make_float2(aa, be - cm * aa);
                if (g.mean) g.mean[col] = cm;
                if (g.rstd) g.rstd[col] = rstd;
            }
        }
    };
    // y = x * a + b for band k, from shared memory
    auto apply = [&](int k) {
        const uint4* buf = bufk(k);
        const int nvb = nvec(k);
        const float2* ab = g.ab + static_cast<int64_t>(k & 1) * BC;
        for (int j = t; j < nvb * kVec; j += kGrT) sab[j] = __ldcg(ab + j);
        __syncthreads();
        const int v = t % bvec;
        if (v < nvb) {
            float2 a2[4], b2[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 u0 = sab[v * kVec + 2 * q], u1 = sab[v * kVec + 2 * q + 1];
                a2[q] = make_float2(u0.x, u1.x);
                b2[q] = make_float2(u0.y, u1.y);
            }
            uint16_t* dst = g.y + r0 * H + static_cast<int64_t>(k * bvec + v) * kVec;
            for (int i = t / bvec; i < n; i += tpv) {
                float2 f[4], o[4];
                unpack8x2(buf[i * pitch + v], f);
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = __ffma2_rn(f[q], a2[q], b2[q]);
                st_stream(dst + static_cast<int64_t>(i) * H, pack8x2(o));
            }
        }
        __syncthreads();  // the buffer and the staged pairs are free again
    };

    grid_dep_wait();
    issue(0);
    issue(1);
    gr_wait<1>();
    __syncthreads();  // band 0 has landed
    stats(0);
    // a CTA that gives up waits for its own copies in flight, then returns
    grid_arrive(arrivals, grid, &target);
    if (!grid_wait(arrivals, &target, kWaitLimitNs, status, &give_up)) {
        gr_wait<0>();
        return;
    }
    merge(0);
    grid_arrive(arrivals, grid, &target);
    if (!grid_wait(arrivals, &target, kWaitLimitNs, status, &give_up)) {
        gr_wait<0>();
        return;
    }
    for (int k = 0; k < nb; ++k) {
        const bool next = k + 1 < nb;
        if (next) {
            gr_wait<0>();
            __syncthreads();  // band k + 1 has landed
            stats(k + 1);
            grid_arrive(arrivals, grid, &target);
        }
        apply(k);  // its stores drain while the grid gathers
        issue(k + 2);
        if (next) {
            if (!grid_wait(arrivals, &target, kWaitLimitNs, status, &give_up)) {
                gr_wait<0>();
                return;
            }
            merge(k + 1);
            grid_arrive(arrivals, grid, &target);
            if (!grid_wait(arrivals, &target, kWaitLimitNs, status, &give_up)) {
                gr_wait<0>();
                return;
            }
        }
    }
    gr_wait<0>();
}

size_t gr_align16(size_t b) { return (b + 15) / 16 * 16; }

}  // namespace

bool grid_shape(int op, int64_t rows, int64_t hidden, int sms, int* vc, size_t* smem) {
    (void)op;
    if (rows < 1 || rows > kGridMaxRows || sms < 1) return false;
    if (hidden < kVec || hidden % kVec != 0 || hidden > kSplitMaxHidden) return false;
    const int64_t nv = hidden / kVec;
    const int64_t per = (nv + sms - 1) / sms;
    const int64_t bytes = rows * per * 16;
    if (bytes > kGrDynMax) return false;
    if (vc) *vc = static_cast<int>(per);
    if (smem) *smem = static_cast<size_t>(bytes < kGrExclusiveSmem ? kGrExclusiveSmem : bytes);
    return true;
}

// Workspace: the row partials, rows x sms float2.
size_t grid_workspace_bytes(int op, int64_t rows, int64_t hidden, int sms) {
    if (!grid_shape(op, rows, hidden, sms, nullptr, nullptr)) return 0;
    return gr_align16(static_cast<size_t>(rows) * sms * sizeof(float2));
}

cudaError_t launch_grid_selftest(void* counter16, uint64_t limit_ns, int* status, cudaStream_t st) {
    unsigned long long* arrivals = static_cast<unsigned long long*>(counter16);
    if (cudaError_t e = cudaMemsetAsync(arrivals, 0, 16, st)) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, grid_barrier_selftest, arrivals, limit_ns, status);
}

// Outer normalization on chip: the widest band (a power of two from 16 to
// 512 vectors, no wider than the matrix needs) whose two stripe buffers and
// pairs fit one CTA's shared memory.
bool outer_grid_shape(int64_t rows, int64_t hidden, int sms, int* bvec, size_t* smem) {
    if (rows < 1 || sms < 1 || sms > kOgMaxGrid || hidden < kVec || hidden % kVec != 0) return false;
    const int64_t rs = (rows + sms - 1) / sms;
    const int64_t nv = hidden / kVec;
    int cap = 512;
    while (cap > 16 && cap / 2 >= nv) cap /= 2;
    for (int b = cap; b >= 16; b /= 2) {
        const int64_t bytes = 2 * rs * (b + 1) * 16 + static_cast<int64_t>(b) * kVec * 8;
        if (bytes <= kGrDynMax) {
            if (bvec) *bvec = b;
            if (smem) *smem = static_cast<size_t>(bytes < kGrExclusiveSmem ? kGrExclusiveSmem : bytes);
            return true;
        }
    }
    return false;
}

// Workspace: the CTAs' partials of a band [2][sms][bvec * 8] float2, then
// a band's (a, b) pairs [2][bvec * 8] float2 (two slots, by band parity).
size_t outer_grid_workspace_bytes(int64_t rows, int64_t hidden, int sms) {
    int bvec;
    if (!outer_grid_shape(rows, hidden, sms, &bvec, nullptr)) return 0;
    return 2 * static_cast<size_t>(sms + 1) * bvec * kVec * sizeof(float2);
}

cudaError_t launch_outer_grid_fwd(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                                  const void* beta, int64_t rows, int64_t hidden, float eps,
                                  void* workspace, int sms, int* status, cudaStream_t st) {
    int bvec;
    size_t smem;
    if (!outer_grid_shape(rows, hidden, sms, &bvec, &smem)) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaError_t e = cudaFuncSetAttribute(outer_grid_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kGrDynMax))
            return e;
        attr_set = true;
    }
    OuterGridArgs g{};
    g.y = static_cast<uint16_t*>(y);
    g.x = static_cast<const uint16_t*>(x);
    g.gamma = static_cast<const uint16_t*>(gamma);
    g.beta = static_cast<const uint16_t*>(beta);
    g.mean = mean;
    g.rstd = rstd;
    g.part = static_cast<float2*>(workspace);
    g.ab = g.part + 2 * static_cast<int64_t>(sms) * bvec * kVec;
    g.rows = rows;
    g.hidden = static_cast<int>(hidden);
    g.eps = eps;
    g.bvec = bvec;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kGrT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, outer_grid_fwd, g, status);
}

// a.cols0 / a.cols1 are the backward column outputs (dgamma / dbeta, dw).
cudaError_t launch_grid(int op, const DynArgs& a, void* workspace, int sms, int* status, cudaStream_t st) {
    int vc;
    size_t smem;
    if (!grid_shape(op, a.rows, a.hidden, sms, &vc, &smem)) return cudaErrorInvalidValue;
    float2* part = static_cast<float2*>(workspace);
    switch (op) {
        case 0: return launch_op<0>(a, part, vc, sms, smem, status, st);
        case 1: return launch_op<1>(a, part, vc, sms, smem, status, st);
        case 2: return launch_op<2>(a, part, vc, sms, smem, status, st);
        case 3: return launch_op<3>(a, part, vc, sms, smem, status, st);
        case 4:
            return a.add ? launch_op<4, true>(a, part, vc, sms, smem, status, st)
                         : launch_op<4, false>(a, part, vc, sms, smem, status, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nf
