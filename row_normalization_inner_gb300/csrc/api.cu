// C ABI of libnf.so: argument validation, planning and dispatch.
//
// Every entry point validates all arguments before it touches the GPU,
// chooses a plan with nf_plan_compute (pure host code) and launches on the
// caller's stream.  The scheduler lessons of "TMA inner persistent
// scheduler" (NVIDIA/Fuser PR #5587, reviewer guide: a missing null check,
// an unchecked cast, a possible divide by zero) apply here as: check every
// pointer, never divide by a derived count that could be zero, and return a
// status instead of crashing.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/nf.h"
#include "common.cuh"
#include "internal.h"
#include "launch.h"
#include "pdl.cuh"

namespace nf {

// The device status word: kernels that give up on a bounded wait record
// their error code here (first one wins).
__device__ int g_device_status = 0;

bool reg_shape(int64_t hidden, int* tpr, int* rpc) {
    switch (hidden) {
        case 1024:  *tpr = RegShape<1024>::TPR;  *rpc = RegShape<1024>::RPC;  return true;
        case 2048:  *tpr = RegShape<2048>::TPR;  *rpc = RegShape<2048>::RPC;  return true;
        case 4096:  *tpr = RegShape<4096>::TPR;  *rpc = RegShape<4096>::RPC;  return true;
        case 5120:  *tpr = RegShape<5120>::TPR;  *rpc = RegShape<5120>::RPC;  return true;
        case 8192:  *tpr = RegShape<8192>::TPR;  *rpc = RegShape<8192>::RPC;  return true;
        case 12288: *tpr = RegShape<12288>::TPR; *rpc = RegShape<12288>::RPC; return true;
        default: return false;
    }
}

namespace {

// Resident stage-1 CTAs per SM for the LayerNorm backward register path.
// The stage-1 grid is SMs x this, so the row-to-partial assignment (and
// therefore the bit pattern of dgamma/dbeta) depends only on the device.
int bwd_ctas_per_sm(int64_t hidden) {
    // The stage-1 kernels keep gamma, the row and 2 x 32 column
    // accumulators per thread in registers (~170-185 registers), so one
    // CTA fits per SM at every compiled size.
    (void)hidden;
    return 1;
}

// The library's own path choice, from the per-path timings on GB300 (CUDA
// graphs of back-to-back launches over L2-cold inputs, every op x size x
// path):
//  - forward ops: the register path is fastest at every row count, from 1
//    row (1.4-2.3 us per launch, where a cluster split only adds its
//    barrier latency: 2.8-3.1 us) to 65536 rows (1.0x the measured copy
//    bandwidth; LayerNorm 16384 x 8192: 0.98 against 0.88 for the bulk
//    ring); the exception is hidden 12288 RMSNorm / LayerNorm forward from
//    1024 rows, where the bulk ring keeps more bytes in flight than the
//    register-resident rows can (LayerNorm 16384 x 12288: 0.96 against 0.72);
//  - backward ops: the bulk path (its row groups fold their column partials
//    inside the CTA, so stage 2 stays small), except the RMSNorm backward
//    (and with it the fused-add backward) at hidden 5120 and 12288 from 1024
//    rows, where the runtime-hidden kernels with their per-thread copy ring
//    were faster (fused-add 16384 x 12288: 238 against 310 us, RMSNorm 194
//    against 228 us; 5120: 104 / 82 against 111 / 89 us; at 8192 and below,
//    and for every LayerNorm size, the bulk and row-block kernels won).
nf_path auto_path(nf_op op, int64_t rows, int64_t hidden, int rpc, int sms) {
    (void)rpc;
    (void)sms;
    const bool fwd = op == NF_OP_FUSED_ADD_RMSNORM || op == NF_OP_RMSNORM_FWD ||
                     op == NF_OP_LAYERNORM_FWD;
    if (!fwd) {
        if (op == NF_OP_RMSNORM_BWD && rows >= 1024 && (hidden == 5120 || hidden == 12288))
            return NF_PATH_DYNAMIC;
        return NF_PATH_BULK;
    }
    if (hidden >= 12288 && rows >= 1024 &&
        (op == NF_OP_RMSNORM_FWD || op == NF_OP_LAYERNORM_FWD))
        return NF_PATH_BULK;
    return NF_PATH_REG;
}

// Column-partial planes a backward op keeps per slot (LayerNorm: dgamma and
// dbeta; RMSNorm: dw).
int bwd_planes(nf_op op) { return op == NF_OP_LAYERNORM_BWD ? 2 : 1; }

std::atomic<int> g_forced_path{NF_PATH_AUTO};

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int*> g_status_addr[kMaxDevices];

nf_status current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return NF_ERR_CUDA;
    if (*dev < 0 || *dev >= kMaxDevices) return NF_ERR_CUDA;
    return NF_OK;
}

nf_status device_sm_count(int* sms) {
    int dev;
    if (nf_status st = current_device(&dev)) return st;
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            return NF_ERR_CUDA;
        g_sm_count[dev].store(v, std::memory_order_relaxed);
    }
    *sms = v;
    return NF_OK;
}

nf_status device_status_addr(int** addr) {
    int dev;
    if (nf_status st = current_device(&dev)) return st;
    int* p = g_status_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        void* q = nullptr;
        if (cudaGetSymbolAddress(&q, g_device_status) != cudaSuccess || !q) return NF_ERR_CUDA;
        p = static_cast<int*>(q);
        g_status_addr[dev].store(p, std::memory_order_release);
    }
    *addr = p;
    return NF_OK;
}

// A size with kernels specialized at compile time.
bool hidden_ok(int64_t h) {
    int a, b;
    return reg_shape(h, &a, &b);
}

// A size some kernel of `op` handles (compiled, the runtime-hidden path, or
// the grid-parallel cluster path for long rows).
bool split_ok(int64_t h) { return h >= kVec && h % kVec == 0 && h <= kSplitMaxHidden; }

bool hidden_supported(nf_op op, int64_t h) {
    int t, c, sl;
    return hidden_ok(h) || dyn_shape(op, h, &t) || long_shape(op, h, &c, &t, &sl) || split_ok(h);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Span {
    const void* p;
    int64_t bytes;
};

bool overlap(Span a, Span b) {
    if (!a.p || !b.p || a.bytes <= 0 || b.bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + static_cast<uintptr_t>(b.bytes) && b0 < a0 + static_cast<uintptr_t>(a.bytes);
}

// Overlap allowed only as the exact same buffer.
bool bad_overlap_except_alias(Span out, Span in) {
    if (out.p == in.p && out.bytes == in.bytes) return false;
    return overlap(out, in);
}

nf_status common_checks(nf_op op, int64_t rows, int64_t hidden, float eps, bool check_eps) {
    if (!hidden_supported(op, hidden)) return NF_ERR_UNSUPPORTED_HIDDEN;
    if (rows < 0) return NF_ERR_INVALID_ARG;
    // keep rows * hidden * 4 bytes representable
    if (rows > (INT64_MAX / 8) / hidden) return NF_ERR_INVALID_ARG;
    if (check_eps && !(std::isfinite(eps) && eps > 0.f)) return NF_ERR_INVALID_ARG;
    return NF_OK;
}

nf_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NF_OK : NF_ERR_CUDA; }

// The split and grid families: the launch of a planned call.
nf_status launch_split_family(const nf_plan& pl, nf_op op, const DynArgs& a, void* workspace,
                              cudaStream_t s) {
    int sms;
    if (nf_status st = device_sm_count(&sms)) return st;
    if (pl.path == NF_PATH_GRID) {
        int* status;
        if (nf_status st = device_status_addr(&status)) return st;
        return from_cuda(launch_grid(op, a, workspace, sms, status, s));
    }
    return from_cuda(launch_split(op, a, workspace, sms, s));
}

nf_status plan_for_call(nf_op op, int64_t rows, int64_t hidden, nf_plan* plan) {
    int sms;
    if (nf_status st = device_sm_count(&sms)) return st;
    return nf_plan_compute(op, rows, hidden, sms,
                           static_cast<nf_path>(g_forced_path.load(std::memory_order_relaxed)), plan);
}

// The plan of a forward call.  Without a workspace, an automatic split (or grid) plan
// falls back to the cluster family where that holds the row, so the plain
// forward entry points keep working up to the cluster limit.
nf_status plan_for_fwd(nf_op op, int64_t rows, int64_t hidden, bool have_ws, nf_plan* plan) {
    if (nf_status st = plan_for_call(op, rows, hidden, plan)) return st;
    if (have_ws || (plan->path != NF_PATH_SPLIT && plan->path != NF_PATH_GRID) ||
        g_forced_path.load(std::memory_order_relaxed) != NF_PATH_AUTO)
        return NF_OK;
    int sms;
    if (nf_status st = device_sm_count(&sms)) return st;
    nf_plan alt;
    if (nf_plan_compute(op, rows, hidden, sms, NF_PATH_CLUSTER, &alt) == NF_OK) *plan = alt;
    return NF_OK;
}

// Workspace bytes for `op` enough for every kernel family, so a later
// nf_set_path cannot make a previously sized workspace too small.
size_t any_path_workspace_bytes(nf_op op, int64_t rows, int64_t hidden) {
    if (!hidden_supported(op, hidden) || rows <= 0) return 0;
    int sms;
    if (device_sm_count(&sms) != NF_OK) return 0;
    size_t most = 0;
    for (nf_path p : {NF_PATH_REG, NF_PATH_BULK, NF_PATH_DYNAMIC, NF_PATH_CLUSTER, NF_PATH_SPLIT, NF_PATH_GRID}) {
        nf_plan pl;
        if (nf_plan_compute(op, rows, hidden, sms, p, &pl) != NF_OK) continue;
        const size_t b = plan_workspace_bytes(op, rows, hidden, sms, pl.path, pl.partials);
        if (b > most) most = b;
    }
    return most;
}

size_t bwd_workspace_bytes(nf_op op, int64_t rows, int64_t hidden) {
    return any_path_workspace_bytes(op, rows, hidden);
}

// The workspace a call needs under its plan, with the usual checks:
// NF_ERR_WORKSPACE_TOO_SMALL when it is short (or missing), NF_ERR_MISALIGNED
// when it is not 16-byte aligned.  *need = 0 for plans that use none.
nf_status check_workspace(nf_op op, int64_t rows, int64_t hidden, const nf_plan& pl,
                          const void* workspace, size_t workspace_bytes, size_t* need) {
    int sms;
    if (nf_status st = device_sm_count(&sms)) return st;
    *need = plan_workspace_bytes(op, rows, hidden, sms, pl.path, pl.partials);
    if (*need == 0) return NF_OK;
    if (!workspace || workspace_bytes < *need) return NF_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 16)) return NF_ERR_MISALIGNED;
    return NF_OK;
}

// The selftest kernel: one thread waits on a barrier nothing will complete.
__global__ void wait_selftest_kernel(int* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait(&bar, 0, timeout_ns)) record_status(status, kStatusTimeout);
    }
}

// Launch-floor probes (nf_selftest_floor): an empty dependent launch, and a
// plain copy of 16-byte vectors, 4 per thread, launched the same way as the
// operations' kernels.
__global__ void floor_empty_kernel() {
    grid_dep_wait();
    grid_dep_release();
}

constexpr int kFloorThreads = 256;

__global__ void __launch_bounds__(kFloorThreads)
floor_copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int64_t n16) {
    grid_dep_wait();
    grid_dep_release();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * 4 * kFloorThreads + threadIdx.x;
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t i = base + k * kFloorThreads;
        if (i < n16) v[k] = ld_stream(src + i);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t i = base + k * kFloorThreads;
        if (i < n16) st_stream(dst + i, v[k]);
    }
}

}  // namespace

size_t plan_workspace_bytes(int op, int64_t rows, int64_t hidden, int sms, int path, int partials) {
    if (path == NF_PATH_SPLIT) return split_workspace_bytes(op, rows, hidden, sms);
    if (path == NF_PATH_GRID) return grid_workspace_bytes(op, rows, hidden, sms);
    if (op == NF_OP_LAYERNORM_BWD || op == NF_OP_RMSNORM_BWD)
        return static_cast<size_t>(partials) * bwd_planes(static_cast<nf_op>(op)) *
               static_cast<size_t>(hidden) * sizeof(float);
    return 0;
}

cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace nf

using namespace nf;

extern "C" {

nf_status nf_plan_compute(nf_op op, int64_t rows, int64_t hidden, int32_t sm_count, nf_path path,
                          nf_plan* out) {
    if (!out || rows < 0 || sm_count < 1) return NF_ERR_INVALID_ARG;
    if (op < NF_OP_FUSED_ADD_RMSNORM || op > NF_OP_RMSNORM_BWD) return NF_ERR_INVALID_ARG;
    if (path < NF_PATH_AUTO || path > NF_PATH_GRID) return NF_ERR_INVALID_ARG;
    const bool fwd = op == NF_OP_FUSED_ADD_RMSNORM || op == NF_OP_RMSNORM_FWD ||
                     op == NF_OP_LAYERNORM_FWD;
    int tpr = 0, rpc = 1, dyn_threads = 0, long_c = 0, long_t = 0, long_slice = 0;
    const bool compiled = reg_shape(hidden, &tpr, &rpc);
    const bool dyn_ok = dyn_shape(op, hidden, &dyn_threads);
    const bool long_ok = long_shape(op, hidden, &long_c, &long_t, &long_slice);
    const bool splittable = split_ok(hidden);
    int grid_vc = 0;
    size_t grid_smem = 0;
    const bool grid_fits = grid_shape(op, rows, hidden, sm_count, &grid_vc, &grid_smem);
    if (!compiled && !dyn_ok && !long_ok && !splittable) return NF_ERR_UNSUPPORTED_HIDDEN;

    nf_path p = path;
    if (p == NF_PATH_AUTO)
        // beyond the runtime-hidden limits the split family beat the
        // cluster kernels at every measured row count (1.1-2.3x); where the
        // rows fit on chip the grid family beat it for the forward ops and
        // the LayerNorm backward (the RMSNorm backward keeps the split
        // family's copy-ring apply pass, which measured faster)
        p = compiled ? auto_path(op, rows, hidden, rpc, sm_count)
            : dyn_ok ? NF_PATH_DYNAMIC
            : splittable ? (grid_fits && op != NF_OP_RMSNORM_BWD ? NF_PATH_GRID : NF_PATH_SPLIT)
                         : NF_PATH_CLUSTER;
    if (p == NF_PATH_SPLIT && !splittable) return NF_ERR_UNSUPPORTED_PATH;
    if (p == NF_PATH_GRID && !grid_fits) return NF_ERR_UNSUPPORTED_PATH;
    if ((p == NF_PATH_REG || p == NF_PATH_BULK) && !compiled) return NF_ERR_UNSUPPORTED_PATH;
    if (p == NF_PATH_DYNAMIC && !dyn_ok) return NF_ERR_UNSUPPORTED_PATH;
    // the cluster family: the static kernels for compiled forward sizes,
    // the long-row (runtime hidden) kernels otherwise and for backward ops
    const bool long_cluster = p == NF_PATH_CLUSTER && !(fwd && compiled);
    if (long_cluster && !long_ok) return NF_ERR_UNSUPPORTED_PATH;

    nf_plan pl;
    std::memset(&pl, 0, sizeof pl);
    pl.path = p;
    constexpr int64_t kMaxGrid = 0x7FFFFFFF;
    if (p == NF_PATH_GRID) {
        // one cooperative launch, one CTA per SM holding its column slice of
        // every row; the backward writes dgamma / dbeta (dw) itself
        pl.grid = sm_count;
        pl.block = 512;
        pl.cluster = 1;
        pl.rows_per_cta = static_cast<int32_t>(rows);
        pl.smem_bytes = static_cast<int32_t>(grid_smem);
        pl.launches = 1;
        pl.partials = fwd ? 0 : 1;
    } else if (p == NF_PATH_SPLIT) {
        int nc, rb;
        split_shape(op, rows, hidden, sm_count, &nc, &rb);
        const int64_t ry = rows < 65535 ? (rows > 0 ? rows : 1) : 65535;
        pl.block = 256;
        pl.cluster = 1;
        pl.rows_per_cta = 1;
        if (fwd) {
            pl.grid = static_cast<int32_t>(static_cast<int64_t>(nc) * ry);
            // statistics, then apply (RMSNorm and the fused op merge their row's
            // partials there; LayerNorm has a merge launch between)
            pl.launches = op == NF_OP_LAYERNORM_FWD ? 3 : 2;
        } else {
            pl.grid = static_cast<int32_t>(static_cast<int64_t>(nc) * rb);
            // statistics, a merge launch unless the row blocks are short
            // enough to merge in the apply pass, apply, and the column
            // reduction unless one row block writes dgamma / dbeta itself
            const int64_t rows_per_block = (rows + rb - 1) / (rb > 0 ? rb : 1);
            pl.launches = 2 + (rows_per_block > kSplitMergeRows ? 1 : 0) + (rb > 1 ? 1 : 0);
            pl.partials = rb;
        }
    } else if (p == NF_PATH_REG && fwd) {
        // small calls: one row per CTA, twice the threads per row
        const bool small = rows <= kSmallCallRows;
        const int frpc = small ? 1 : rpc;
        const int64_t blocks = (rows + frpc - 1) / frpc;
        pl.grid = static_cast<int32_t>(blocks < kMaxGrid ? blocks : kMaxGrid);
        pl.block = (small ? 2 * tpr : tpr) * frpc;
        pl.cluster = 1;
        pl.rows_per_cta = frpc;
        pl.launches = 1;
    } else if (long_cluster) {
        pl.block = long_t;
        pl.cluster = long_c;
        pl.rows_per_cta = 1;
        if (fwd) {
            const int64_t max_clusters = kMaxGrid / long_c;
            const int64_t clusters = rows < max_clusters ? rows : max_clusters;
            pl.grid = static_cast<int32_t>(clusters * long_c);
            pl.launches = 1;
        } else {
            int64_t clusters = sm_count / long_c;
            if (clusters > rows) clusters = rows;
            if (clusters < 1) clusters = 1;
            pl.grid = static_cast<int32_t>(clusters * long_c);
            pl.launches = 2;
            pl.partials = static_cast<int32_t>(clusters);
        }
    } else if (p == NF_PATH_CLUSTER) {
        int c, t;
        if (!cluster_shape(hidden, &c, &t)) return NF_ERR_UNSUPPORTED_HIDDEN;
        const int64_t max_clusters = kMaxGrid / c;
        const int64_t clusters = rows < max_clusters ? rows : max_clusters;
        pl.grid = static_cast<int32_t>(clusters * c);
        pl.block = t;
        pl.cluster = c;
        pl.rows_per_cta = 1;
        pl.launches = 1;
    } else if (p == NF_PATH_DYNAMIC) {
        pl.block = dyn_threads;
        pl.cluster = 1;
        pl.rows_per_cta = 1;
        if (fwd) {
            // one CTA per row, or on rows of one warp one wave of resident
            // CTAs with a copy ring each
            const size_t ring = dyn_fwd_smem(op, hidden);
            const int64_t most = ring ? static_cast<int64_t>(sm_count) * dyn_fwd_per_sm(op, hidden) : kMaxGrid;
            pl.grid = static_cast<int32_t>(rows < most ? rows : most);
            pl.launches = 1;
            pl.smem_bytes = static_cast<int32_t>(ring);
        } else {
            // one wave of the CTAs that stay resident (for the RMSNorm
            // backward, counted with the fused-add backward's larger ring)
            const int64_t resident =
                static_cast<int64_t>(sm_count) * dyn_bwd_per_sm(hidden, op == NF_OP_RMSNORM_BWD);
            int64_t g = rows < resident ? rows : resident;
            if (g < 1) g = 1;
            pl.grid = static_cast<int32_t>(g);
            pl.launches = 2;
            pl.partials = static_cast<int32_t>(g);
            pl.smem_bytes = static_cast<int32_t>(dyn_bwd_smem(hidden, false));
        }
    } else if (p == NF_PATH_BULK) {
        int threads, stages, smem, groups, per_sm = 1;
        if (!bulk_shape(op, hidden, &threads, &stages, &smem, &groups)) return NF_ERR_UNSUPPORTED_PATH;
        int t2, s2, m2, g2;
        if (!fwd) rows_bwd_shape(op, hidden, &t2, &s2, &m2, &g2, &per_sm);  // row-block kernels
        const int64_t slots = static_cast<int64_t>(sm_count) * per_sm;
        int64_t g = rows < slots ? rows : slots;
        if (g < 1) g = 1;
        pl.grid = static_cast<int32_t>(g);
        pl.block = threads;
        pl.cluster = 1;
        pl.rows_per_cta = groups;  // rows being computed at once per CTA
        pl.smem_bytes = smem;
        pl.launches = fwd ? 1 : 2;
        pl.partials = fwd ? 0 : static_cast<int32_t>(g);  // groups fold into one slot per CTA
    } else {  // register-path backward: persistent stage 1 + column reduce
        const int64_t blocks = (rows + rpc - 1) / rpc;
        const int64_t resident = static_cast<int64_t>(sm_count) * bwd_ctas_per_sm(hidden);
        int64_t g = blocks < resident ? blocks : resident;
        if (g < 1) g = 1;
        pl.grid = static_cast<int32_t>(g);
        pl.block = tpr * rpc;
        pl.cluster = 1;
        pl.rows_per_cta = rpc;
        pl.launches = 2;
        pl.partials = static_cast<int32_t>(g * rpc);
    }
    *out = pl;
    return NF_OK;
}

nf_status nf_set_path(nf_path path) {
    if (path < NF_PATH_AUTO || path > NF_PATH_GRID) return NF_ERR_INVALID_ARG;
    g_forced_path.store(path, std::memory_order_relaxed);
    return NF_OK;
}

nf_status nf_plan_query(nf_op op, int64_t rows, int64_t hidden, nf_plan* out) {
    if (!out) return NF_ERR_INVALID_ARG;
    if (op < NF_OP_FUSED_ADD_RMSNORM || op > NF_OP_RMSNORM_BWD) return NF_ERR_INVALID_ARG;
    if (!hidden_supported(op, hidden)) return NF_ERR_UNSUPPORTED_HIDDEN;
    if (rows < 0) return NF_ERR_INVALID_ARG;
    return plan_for_call(op, rows, hidden, out);
}

size_t nf_workspace_size(nf_op op, int64_t rows, int64_t hidden) {
    if (op < NF_OP_FUSED_ADD_RMSNORM || op > NF_OP_RMSNORM_BWD) return 0;
    return any_path_workspace_bytes(op, rows, hidden);
}

nf_status nf_fused_add_rmsnorm(void* x, void* residual, const void* weight, int64_t rows,
                               int64_t hidden, float eps, nf_stream stream) {
    return nf_fused_add_rmsnorm_ws(x, residual, weight, rows, hidden, eps, nullptr, 0, stream);
}

nf_status nf_fused_add_rmsnorm_ws(void* x, void* residual, const void* weight, int64_t rows,
                                  int64_t hidden, float eps, void* workspace,
                                  size_t workspace_bytes, nf_stream stream) {
    if (nf_status st = common_checks(NF_OP_FUSED_ADD_RMSNORM, rows, hidden, eps, true)) return st;
    if (rows == 0) return NF_OK;
    if (!x || !residual || !weight) return NF_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(weight, 16)) return NF_ERR_MISALIGNED;
    const int64_t act = rows * hidden * 2, par = hidden * 2;
    if (overlap({x, act}, {residual, act}) || overlap({x, act}, {weight, par}) ||
        overlap({residual, act}, {weight, par}))
        return NF_ERR_INVALID_ARG;
    nf_plan pl;
    if (nf_status st = plan_for_fwd(NF_OP_FUSED_ADD_RMSNORM, rows, hidden, workspace != nullptr, &pl))
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (pl.path == NF_PATH_SPLIT || pl.path == NF_PATH_GRID) {
        size_t need;
        if (nf_status st = check_workspace(NF_OP_FUSED_ADD_RMSNORM, rows, hidden, pl, workspace,
                                           workspace_bytes, &need))
            return st;
        const Span sws{workspace, static_cast<int64_t>(need)};
        if (overlap(sws, {x, act}) || overlap(sws, {residual, act}) || overlap(sws, {weight, par}))
            return NF_ERR_INVALID_ARG;
        DynArgs a{};
        a.out0 = static_cast<uint16_t*>(x);
        a.out1 = static_cast<uint16_t*>(residual);
        a.in0 = static_cast<const uint16_t*>(x);
        a.in1 = static_cast<const uint16_t*>(residual);
        a.p0 = static_cast<const uint16_t*>(weight);
        a.rows = rows;
        a.hidden = static_cast<int>(hidden);
        a.eps = eps;
        return launch_split_family(pl, NF_OP_FUSED_ADD_RMSNORM, a, workspace, s);
    }
    if (pl.path == NF_PATH_CLUSTER && hidden_ok(hidden))
        return from_cuda(launch_fused_cluster(hidden, x, residual, weight, rows, eps, pl.grid, s));
    if (pl.path == NF_PATH_DYNAMIC || pl.path == NF_PATH_CLUSTER) {
        DynArgs a{};
        a.out0 = static_cast<uint16_t*>(x);
        a.out1 = static_cast<uint16_t*>(residual);
        a.in0 = static_cast<const uint16_t*>(x);
        a.in1 = static_cast<const uint16_t*>(residual);
        a.p0 = static_cast<const uint16_t*>(weight);
        a.rows = rows;
        a.hidden = static_cast<int>(hidden);
        a.eps = eps;
        if (pl.path == NF_PATH_CLUSTER) return from_cuda(launch_long(NF_OP_FUSED_ADD_RMSNORM, a, pl.grid, s));
        return from_cuda(launch_dyn(NF_OP_FUSED_ADD_RMSNORM, a, pl.grid, s));
    }
    if (pl.path == NF_PATH_BULK) {
        int* status;
        if (nf_status st = device_status_addr(&status)) return st;
        return from_cuda(launch_fused_bulk(hidden, x, residual, weight, rows, eps, pl.grid, status, s));
    }
    int sms;
    if (nf_status st = device_sm_count(&sms)) return st;
    return from_cuda(launch_fused_reg(hidden, x, residual, weight, rows, eps, pl.grid, sms, s));
}

nf_status nf_rmsnorm_fwd(void* y, const void* x, const void* weight, int64_t rows, int64_t hidden,
                         float eps, nf_stream stream) {
    return nf_rmsnorm_fwd_ws(y, x, weight, rows, hidden, eps, nullptr, 0, stream);
}

nf_status nf_rmsnorm_fwd_ws(void* y, const void* x, const void* weight, int64_t rows,
                            int64_t hidden, float eps, void* workspace, size_t workspace_bytes,
                            nf_stream stream) {
    if (nf_status st = common_checks(NF_OP_RMSNORM_FWD, rows, hidden, eps, true)) return st;
    if (rows == 0) return NF_OK;
    if (!y || !x || !weight) return NF_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(x, 16) || !aligned(weight, 16)) return NF_ERR_MISALIGNED;
    const int64_t act = rows * hidden * 2, par = hidden * 2;
    if (bad_overlap_except_alias({y, act}, {x, act}) || overlap({y, act}, {weight, par}))
        return NF_ERR_INVALID_ARG;
    nf_plan pl;
    if (nf_status st = plan_for_fwd(NF_OP_RMSNORM_FWD, rows, hidden, workspace != nullptr, &pl))
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (pl.path == NF_PATH_SPLIT || pl.path == NF_PATH_GRID) {
        size_t need;
        if (nf_status st = check_workspace(NF_OP_RMSNORM_FWD, rows, hidden, pl, workspace,
                                           workspace_bytes, &need))
            return st;
        const Span sws{workspace, static_cast<int64_t>(need)};
        if (overlap(sws, {y, act}) || overlap(sws, {x, act}) || overlap(sws, {weight, par}))
            return NF_ERR_INVALID_ARG;
        DynArgs a{};
        a.out0 = static_cast<uint16_t*>(y);
        a.in0 = static_cast<const uint16_t*>(x);
        a.p0 = static_cast<const uint16_t*>(weight);
        a.rows = rows;
        a.hidden = static_cast<int>(hidden);
        a.eps = eps;
        return launch_split_family(pl, NF_OP_RMSNORM_FWD, a, workspace, s);
    }
    if (pl.path == NF_PATH_CLUSTER && hidden_ok(hidden))
        return from_cuda(launch_rms_cluster(hidden, y, x, weight, rows, eps, pl.grid, s));
    if (pl.path == NF_PATH_DYNAMIC || pl.path == NF_PATH_CLUSTER) {
        DynArgs a{};
        a.out0 = static_cast<uint16_t*>(y);
        a.in0 = static_cast<const uint16_t*>(x);
        a.p0 = static_cast<const uint16_t*>(weight);
        a.rows = rows;
        a.hidden = static_cast<int>(hidden);
        a.eps = eps;
        if (pl.path == NF_PATH_CLUSTER) return from_cuda(launch_long(NF_OP_RMSNORM_FWD, a, pl.grid, s));
        return from_cuda(launch_dyn(NF_OP_RMSNORM_FWD, a, pl.grid, s));
    }
    if (pl.path == NF_PATH_BULK) {
        int* status;
        if (nf_status st = device_status_addr(&status)) return st;
        return from_cuda(launch_rms_bulk(hidden, y, x, weight, rows, eps, pl.grid, status, s));
    }
    int sms;
    if (nf_status st = device_sm_count(&sms)) return st;
    return from_cuda(launch_rms_reg(hidden, y, x, weight, rows, eps, pl.grid, sms, s));
}

nf_status nf_layernorm_fwd(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                           const void* beta, int64_t rows, int64_t hidden, float eps,
                           nf_stream stream) {
    return nf_layernorm_fwd_ws(y, mean, rstd, x, gamma, beta, rows, hidden, eps, nullptr, 0,
                               stream);
}

nf_status nf_layernorm_fwd_ws(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                              const void* beta, int64_t rows, int64_t hidden, float eps,
                              void* workspace, size_t workspace_bytes, nf_stream stream) {
    if (nf_status st = common_checks(NF_OP_LAYERNORM_FWD, rows, hidden, eps, true)) return st;
    if (rows == 0) return NF_OK;
    if (!y || !x || !gamma || !beta) return NF_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(x, 16) || !aligned(gamma, 16) || !aligned(beta, 16))
        return NF_ERR_MISALIGNED;
    if (!aligned(mean, 4) || !aligned(rstd, 4)) return NF_ERR_MISALIGNED;
    const int64_t act = rows * hidden * 2, par = hidden * 2, stat = rows * 4;
    if (bad_overlap_except_alias({y, act}, {x, act}) || overlap({y, act}, {gamma, par}) ||
        overlap({y, act}, {beta, par}) || overlap({mean, stat}, {rstd, stat}))
        return NF_ERR_INVALID_ARG;
    for (Span o : {Span{mean, stat}, Span{rstd, stat}})
        if (overlap(o, {y, act}) || overlap(o, {x, act}) || overlap(o, {gamma, par}) ||
            overlap(o, {beta, par}))
            return NF_ERR_INVALID_ARG;
    nf_plan pl;
    if (nf_status st = plan_for_fwd(NF_OP_LAYERNORM_FWD, rows, hidden, workspace != nullptr, &pl))
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (pl.path == NF_PATH_SPLIT || pl.path == NF_PATH_GRID) {
        size_t need;
        if (nf_status st = check_workspace(NF_OP_LAYERNORM_FWD, rows, hidden, pl, workspace,
                                           workspace_bytes, &need))
            return st;
        const Span sws{workspace, static_cast<int64_t>(need)};
        if (overlap(sws, {y, act}) || overlap(sws, {x, act}) || overlap(sws, {gamma, par}) ||
            overlap(sws, {beta, par}) || overlap(sws, {mean, stat}) || overlap(sws, {rstd, stat}))
            return NF_ERR_INVALID_ARG;
        DynArgs a{};
        a.out0 = static_cast<uint16_t*>(y);
        a.in0 = static_cast<const uint16_t*>(x);
        a.p0 = static_cast<const uint16_t*>(gamma);
        a.p1 = static_cast<const uint16_t*>(beta);
        a.mean = mean;
        a.rstd = rstd;
        a.rows = rows;
        a.hidden = static_cast<int>(hidden);
        a.eps = eps;
        return launch_split_family(pl, NF_OP_LAYERNORM_FWD, a, workspace, s);
    }
    if (pl.path == NF_PATH_CLUSTER && hidden_ok(hidden))
        return from_cuda(launch_ln_fwd_cluster(hidden, y, mean, rstd, x, gamma, beta, rows, eps,
                                               pl.grid, s));
    if (pl.path == NF_PATH_DYNAMIC || pl.path == NF_PATH_CLUSTER) {
        DynArgs a{};
        a.out0 = static_cast<uint16_t*>(y);
        a.in0 = static_cast<const uint16_t*>(x);
        a.p0 = static_cast<const uint16_t*>(gamma);
        a.p1 = static_cast<const uint16_t*>(beta);
        a.mean = mean;
        a.rstd = rstd;
        a.rows = rows;
        a.hidden = static_cast<int>(hidden);
        a.eps = eps;
        if (pl.path == NF_PATH_CLUSTER) return from_cuda(launch_long(NF_OP_LAYERNORM_FWD, a, pl.grid, s));
        return from_cuda(launch_dyn(NF_OP_LAYERNORM_FWD, a, pl.grid, s));
    }
    if (pl.path == NF_PATH_BULK) {
        int* status;
        if (nf_status st = device_status_addr(&status)) return st;
        return from_cuda(launch_ln_fwd_bulk(hidden, y, mean, rstd, x, gamma, beta, rows, eps,
                                            pl.grid, status, s));
    }
    int sms;
    if (nf_status st = device_sm_count(&sms)) return st;
    return from_cuda(launch_ln_fwd_reg(hidden, y, mean, rstd, x, gamma, beta, rows, eps, pl.grid, sms, s));
}

size_t nf_layernorm_bwd_workspace_size(int64_t rows, int64_t hidden) {
    return bwd_workspace_bytes(NF_OP_LAYERNORM_BWD, rows, hidden);
}

nf_status nf_layernorm_bwd(void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                           const float* mean, const float* rstd, const void* gamma, int64_t rows,
                           int64_t hidden, void* workspace, size_t workspace_bytes,
                           nf_stream stream) {
    return nf::layernorm_bwd_impl(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows, hidden,
                                  workspace, workspace_bytes, nullptr, stream);
}

}  // extern "C"

namespace nf {

// (declared in internal.h)
nf_status layernorm_bwd_impl(void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                             const float* mean, const float* rstd, const void* gamma, int64_t rows,
                             int64_t hidden, void* workspace, size_t workspace_bytes,
                             nf_status (*scratch)(void**), nf_stream stream) {
    if (nf_status st = common_checks(NF_OP_LAYERNORM_BWD, rows, hidden, 0.f, false)) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0) {
        // an empty sum: dgamma = dbeta = 0
        if (dgamma && !aligned(dgamma, 16)) return NF_ERR_MISALIGNED;
        if (dbeta && !aligned(dbeta, 16)) return NF_ERR_MISALIGNED;
        if (dgamma && cudaMemsetAsync(dgamma, 0, hidden * sizeof(float), s) != cudaSuccess) return NF_ERR_CUDA;
        if (dbeta && cudaMemsetAsync(dbeta, 0, hidden * sizeof(float), s) != cudaSuccess) return NF_ERR_CUDA;
        return NF_OK;
    }
    if (!dx || !dgamma || !dbeta || !dy || !x || !mean || !rstd || !gamma || (!scratch && !workspace))
        return NF_ERR_INVALID_ARG;
    if (!aligned(dx, 16) || !aligned(dy, 16) || !aligned(x, 16) || !aligned(gamma, 16) ||
        (!scratch && !aligned(workspace, 16)) || !aligned(dgamma, 16) || !aligned(dbeta, 16) ||
        !aligned(mean, 4) || !aligned(rstd, 4))
        return NF_ERR_MISALIGNED;
    nf_plan pl;
    if (nf_status st = plan_for_call(NF_OP_LAYERNORM_BWD, rows, hidden, &pl)) return st;
    size_t need;
    if (scratch) {
        int sms;
        if (nf_status st = device_sm_count(&sms)) return st;
        need = plan_workspace_bytes(NF_OP_LAYERNORM_BWD, rows, hidden, sms, pl.path, pl.partials);
        if (need > workspace_bytes) return NF_ERR_WORKSPACE_TOO_SMALL;
        workspace = nullptr;  // the library's own area cannot overlap the caller's buffers
    } else if (nf_status st = check_workspace(NF_OP_LAYERNORM_BWD, rows, hidden, pl, workspace,
                                              workspace_bytes, &need)) {
        return st;
    }
    const int64_t act = rows * hidden * 2, par = hidden * 2, stat = rows * 4, grad = hidden * 4;
    const Span sdx{dx, act}, sdg{dgamma, grad}, sdb{dbeta, grad}, sws{workspace, static_cast<int64_t>(need)};
    const Span ins[] = {{dy, act}, {x, act}, {mean, stat}, {rstd, stat}, {gamma, par}};
    if (overlap(sdg, sdb) || overlap(sdx, sdg) || overlap(sdx, sdb) || overlap(sws, sdx) ||
        overlap(sws, sdg) || overlap(sws, sdb))
        return NF_ERR_INVALID_ARG;
    for (int i = 0; i < 5; ++i) {
        const Span& in = ins[i];
        // dx may be exactly dy or x (each row is read before it is written)
        const bool dx_clash = i < 2 ? bad_overlap_except_alias(sdx, in) : overlap(sdx, in);
        if (dx_clash || overlap(sdg, in) || overlap(sdb, in) || overlap(sws, in))
            return NF_ERR_INVALID_ARG;
    }
    if (scratch) {
        if (nf_status st = scratch(&workspace)) return st;
    }
    float* ws = static_cast<float*>(workspace);
    if (pl.path == NF_PATH_DYNAMIC || pl.path == NF_PATH_CLUSTER || pl.path == NF_PATH_SPLIT ||
        pl.path == NF_PATH_GRID) {
        DynArgs a{};
        a.out0 = static_cast<uint16_t*>(dx);
        a.in0 = static_cast<const uint16_t*>(x);
        a.in1 = static_cast<const uint16_t*>(dy);
        a.p0 = static_cast<const uint16_t*>(gamma);
        a.mean = const_cast<float*>(mean);
        a.rstd = const_cast<float*>(rstd);
        a.ws = ws;
        a.rows = rows;
        a.hidden = static_cast<int>(hidden);
        int sms = 0;
        if (pl.path == NF_PATH_SPLIT || pl.path == NF_PATH_GRID) {
            if (nf_status st = device_sm_count(&sms)) return st;
            if (pl.partials == 1) {  // one row block: no column reduction
                a.cols0 = dgamma;
                a.cols1 = dbeta;
                return launch_split_family(pl, NF_OP_LAYERNORM_BWD, a, workspace, s);
            }
        }
        const cudaError_t e =
            pl.path == NF_PATH_SPLIT     ? launch_split(NF_OP_LAYERNORM_BWD, a, workspace, sms, s)
            : pl.path == NF_PATH_CLUSTER ? launch_long(NF_OP_LAYERNORM_BWD, a, pl.grid, s)
                                         : launch_dyn(NF_OP_LAYERNORM_BWD, a, pl.grid, s);
        if (e != cudaSuccess) return from_cuda(e);
    } else if (pl.path == NF_PATH_BULK) {
        int* status;
        if (nf_status st = device_status_addr(&status)) return st;
        if (cudaError_t e = launch_ln_bwd_bulk(hidden, dx, ws, dy, x, mean, rstd, gamma, rows,
                                               pl.grid, status, s))
            return from_cuda(e);
    } else if (cudaError_t e = launch_ln_bwd_reg(hidden, dx, ws, dy, x, mean, rstd, gamma, rows,
                                                 pl.grid, s)) {
        return from_cuda(e);
    }
    return from_cuda(launch_column_reduce(ws, dgamma, dbeta, pl.partials, hidden, s));
}

}  // namespace nf

extern "C" {

size_t nf_rmsnorm_bwd_workspace_size(int64_t rows, int64_t hidden) {
    return bwd_workspace_bytes(NF_OP_RMSNORM_BWD, rows, hidden);
}

namespace {
// RMSNorm backward, optionally with a residual-stream gradient `dres` added
// to dx (the fused residual-add + RMSNorm backward).
nf_status rms_bwd(void* dx, float* dw, const void* dy, const void* x, const void* dres,
                  const void* weight, int64_t rows, int64_t hidden, float eps, void* workspace,
                  size_t workspace_bytes, nf_stream stream) {
    if (nf_status st = common_checks(NF_OP_RMSNORM_BWD, rows, hidden, eps, true)) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0) {
        // an empty sum: dw = 0
        if (dw && !aligned(dw, 16)) return NF_ERR_MISALIGNED;
        if (dw && cudaMemsetAsync(dw, 0, hidden * sizeof(float), s) != cudaSuccess) return NF_ERR_CUDA;
        return NF_OK;
    }
    if (!dx || !dw || !dy || !x || !weight || !workspace) return NF_ERR_INVALID_ARG;
    if (!aligned(dx, 16) || !aligned(dy, 16) || !aligned(x, 16) || !aligned(weight, 16) ||
        !aligned(workspace, 16) || !aligned(dw, 16) || !aligned(dres, 16))
        return NF_ERR_MISALIGNED;
    nf_plan pl;
    if (nf_status st = plan_for_call(NF_OP_RMSNORM_BWD, rows, hidden, &pl)) return st;
    size_t need;
    if (nf_status st = check_workspace(NF_OP_RMSNORM_BWD, rows, hidden, pl, workspace,
                                       workspace_bytes, &need))
        return st;
    const int64_t act = rows * hidden * 2, par = hidden * 2, grad = hidden * 4;
    const Span sdx{dx, act}, sdw{dw, grad}, sws{workspace, static_cast<int64_t>(need)};
    const Span ins[] = {{dy, act}, {x, act}, {dres, dres ? act : 0}, {weight, par}};
    if (overlap(sdx, sdw) || overlap(sws, sdx) || overlap(sws, sdw)) return NF_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i) {
        const Span& in = ins[i];
        // dx may be exactly dy, x or dres (each row is read before it is written)
        const bool dx_clash = i < 3 ? bad_overlap_except_alias(sdx, in) : overlap(sdx, in);
        if (dx_clash || overlap(sdw, in) || overlap(sws, in)) return NF_ERR_INVALID_ARG;
    }
    float* ws = static_cast<float*>(workspace);
    if (pl.path == NF_PATH_DYNAMIC || pl.path == NF_PATH_CLUSTER || pl.path == NF_PATH_SPLIT ||
        pl.path == NF_PATH_GRID) {
        DynArgs a{};
        a.out0 = static_cast<uint16_t*>(dx);
        a.in0 = static_cast<const uint16_t*>(x);
        a.in1 = static_cast<const uint16_t*>(dy);
        a.p0 = static_cast<const uint16_t*>(weight);
        a.add = static_cast<const uint16_t*>(dres);
        a.ws = ws;
        a.rows = rows;
        a.hidden = static_cast<int>(hidden);
        a.eps = eps;
        int sms = 0;
        if (pl.path == NF_PATH_SPLIT || pl.path == NF_PATH_GRID) {
            if (nf_status st = device_sm_count(&sms)) return st;
            if (pl.partials == 1) {  // one row block: no column reduction
                a.cols0 = dw;
                return launch_split_family(pl, NF_OP_RMSNORM_BWD, a, workspace, s);
            }
        }
        const cudaError_t e =
            pl.path == NF_PATH_SPLIT     ? launch_split(NF_OP_RMSNORM_BWD, a, workspace, sms, s)
            : pl.path == NF_PATH_CLUSTER ? launch_long(NF_OP_RMSNORM_BWD, a, pl.grid, s)
                                         : launch_dyn(NF_OP_RMSNORM_BWD, a, pl.grid, s);
        if (e != cudaSuccess) return from_cuda(e);
    } else if (pl.path == NF_PATH_BULK) {
        int* status;
        if (nf_status st = device_status_addr(&status)) return st;
        if (cudaError_t e = launch_rms_bwd_bulk(hidden, dx, ws, dy, x, dres, weight, rows, eps,
                                                pl.grid, status, s))
            return from_cuda(e);
    } else if (cudaError_t e = launch_rms_bwd_reg(hidden, dx, ws, dy, x, dres, weight, rows, eps,
                                                  pl.grid, s)) {
        return from_cuda(e);
    }
    return from_cuda(launch_column_reduce1(ws, dw, pl.partials, hidden, s));
}
}  // namespace

nf_status nf_rmsnorm_bwd(void* dx, float* dw, const void* dy, const void* x, const void* weight,
                         int64_t rows, int64_t hidden, float eps, void* workspace,
                         size_t workspace_bytes, nf_stream stream) {
    return rms_bwd(dx, dw, dy, x, nullptr, weight, rows, hidden, eps, workspace, workspace_bytes,
                   stream);
}

nf_status nf_fused_add_rmsnorm_bwd(void* dx, float* dw, const void* dy, const void* dres,
                                   const void* residual, const void* weight, int64_t rows,
                                   int64_t hidden, float eps, void* workspace,
                                   size_t workspace_bytes, nf_stream stream) {
    return rms_bwd(dx, dw, dy, residual, dres, weight, rows, hidden, eps, workspace,
                   workspace_bytes, stream);
}

size_t nf_outer_norm_workspace_size(int64_t rows, int64_t hidden) {
    if (rows <= 0 || hidden < 8 || hidden % 8 != 0 || hidden > 0x7FFFFFFF) return 0;
    int sms;
    if (device_sm_count(&sms) != NF_OK) return 0;
    return outer_workspace_bytes(rows, hidden, sms);
}

namespace {
nf_status outer_checks(int64_t rows, int64_t hidden) {
    if (hidden < 8 || hidden % 8 != 0 || hidden > 0x7FFFFFFF) return NF_ERR_UNSUPPORTED_HIDDEN;
    if (rows < 0 || rows > (INT64_MAX / 8) / hidden) return NF_ERR_INVALID_ARG;
    return NF_OK;
}

// Outer normalization's two forms: the three-launch streaming passes (the
// automatic choice) and the grid family's single launch with the row
// stripes on chip, forced with NF_PATH_GRID (it measured slower at every
// size: 125-136 against 66 us at 16384 x 4096; its two grid barriers and
// merge per band of columns leave DRAM idle between bands).  *grid says
// which.
nf_status outer_form(int64_t rows, int64_t hidden, int sms, bool* grid) {
    const int forced = g_forced_path.load(std::memory_order_relaxed);
    const bool fits = outer_grid_shape(rows, hidden, sms, nullptr, nullptr);
    if (forced == NF_PATH_GRID && !fits) return NF_ERR_UNSUPPORTED_PATH;
    *grid = forced == NF_PATH_GRID;
    return NF_OK;
}
}  // namespace

nf_status nf_outer_norm_fwd(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                            const void* beta, int64_t rows, int64_t hidden, float eps,
                            void* workspace, size_t workspace_bytes, nf_stream stream) {
    if (nf_status st = outer_checks(rows, hidden)) return st;
    if (!(std::isfinite(eps) && eps > 0.f)) return NF_ERR_INVALID_ARG;
    if (rows == 0) return NF_OK;
    if (!y || !x || !gamma || !beta || !workspace) return NF_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(x, 16) || !aligned(gamma, 2) || !aligned(beta, 2) ||
        !aligned(workspace, 16) || !aligned(mean, 4) || !aligned(rstd, 4))
        return NF_ERR_MISALIGNED;
    int sms;
    if (nf_status st = device_sm_count(&sms)) return st;
    bool grid;
    if (nf_status st = outer_form(rows, hidden, sms, &grid)) return st;
    const size_t need = outer_workspace_bytes(rows, hidden, sms);
    if (workspace_bytes < need) return NF_ERR_WORKSPACE_TOO_SMALL;
    const int64_t act = rows * hidden * 2, par = hidden * 2, stat = hidden * 4;
    const Span sy{y, act}, sws{workspace, static_cast<int64_t>(need)};
    const Span ins[] = {{x, act}, {gamma, par}, {beta, par}};
    for (int i = 0; i < 3; ++i) {
        const bool clash = i == 0 ? bad_overlap_except_alias(sy, ins[i]) : overlap(sy, ins[i]);
        if (clash || overlap(sws, ins[i])) return NF_ERR_INVALID_ARG;
    }
    if (overlap(sws, sy) || overlap({mean, stat}, {rstd, stat})) return NF_ERR_INVALID_ARG;
    for (Span o : {Span{mean, stat}, Span{rstd, stat}})
        if (overlap(o, sy) || overlap(o, sws) || overlap(o, ins[0]) || overlap(o, ins[1]) ||
            overlap(o, ins[2]))
            return NF_ERR_INVALID_ARG;
    if (grid) {
        int* status;
        if (nf_status st = device_status_addr(&status)) return st;
        return from_cuda(launch_outer_grid_fwd(y, mean, rstd, x, gamma, beta, rows, hidden, eps,
                                               workspace, sms, status,
                                               reinterpret_cast<cudaStream_t>(stream)));
    }
    return from_cuda(launch_outer_fwd(y, mean, rstd, x, gamma, beta, rows, hidden, eps, workspace,
                                      sms, reinterpret_cast<cudaStream_t>(stream)));
}

nf_status nf_outer_norm_bwd(void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                            const float* mean, const float* rstd, const void* gamma, int64_t rows,
                            int64_t hidden, void* workspace, size_t workspace_bytes,
                            nf_stream stream) {
    if (nf_status st = outer_checks(rows, hidden)) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0) {
        if (dgamma && !aligned(dgamma, 16)) return NF_ERR_MISALIGNED;
        if (dbeta && !aligned(dbeta, 16)) return NF_ERR_MISALIGNED;
        if (dgamma && cudaMemsetAsync(dgamma, 0, hidden * sizeof(float), s) != cudaSuccess) return NF_ERR_CUDA;
        if (dbeta && cudaMemsetAsync(dbeta, 0, hidden * sizeof(float), s) != cudaSuccess) return NF_ERR_CUDA;
        return NF_OK;
    }
    if (!dx || !dgamma || !dbeta || !dy || !x || !mean || !rstd || !gamma || !workspace)
        return NF_ERR_INVALID_ARG;
    if (!aligned(dx, 16) || !aligned(dy, 16) || !aligned(x, 16) || !aligned(gamma, 16) ||
        !aligned(workspace, 16) || !aligned(dgamma, 16) || !aligned(dbeta, 16) ||
        !aligned(mean, 4) || !aligned(rstd, 4))
        return NF_ERR_MISALIGNED;
    int sms;
    if (nf_status st = device_sm_count(&sms)) return st;
    const size_t need = outer_workspace_bytes(rows, hidden, sms);
    if (workspace_bytes < need) return NF_ERR_WORKSPACE_TOO_SMALL;
    const int64_t act = rows * hidden * 2, par = hidden * 2, stat = hidden * 4, grad = hidden * 4;
    const Span sdx{dx, act}, sdg{dgamma, grad}, sdb{dbeta, grad}, sws{workspace, static_cast<int64_t>(need)};
    const Span ins[] = {{dy, act}, {x, act}, {mean, stat}, {rstd, stat}, {gamma, par}};
    if (overlap(sdg, sdb) || overlap(sdx, sdg) || overlap(sdx, sdb) || overlap(sws, sdx) ||
        overlap(sws, sdg) || overlap(sws, sdb))
        return NF_ERR_INVALID_ARG;
    for (int i = 0; i < 5; ++i) {
        const Span& in = ins[i];
        const bool dx_clash = i < 2 ? bad_overlap_except_alias(sdx, in) : overlap(sdx, in);
        if (dx_clash || overlap(sdg, in) || overlap(sdb, in) || overlap(sws, in))
            return NF_ERR_INVALID_ARG;
    }
    return from_cuda(launch_outer_bwd(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows, hidden,
                                      workspace, sms, s));
}

nf_status nf_get_device_status(nf_stream stream) {
    int* addr;
    if (nf_status st = device_status_addr(&addr)) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, addr, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return NF_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return NF_ERR_CUDA;
    if (v != 0) {
        if (cudaMemsetAsync(addr, 0, sizeof(int), s) != cudaSuccess) return NF_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return NF_ERR_CUDA;
    }
    return static_cast<nf_status>(v);
}

nf_status nf_selftest_wait_timeout(int64_t timeout_ns, nf_stream stream) {
    int* addr;
    if (nf_status st = device_status_addr(&addr)) return st;
    if (timeout_ns < 1000) timeout_ns = 1000;
    if (timeout_ns > 1000000000) timeout_ns = 1000000000;
    return from_cuda(launch_wait_selftest(addr, static_cast<uint64_t>(timeout_ns),
                                          reinterpret_cast<cudaStream_t>(stream)));
}

nf_status nf_selftest_grid_timeout(void* workspace, int64_t timeout_ns, nf_stream stream) {
    if (!workspace) return NF_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return NF_ERR_MISALIGNED;
    int* addr;
    if (nf_status st = device_status_addr(&addr)) return st;
    if (timeout_ns < 1000) timeout_ns = 1000;
    if (timeout_ns > 1000000000) timeout_ns = 1000000000;
    return from_cuda(launch_grid_selftest(workspace, static_cast<uint64_t>(timeout_ns), addr,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

nf_status nf_selftest_floor(int32_t kind, void* dst, const void* src, int64_t bytes,
                            nf_stream stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (kind == 0) return from_cuda(launch_with_pdl(floor_empty_kernel, dim3(1), dim3(32), 0, s));
    if (kind != 1) return NF_ERR_INVALID_ARG;
    if (!dst || !src || bytes <= 0 || bytes % 16 != 0) return NF_ERR_INVALID_ARG;
    if (!aligned(dst, 16) || !aligned(src, 16)) return NF_ERR_MISALIGNED;
    if (overlap({dst, bytes}, {src, bytes})) return NF_ERR_INVALID_ARG;
    const int64_t n16 = bytes / 16;
    const int64_t grid = (n16 + 4 * kFloorThreads - 1) / (4 * kFloorThreads);
    if (grid > 0x7FFFFFFF) return NF_ERR_INVALID_ARG;
    return from_cuda(launch_with_pdl(floor_copy_kernel, dim3(static_cast<unsigned>(grid)),
                                     dim3(kFloorThreads), 0, s, static_cast<uint4*>(dst),
                                     static_cast<const uint4*>(src), n16));
}

const char* nf_status_string(nf_status status) {
    switch (status) {
        case NF_OK: return "NF_OK";
        case NF_ERR_INVALID_ARG: return "NF_ERR_INVALID_ARG";
        case NF_ERR_UNSUPPORTED_HIDDEN: return "NF_ERR_UNSUPPORTED_HIDDEN";
        case NF_ERR_MISALIGNED: return "NF_ERR_MISALIGNED";
        case NF_ERR_WORKSPACE_TOO_SMALL: return "NF_ERR_WORKSPACE_TOO_SMALL";
        case NF_ERR_CUDA: return "NF_ERR_CUDA";
        case NF_ERR_TIMEOUT: return "NF_ERR_TIMEOUT";
        case NF_ERR_UNSUPPORTED_PATH: return "NF_ERR_UNSUPPORTED_PATH";
        default: return "NF_ERR_UNKNOWN";
    }
}

const char* nf_version(void) { return "nf 0.1 (sm_103a)"; }

}  // extern "C"
