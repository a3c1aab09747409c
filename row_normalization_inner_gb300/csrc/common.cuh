// Device primitives shared by the row-normalization kernels (sm_103a).
//
// 128-bit vector access to bf16 rows, bf16 <-> fp32 conversion, and the fp32
// warp / row-group reductions.  The per-thread layout follows the static
// split the inner persistent scheduler uses once the hidden size is a
// compile-time constant ("optimize inner persistent scheduler for static
// fusion", reviewer guide, split [R, TIDx, Vect]): element
//     j = (k * TPR + t) * 8 + e,   k < VPT, t < TPR, e < 8,
// so consecutive threads touch consecutive 16-byte vectors (coalesced) and
// each thread keeps VPT vectors of its row in registers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nf {

constexpr int kVec = 8;  // bf16 elements per 128-bit vector

// The compiled hidden sizes and their register-path shape: TPR threads per
// row (a multiple of 32), RPC rows per CTA, VPT = hidden / 8 / TPR vectors
// per thread.
template <int H> struct RegShape;
template <> struct RegShape<1024>  { static constexpr int TPR = 32,  RPC = 2; };
template <> struct RegShape<2048>  { static constexpr int TPR = 64,  RPC = 2; };
template <> struct RegShape<4096>  { static constexpr int TPR = 128, RPC = 2; };
template <> struct RegShape<5120>  { static constexpr int TPR = 160, RPC = 1; };
template <> struct RegShape<8192>  { static constexpr int TPR = 256, RPC = 1; };
template <> struct RegShape<12288> { static constexpr int TPR = 384, RPC = 1; };

// ---- loads / stores -------------------------------------------------------
// Activations are touched once: stream them (evict-first).  Parameters are
// shared by every row: read them through the read-only path so they stay
// in cache.
__device__ __forceinline__ uint4 ld_stream(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ uint4 ld_param(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void st_stream(void* p, uint4 v) { __stcs(reinterpret_cast<uint4*>(p), v); }

// Warm L2 with the line that holds p.  A hint only: no thread reads a
// different value because of it, and L2 is where global memory is kept
// coherent, so a kernel launched as a programmatic dependent may issue it
// for its first rows before griddepcontrol.wait; DRAM then serves those
// rows while the kernel before it drains.  Only addresses inside the
// caller's buffers are passed.
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// A read-only load that asks L2 to keep the line (evict-last priority): for
// data a later kernel of the same operation reads again.
__device__ __forceinline__ uint4 ld_keep(const void* p) {
    uint4 v;
    asm volatile("{\n\t.reg .b64 pol;\n\t"
                 "createpolicy.fractional.L2::evict_last.b64 pol, 1.0;\n\t"
                 "ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], pol;\n\t}"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// ---- bf16 <-> fp32 ----------------------------------------------------------
// Widening is exact: a bf16 is the high half of a binary32 pattern.
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
    f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
    f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// Round two floats to bf16 (nearest, ties to even) and pack them, the first
// in the low half (lower address).
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 v;
    v.x = pack2(f[0], f[1]);
    v.y = pack2(f[2], f[3]);
    v.z = pack2(f[4], f[5]);
    v.w = pack2(f[6], f[7]);
    return v;
}

// ---- reductions ----------------------------------------------------------------
template <int N>
__device__ __forceinline__ void warp_sum(float (&v)[N]) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], off);
    }
}

// Sum N values over the TPR threads of one row group.  `red` is a shared
// buffer of RPC * (TPR/32) * N floats used by this call only (each call
// site passes its own, so no barrier is needed before reuse).  Every thread
// of the group gets the same result: warps are summed in a fixed order.
// All threads of the CTA must call this (it contains __syncthreads when a
// row spans several warps).
template <int TPR, int N>
__device__ __forceinline__ void group_sum(float (&v)[N], float* red, int group, int t) {
    warp_sum<N>(v);
    if constexpr (TPR > 32) {
        constexpr int W = TPR / 32;
        const int warp = t >> 5, lane = t & 31;
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < N; ++i) red[(group * W + warp) * N + i] = v[i];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < N; ++i) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) s += red[(group * W + w) * N + i];
            v[i] = s;
        }
    }
}

// ---- shared-memory barriers with bounded waits ------------------------------
// Every wait on an mbarrier gives up after a time limit measured on the
// global nanosecond timer, so a kernel can never spin forever: the caller
// records NF_ERR_TIMEOUT (6) in the device status word and returns.
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed, or until
// `timeout_ns` has passed.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

// First error wins; later ones do not overwrite it.
__device__ __forceinline__ void record_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

constexpr int kStatusTimeout = 6;                   // = NF_ERR_TIMEOUT
constexpr uint64_t kWaitLimitNs = 2000000000ull;    // 2 s: far above any legal wait

}  // namespace nf

// Expand the statement list once per compiled hidden size with `H` bound to
// that size as a constant expression; other sizes return
// cudaErrorInvalidValue from the enclosing function.
#define NF_HIDDEN_SWITCH(hidden, ...)                              \
    switch (hidden) {                                              \
        case 1024:  { constexpr int H = 1024;  __VA_ARGS__ } break; \
        case 2048:  { constexpr int H = 2048;  __VA_ARGS__ } break; \
        case 4096:  { constexpr int H = 4096;  __VA_ARGS__ } break; \
        case 5120:  { constexpr int H = 5120;  __VA_ARGS__ } break; \
        case 8192:  { constexpr int H = 8192;  __VA_ARGS__ } break; \
        case 12288: { constexpr int H = 12288; __VA_ARGS__ } break; \
        default: break;                                            \
    }                                                              \
    return cudaErrorInvalidValue;
