// LayerNorm backward without a caller-provided workspace.
//
// nf_layernorm_bwd needs a scratch buffer for its per-CTA column partials,
// and its caller has to allocate it.  Some callers cannot allocate device
// memory at the point where they run the backward pass: code that runs
// while an allocator is forbidden or unavailable (inside a region where the
// framework's caching allocator must not be entered, in a plugin that only
// receives pre-allocated tensors, in a real-time path where cudaMalloc's
// implicit synchronization is not acceptable).  For them this file keeps a
// fixed scratch area in the library's own static device memory and runs
// the ordinary LayerNorm backward on it.
//
// The area is a file-scope __device__ array: every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  In
// host code its name only stands in for the device object, so the device
// address is looked up once per device with cudaGetSymbolAddress (with that
// device current) and cached; that first call on a device should come
// before any stream capture.  A cudaDeviceReset ends the context that owns
// the area, so the cached address is stale afterwards: a process that
// resets a device must not call this entry point on it again.  Calls that
// overlap on the GPU (different streams, or different host threads) share
// the one area and race.
#include <cuda_runtime.h>

#include <atomic>

#include "internal.h"

namespace nf {
namespace {

constexpr size_t kNoAllocScratchBytes = NF_LAYERNORM_BWD_NOALLOC_SCRATCH_BYTES;  // 16 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

nf_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NF_ERR_CUDA;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        void* q = nullptr;
        if (cudaGetSymbolAddress(&q, g_noalloc_scratch) != cudaSuccess || !q) return NF_ERR_CUDA;
        g_scratch_addr[dev].store(q, std::memory_order_release);
        p = q;
    }
    *out = p;
    return NF_OK;
}

}  // namespace
}  // namespace nf

extern "C" {

nf_status nf_layernorm_bwd_noalloc(void* dx, float* dgamma, float* dbeta, const void* dy,
                                   const void* x, const float* mean, const float* rstd,
                                   const void* gamma, int64_t rows, int64_t hidden,
                                   nf_stream stream) {
    // Stage 1 writes every partial slot it uses before stage 2 reads it, so
    // the area needs no clearing between calls.
    return nf::layernorm_bwd_impl(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows, hidden,
                                  nullptr, nf::kNoAllocScratchBytes, nf::scratch_address, stream);
}

}  // extern "C"
