// norm_bwd_noalloc.cu -- rms_bwd_noalloc: the RMSNorm backward for callers
// that cannot allocate device memory.
//
// rms_bwd needs a caller-provided workspace for its per-CTA partial rows.
// Some callers cannot call cudaMalloc (or an allocating library routine) at
// the point where they run the backward: code running inside an allocator's
// own callback, where allocating would re-enter it; engines and plugins that
// work under a device-memory budget fixed up front and get no workspace;
// latency-critical loops that cannot take the implicit device
// synchronisation a cudaMalloc / cudaFree may cause.  For them this entry
// point keeps the workspace in a file-scope static device array instead,
// and allocates nothing.
//
// The array is GBN_NOALLOC_SCRATCH_BYTES (16 MiB).  Every GPU that loads
// this library holds its own copy of it until the process exits.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "gbnorm.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GBN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::atomic<int> g_scratch_ready[kMaxDevices];
std::mutex g_scratch_mu;

// The device address of this device's scratch array.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.  Host threads may
// race on the first call: the cache is filled under a lock, and read
// without one once its ready flag is seen.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GBN_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return GBN_ECUDA;
    if (!g_scratch_ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (g_scratch_ready[dev].load(std::memory_order_relaxed)) {
            *out = g_scratch_ptr[dev];
            return GBN_OK;
        }
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return GBN_ECUDA;
        }
        g_scratch_ptr[dev] = p;
        g_scratch_ready[dev].store(1, std::memory_order_release);
    }
    *out = g_scratch_ptr[dev];
    return GBN_OK;
}

}  // namespace

extern "C" int rms_bwd_noalloc(const void *dy, const void *x, const void *gamma, const float *rstd, void *dx,
                               float *dgamma, float eps, int64_t M, int64_t N, int dtype, cudaStream_t stream) {
    // problems whose partial rows do not fit the array are refused before
    // anything is enqueued (rms_bwd would refuse them too, as a workspace
    // smaller than it needs)
    const size_t need = gbn_bwd_workspace_bytes(M, N, dtype, 0);
    if (need > GBN_NOALLOC_SCRATCH_BYTES) return GBN_ESCRATCH;
    void *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != GBN_OK) return st;
    // every partial element the reduce reads is written by this call's first
    // kernel, so the array needs no clearing between calls
    return rms_bwd(dy, x, gamma, rstd, dx, dgamma, eps, M, N, dtype, scratch, GBN_NOALLOC_SCRATCH_BYTES, stream);
}
