// gbn_launch.h -- kernel parameter blocks and the launch functions that the
// C ABI layer (gbnorm_api.cu) calls.  Internal to libgbnorm.so.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <stddef.h>
#include <stdint.h>

namespace gbn {

// threads of the bulk-copy (TMA) staged kernels and of the plain-load ones
constexpr int kRingThreads = 512;
constexpr int kGenericThreads = 256;
// most rows one CTA takes; its rows' statistics are staged in shared memory
constexpr int kMaxRowsPerCta = 2048;
// most 16-byte vectors one thread holds per row in the staged kernels
constexpr int kMaxVecPerThread = 4;
// default limit of a wait on another warp or on a bulk copy, and the limit
// of the wait for a CTA's own copies still in flight before it exits
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 100000000ull;

struct FwdParams {
    const void *x;
    const void *gamma;
    const void *beta;  // LayerNorm only
    void *y;
    float *mean;       // LayerNorm only
    float *rstd;
    float eps;
    int64_t M;
    int N;
    int G;          // CTAs; CTA b takes the rows of block_rows(M, G, b)
    int tpr;        // staged: threads per row slot (multiple of 32)
    int stages;     // staged: ring stages per row slot
    int stat_rows;  // unused by the forward (kept for a uniform layout)
    int *err;       // the device's error flag
    int64_t ld_x;   // row strides, in elements, of x and y
    int64_t ld_y;
};

struct BwdParams {
    const void *dy;
    const void *x;
    const void *gamma;
    const float *mean;  // LayerNorm only; nullptr with rstd: recomputed from x
    const float *rstd;  // nullptr: no saved statistics, recomputed from x with eps
    void *dx;
    float *part;        // [G][ldp] dgamma partials, then [G][ldp] dbeta partials (LayerNorm)
    float *part_b;      // non-null: the [G][ldp] dbeta partials start here instead
    int64_t M;
    int N;
    int ldp;            // row stride of the partials, in floats (multiple of 4)
    int G;
    int tpr;
    int stages;
    int stat_rows;      // capacity, in rows, of the staged statistics
    int *err;           // the device's error flag
    uint64_t wait_ns;   // limit of the waits between warps and on bulk copies
    int64_t ld_x;       // row strides, in elements, of x, dy and dx
    int64_t ld_dy;
    int64_t ld_dx;
    float eps;          // used when no statistics were saved (rstd == nullptr)
    // reduction ablation: non-null, the CTA adds its partial row(s) into
    // these fp32 buffers with atomics instead of storing them in `part`
    float *atom_g;
    float *atom_b;
};

// Shared-memory layout of the staged kernels, computed identically on the
// host (to size the launch) and on the device (to carve the buffer).
struct RingLayout {
    size_t ring_off, ring_bytes;  // [slots][stages][stage_bytes]; reused for the partial combine
    size_t gam_off;               // [N] fp32 gamma (backward kernels that stage it), else empty
    size_t bar_off;               // [slots][stages] mbarriers
    size_t stat_off;              // [stat_rows] rstd, then [stat_rows] mean (LayerNorm)
    size_t red_off;               // [slots][4 buffers][2][kRedStride = 16] floats
    size_t flag_off;              // [slots] ints: per-slot abort flags
    size_t total;
};

__host__ __device__ inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// What the staged backward keeps in registers between its two passes, for a
// thread that owns `elems` elements of a row:
//   kHoldAll: xhat and dyhat in fp32 (up to 16 elements), gamma in registers;
//   kHoldX:   x as raw 16-byte vectors and dyhat in fp32 (RMSNorm, up to 32
//             elements), gamma unpacked once into shared memory;
//   kReread:  nothing; pass 2 re-reads the staged row.
enum BwdHold : int { kHoldAll = 0, kHoldX = 1, kReread = 2 };
__host__ __device__ constexpr int bwd_hold_mode(bool ln, int elems) {
    return elems <= 16 ? kHoldAll : (!ln && elems <= 32 ? kHoldX : kReread);
}
__host__ __device__ constexpr bool bwd_gamma_smem(bool ln, int elems) { return bwd_hold_mode(ln, elems) == kHoldX; }

__host__ __device__ inline RingLayout ring_layout(bool bwd, bool ln, int es, int N, int tpr, int stages,
                                                  int stat_rows, int threads, bool gamma_smem = false) {
    RingLayout L;
    const int slots = threads / tpr;
    const size_t stage_bytes = (bwd ? 2u : 1u) * (size_t)N * es;
    size_t ring = (size_t)slots * stages * stage_bytes;
    if (bwd) {
        const size_t combine = (size_t)slots * round_up((size_t)N, 4) * 4 * (ln ? 2 : 1);
        if (slots > 1 && combine > ring) ring = combine;
    }
    L.ring_off = 0;
    L.ring_bytes = round_up(ring, 128);
    L.gam_off = L.ring_bytes;
    L.bar_off = L.gam_off + (gamma_smem ? round_up((size_t)N * 4, 128) : 0);
    L.stat_off = L.bar_off + round_up((size_t)slots * stages * 8, 16);
    L.red_off = L.stat_off + round_up((size_t)stat_rows * 4 * (ln ? 2 : 1), 16);
    L.flag_off = L.red_off + (size_t)slots * 4 * 2 * 16 * 4;
    L.total = round_up(L.flag_off + (size_t)slots * 4, 128);
    return L;
}

// dtype codes as in gbnorm.h
// full: every thread's NV vectors lie inside the row (no bounds checks)
cudaError_t launch_fwd_staged(int dtype, bool ln, int nv, bool full, const FwdParams &p, size_t smem,
                              cudaStream_t s);
cudaError_t launch_fwd_plain(int dtype, bool ln, const FwdParams &p, cudaStream_t s);
cudaError_t launch_bwd_staged(int dtype, bool ln, int nv, bool full, const BwdParams &p, size_t smem,
                              cudaStream_t s);
cudaError_t launch_bwd_plain(int dtype, bool ln, const BwdParams &p, cudaStream_t s);
// warp-specialised backward (bwd_ws.cuh): vo vectors per output lane
cudaError_t launch_bwd_ws(int dtype, bool ln, int vo, const BwdParams &p, size_t smem, cudaStream_t s);
// dgamma / dbeta from the partial rows; out_dtype is GBN_F32 or the storage
// dtype of the parameters (rounded to nearest even); accumulate adds the
// buffers' previous contents (widened) to the sums before the store; sms:
// the device's SM count (the grid shape, not the order, depends on it)
cudaError_t launch_colsum(const float *part, int G, int ldp, int N, void *dgamma, void *dbeta, int out_dtype,
                          bool accumulate, bool small, int sms, cudaStream_t s);

// reduction ablation: dgamma (dbeta) = sum over rows of dy*xhat (dy), each CTA
// owning 32 columns and walking every row of x and dy in order
cudaError_t launch_colwalk(int dtype, bool ln, const BwdParams &p, float *dgamma, float *dbeta, bool accumulate,
                           cudaStream_t s);

// opts a kernel into the device's full dynamic shared memory, once per device
template <typename K>
cudaError_t ensure_smem_optin(K kernel, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && ((done.load(std::memory_order_acquire) >> dev) & 1u)) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e == cudaSuccess && dev < 64) done.fetch_or(uint64_t(1) << dev, std::memory_order_release);
    return e;
}

// activation backward dx = dy * f'(preact) over n contiguous elements
enum : int { kActSilu = 0, kActGelu = 1 };
struct ActParams {
    const void *dy, *pre;
    void *dx;
    int64_t n;
    int64_t nchunks;  // full chunks of the kernel's shape (0 when a pointer is unaligned)
    int vec_ok;
    int *err;
};
cudaError_t launch_act_bwd(int act, int dtype, const void *dy, const void *pre, void *dx, int64_t n, int sms,
                           int *err, cudaStream_t s);

// the current device's error flag: its device address, and a synchronising read
cudaError_t error_flag_address(int **addr);
cudaError_t read_error_flag(int *value, bool clear);

}  // namespace gbn
