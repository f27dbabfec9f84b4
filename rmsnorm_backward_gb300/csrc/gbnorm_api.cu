// gbnorm_api.cu -- the extern "C" entry points of libgbnorm.so declared in
// include/gbnorm.h: argument checks, choice of kernel and launch shape, and
// the workspace contract of the deterministic dgamma / dbeta reduction.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "bwd_ws_layout.h"
#include "gbn_launch.h"
#include "gbnorm.h"

namespace gbn {
namespace {

constexpr int kMaxDevices = 64;

struct DevInfo {
    int sms = 0;
    int smem_optin = 0;
    int *err = nullptr;
};

// per-device properties, filled once per device under a lock, then read
// without one once the ready flag is seen
DevInfo g_dev[kMaxDevices];
std::atomic<int> g_dev_ready[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DevInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GBN_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return GBN_ECUDA;
    if (!g_dev_ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        if (g_dev_ready[dev].load(std::memory_order_relaxed)) {
            *out = g_dev[dev];
            return GBN_OK;
        }
        DevInfo d;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            error_flag_address(&d.err) != cudaSuccess) {
            cudaGetLastError();
            return GBN_ECUDA;
        }
        g_dev[dev] = d;
        g_dev_ready[dev].store(1, std::memory_order_release);
    }
    *out = g_dev[dev];
    return GBN_OK;
}

int elem_bytes(int dtype) { return dtype == GBN_F32 ? 4 : 2; }

bool valid_dtype(int dtype) { return dtype == GBN_F32 || dtype == GBN_F16 || dtype == GBN_BF16; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Number of row blocks (CTAs) G: one per SM, more only when a block would
// exceed kMaxRowsPerCta rows.  It depends on (M, SM count) only, so the
// workspace size and the column reduce's order do not depend on buffer
// alignment or on the kernel that takes the rows.
int grid_rows(int64_t M, const DevInfo &d) {
    if (M <= 0) return 0;
    int64_t G = d.sms;
    if (G > M) G = M;
    const int64_t min_g = (M + kMaxRowsPerCta - 1) / kMaxRowsPerCta;
    if (G < min_g) G = min_g;
    return static_cast<int>(G);
}

int partial_ld(int64_t N) { return static_cast<int>((N + 3) / 4 * 4); }

struct StagedPlan {
    bool ok = false;
    bool full = false;  // nv * tpr vectors exactly cover the row
    int tpr = 0, nv = 0, stages = 0, stat_rows = 0;
    size_t smem = 0;
};

// Launch shape of the bulk-copy staged kernels for rows of N elements, if
// the row divides into 16-byte vectors and enough stages fit in shared memory.
StagedPlan staged_plan(bool bwd, bool ln, int dtype, int64_t M, int64_t N, int G, const DevInfo &d) {
    StagedPlan P;
    const int es = elem_bytes(dtype);
    const int V = 16 / es;
    if (N % V != 0) return P;
    const int64_t nvec = N / V;
    // Slot width W warps: the smallest W whose threads cover the row within
    // a cap on the vectors a thread owns, trying the caps in order.
    // Backward: 16 elements (xhat, dyhat held in registers), then for
    // RMSNorm 32 (raw x and dyhat held), then kMaxVecPerThread vectors
    // (re-read).  Forward: kMaxVecPerThread vectors (more rows in flight per
    // CTA measured faster than fewer elements per thread).
    int caps[3] = {kMaxVecPerThread, kMaxVecPerThread, kMaxVecPerThread};
    if (bwd) {
        caps[0] = 16 / V < kMaxVecPerThread ? 16 / V : kMaxVecPerThread;
        caps[1] = !ln && 32 / V < kMaxVecPerThread ? 32 / V : kMaxVecPerThread;
    }
    int W = 0;
    for (int pass = 0; pass < 3 && !W; ++pass) {
        for (int w = 1; w <= kRingThreads / 32; w *= 2) {
            if ((int64_t)32 * w * caps[pass] >= nvec) {
                W = w;
                break;
            }
        }
    }
    if (!W) return P;
    P.tpr = 32 * W;
    P.nv = static_cast<int>((nvec + P.tpr - 1) / P.tpr);
    // exact tiling drops the bounds checks, except in the x-holding backward
    // mode, where the unchecked variant measured slower (register spills)
    P.full = (int64_t)P.nv * P.tpr == nvec && !(bwd && bwd_hold_mode(ln, P.nv * V) == kHoldX && P.nv * V > 16);
    P.stat_rows = static_cast<int>((M + G - 1) / G);
    const int slots = kRingThreads / P.tpr;
    // as many stages as fit, at most 16 per slot
    for (int S = 16; S >= 2; --S) {
        const RingLayout L = ring_layout(bwd, ln, es, static_cast<int>(N), P.tpr, S, P.stat_rows, kRingThreads,
                                         bwd && bwd_gamma_smem(ln, P.nv * V));
        if (L.total <= static_cast<size_t>(d.smem_optin)) {
            P.stages = S;
            P.smem = L.total;
            P.ok = true;
            break;
        }
    }
    (void)slots;
    return P;
}

// Workspace: from its first 256-byte boundary, the [G, ldp] partial rows
// (twice for LayerNorm).
size_t workspace_bytes(int64_t M, int64_t N, bool ln, const DevInfo &d) {
    const int G = grid_rows(M, d);
    return (size_t)G * partial_ld(N) * 4 * (ln ? 2 : 1) + 256;
}

float *workspace_partials(void *ws) {
    const uintptr_t p = (reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255);
    return reinterpret_cast<float *>(p);
}

int check_shape(int64_t M, int64_t N, int dtype) {
    if (!valid_dtype(dtype)) return GBN_EDTYPE;
    if (M < 0 || N < 1 || N > GBN_MAX_N) return GBN_EINVAL;
    if (M > (int64_t(1) << 40)) return GBN_EINVAL;
    return GBN_OK;
}

// gbn_options resolved: strides in elements, accumulate, dgamma/dbeta dtype,
// kernel choice, host-buffer chunk, wait limit
struct Opts {
    int64_t ld_x = 0, ld_dy = 0, ld_out = 0;
    bool accumulate = false;
    int grad_dtype = GBN_F32;
    int reduce_mode = GBN_REDUCE_PARTIALS;
    int kernel = GBN_KERNEL_AUTO;
    int64_t host_chunk = 0;
    uint64_t wait_ns = kWaitNs;
};

// fields every call reads: the kernel choice and the wait limit
int resolve_common(const gbn_options *o, Opts *r) {
    if (!o) return GBN_OK;
    if (o->kernel < GBN_KERNEL_AUTO || o->kernel > GBN_KERNEL_PLAIN || o->wait_limit_ns < 0) return GBN_EINVAL;
    r->kernel = o->kernel;
    if (o->wait_limit_ns > 0) r->wait_ns = static_cast<uint64_t>(o->wait_limit_ns);
    return GBN_OK;
}

// the device-buffer calls: everything but host_chunk
int resolve_options(const gbn_options *o, int64_t N, int dtype, Opts *r) {
    int st = resolve_common(o, r);
    if (st != GBN_OK) return st;
    if (o && o->host_chunk != 0) return GBN_EINVAL;
    r->ld_x = o && o->ld_x ? o->ld_x : N;
    r->ld_dy = o && o->ld_dy ? o->ld_dy : N;
    r->ld_out = o && o->ld_out ? o->ld_out : N;
    if (r->ld_x < N || r->ld_dy < N || r->ld_out < N) return GBN_EINVAL;
    if (o && o->accumulate != 0 && o->accumulate != 1) return GBN_EINVAL;
    r->accumulate = o && o->accumulate == 1;
    r->grad_dtype = o ? o->grad_dtype : GBN_F32;
    if (r->grad_dtype != GBN_F32 && r->grad_dtype != dtype) return GBN_EDTYPE;
    r->reduce_mode = o ? o->reduce_mode : GBN_REDUCE_PARTIALS;
    if (r->reduce_mode < GBN_REDUCE_PARTIALS || r->reduce_mode > GBN_REDUCE_COLWALK) return GBN_EINVAL;
    if (r->reduce_mode != GBN_REDUCE_PARTIALS && r->grad_dtype != GBN_F32) return GBN_EDTYPE;
    return GBN_OK;
}

// the host-buffer calls: host_chunk, kernel and the wait limit only
int resolve_host_options(const gbn_options *o, Opts *r) {
    int st = resolve_common(o, r);
    if (st != GBN_OK) return st;
    if (!o) return GBN_OK;
    if (o->ld_x || o->ld_dy || o->ld_out || o->accumulate || o->grad_dtype || o->reduce_mode || o->host_chunk < 0)
        return GBN_EINVAL;
    r->host_chunk = o->host_chunk;
    return GBN_OK;
}

// rows starting on 16-byte boundaries, given a 16-byte aligned base
bool stride16(int64_t ld, int dtype) { return (ld * elem_bytes(dtype)) % 16 == 0; }

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GBN_OK;
    cudaGetLastError();
    return GBN_ECUDA;
}

int fwd_impl(bool ln, const void *x, const void *gamma, const void *beta, void *y, float *mean, float *rstd,
             float eps, int64_t M, int64_t N, int dtype, const Opts &o, cudaStream_t stream) {
    int st = check_shape(M, N, dtype);
    if (st != GBN_OK) return st;
    if (!(eps >= 0.f) || !isfinite(eps)) return GBN_EINVAL;
    if (M == 0) return GBN_OK;
    if (!x || !gamma || !y || !rstd || (ln && (!beta || !mean))) return GBN_EINVAL;
    DevInfo d;
    if ((st = device_info(&d)) != GBN_OK) return st;
    FwdParams p{};
    p.x = x; p.gamma = gamma; p.beta = beta; p.y = y; p.mean = mean; p.rstd = rstd; p.eps = eps;
    p.M = M; p.N = static_cast<int>(N); p.G = grid_rows(M, d); p.err = d.err;
    p.ld_x = o.ld_x; p.ld_y = o.ld_out;
    const bool aligned = aligned16(x) && aligned16(y) && aligned16(gamma) && (!ln || aligned16(beta)) &&
                         stride16(o.ld_x, dtype) && stride16(o.ld_out, dtype);
    StagedPlan P;
    if (aligned && o.kernel != GBN_KERNEL_PLAIN) P = staged_plan(false, ln, dtype, M, N, p.G, d);
    if (P.ok) {
        p.tpr = P.tpr; p.stages = P.stages; p.stat_rows = P.stat_rows;
        return cuda_status(launch_fwd_staged(dtype, ln, P.nv, P.full, p, P.smem, stream));
    }
    return cuda_status(launch_fwd_plain(dtype, ln, p, stream));
}

// The warp-specialised backward's launch: rows of 16 output warps x 32
// lanes x 1-2 vectors, where it measured faster (shorter rows leave too few
// output warps; at 4 vectors a lane the slot kernel was faster), and >= 2
// stages.  stat_rows: the saved statistics it stages per CTA (0 when none
// were saved).
struct WsPlan {
    bool ok = false;
    int vo = 0, stages = 0, stat_rows = 0;
    size_t smem = 0;
};

WsPlan ws_plan(bool ln, int dtype, int64_t N, int stat_rows, const DevInfo &d) {
    WsPlan w;
    const int V = 16 / elem_bytes(dtype);
    int vo = 0;
    if (N % V != 0 || !ws_shape(static_cast<int>(N / V), &vo)) return w;
    const size_t rowb = (size_t)N * elem_bytes(dtype);
    for (int S = 16; S >= 2; --S) {
        const WsLayout L = ws_layout(ln, rowb, S, stat_rows);
        if (L.total <= static_cast<size_t>(d.smem_optin)) {
            w.ok = true;
            w.vo = vo;
            w.stages = S;
            w.stat_rows = stat_rows;
            w.smem = L.total;
            break;
        }
    }
    return w;
}

// the statistics rows one CTA stages: ceil(M / G)
int stat_rows_of(int64_t M, int G) { return G > 0 ? static_cast<int>((M + G - 1) / G) : 0; }

// Slices of the column reduce's CTAs: 8 (256 threads) where the
// warp-specialised kernel takes the shape, so that they fit on an SM beside
// it and start as soon as its grid completes; 16 (512 threads) beside the
// other kernels, which leave no room for them.  A function of the shape and
// the device only (not of alignment or options), so every call that reduces
// the same [G, N] partial rows sums them in the same order.
bool colsum_small(int dtype, int64_t N, const DevInfo &d) {
    const int V = 16 / elem_bytes(dtype);
    int vo = 0;
    return N % V == 0 && ws_shape(static_cast<int>(N / V), &vo);
}

// recompute_eps >= 0: no saved statistics (mean / rstd null), the kernels
// form them from x with this eps; < 0: the statistics are required.
int bwd_rows_impl(bool ln, const void *dy, const void *x, const void *gamma, const float *mean, const float *rstd,
                  void *dx, int64_t M, int64_t N, int dtype, void *workspace, size_t workspace_bytes_given,
                  const Opts &o, cudaStream_t stream, float recompute_eps = -1.f, float *dgamma = nullptr,
                  float *dbeta = nullptr, float *part_g = nullptr, float *part_b = nullptr) {
    int st = check_shape(M, N, dtype);
    if (st != GBN_OK) return st;
    if (M == 0) return GBN_OK;
    const bool recompute = recompute_eps >= 0.f;
    // part_g given (the host-buffer pipeline): the partial rows go there and
    // to part_b, not into a workspace
    if (!dy || !x || !gamma || !dx || (!workspace && !part_g)) return GBN_EINVAL;
    if (recompute ? (rstd || mean) : (!rstd || (ln && !mean))) return GBN_EINVAL;
    DevInfo d;
    if ((st = device_info(&d)) != GBN_OK) return st;
    if (!part_g && workspace_bytes_given < workspace_bytes(M, N, ln, d)) return GBN_EWORKSPACE;
    BwdParams p{};
    p.dy = dy; p.x = x; p.gamma = gamma; p.mean = mean; p.rstd = rstd; p.dx = dx;
    p.part = part_g ? part_g : workspace_partials(workspace);
    p.part_b = part_b;
    p.M = M; p.N = static_cast<int>(N); p.ldp = partial_ld(N); p.G = grid_rows(M, d); p.err = d.err;
    p.wait_ns = o.wait_ns;
    p.ld_x = o.ld_x; p.ld_dy = o.ld_dy; p.ld_dx = o.ld_out;
    p.eps = recompute ? recompute_eps : 0.f;
    if (o.reduce_mode == GBN_REDUCE_ATOMIC) {  // the caller zeroed them, unless accumulating
        p.atom_g = dgamma;
        p.atom_b = ln ? dbeta : nullptr;
    }
    const bool aligned = aligned16(x) && aligned16(dy) && aligned16(dx) && aligned16(gamma) &&
                         stride16(o.ld_x, dtype) && stride16(o.ld_dy, dtype) && stride16(o.ld_out, dtype);
    // the warp-specialised kernel (every reduce mode, so dx does not depend on it)
    bool launched = false;
    if (aligned && o.kernel == GBN_KERNEL_AUTO) {
        const WsPlan w = ws_plan(ln, dtype, N, recompute ? 0 : stat_rows_of(M, p.G), d);
        if (w.ok) {
            p.stages = w.stages;
            p.stat_rows = w.stat_rows;
            st = cuda_status(launch_bwd_ws(dtype, ln, w.vo, p, w.smem, stream));
            launched = true;
        }
    }
    if (!launched) {
        StagedPlan P;
        if (aligned && o.kernel != GBN_KERNEL_PLAIN) P = staged_plan(true, ln, dtype, M, N, p.G, d);
        if (P.ok) {
            p.tpr = P.tpr; p.stages = P.stages; p.stat_rows = P.stat_rows;
            st = cuda_status(launch_bwd_staged(dtype, ln, P.nv, P.full, p, P.smem, stream));
        } else {
            st = cuda_status(launch_bwd_plain(dtype, ln, p, stream));
        }
    }
    if (st == GBN_OK && o.reduce_mode == GBN_REDUCE_COLWALK)
        st = cuda_status(launch_colwalk(dtype, ln, p, dgamma, ln ? dbeta : nullptr, o.accumulate, stream));
    return st;
}

// The column reduce of the partial rows in the workspace.  Its order is a
// function of (M, N, dtype, device) only, whichever rows kernel ran.
int reduce_impl(const void *workspace, size_t workspace_bytes_given, int64_t M, int64_t N, int dtype, bool ln,
                void *dgamma, void *dbeta, const Opts &o, cudaStream_t stream) {
    int st = check_shape(M, N, dtype);
    if (st != GBN_OK) return st;
    if (!dgamma || (ln && !dbeta)) return GBN_EINVAL;
    if (M == 0) {
        if (o.accumulate) return GBN_OK;  // nothing to add
        const size_t bytes = (size_t)N * elem_bytes(o.grad_dtype);  // all-zero bits are 0.0 in every dtype
        st = cuda_status(cudaMemsetAsync(dgamma, 0, bytes, stream));
        if (st == GBN_OK && ln) st = cuda_status(cudaMemsetAsync(dbeta, 0, bytes, stream));
        return st;
    }
    if (!workspace) return GBN_EINVAL;
    DevInfo d;
    if ((st = device_info(&d)) != GBN_OK) return st;
    if (workspace_bytes_given < workspace_bytes(M, N, ln, d)) return GBN_EWORKSPACE;
    const int G = grid_rows(M, d);
    return cuda_status(launch_colsum(workspace_partials(const_cast<void *>(workspace)), G, partial_ld(N),
                                     static_cast<int>(N), dgamma, ln ? dbeta : nullptr, o.grad_dtype,
                                     o.accumulate, colsum_small(dtype, N, d), d.sms, stream));
}

// ---------------------------------------------------------------------------
// Backward from host buffers: the rows are cut into chunks of R rows, about
// kHostChunkBytes per input (each copy costs a few microseconds besides its
// bytes, so chunks are large), after a ramp of R/8, R/4, R/2 rows that
// starts the pipeline sooner; chunk i's x and dy are copied in on one
// internal stream while chunk i-1's backward kernel runs on the caller's
// stream and chunk i-2's dx is copied out on another, through kHostBufs
// device buffers per tensor (three: two leave the copies no slack).  gamma
// and all the statistics are copied in once, first.  Every chunk writes its
// partial rows at its own offset of one [sum of the chunks' G, ldp] block,
// and one column reduce over the block (fixed order) gives dgamma / dbeta,
// copied out last.
// ---------------------------------------------------------------------------
constexpr size_t kHostChunkBytes = size_t(16) << 20;
constexpr int kHostBufs = 3;

struct HostPlan {
    int64_t R = 0, nchunks = 0, Gtot = 0;
    size_t gam, st, x[kHostBufs], dy[kHostBufs], dx[kHostBufs], grad, part, total;
};

// rows of chunk i: R0 * 2^i, capped at R (the ramp), the last chunk what is left
int64_t host_chunk_rows(int64_t R, int64_t i) {
    const int64_t r0 = R / 8 > 0 ? R / 8 : 1;
    return i >= 4 || (r0 << i) >= R ? R : r0 << i;
}

// chunk_rows: rows per chunk after the ramp, 0 for about kHostChunkBytes of
// each input
HostPlan host_plan(int64_t M, int64_t N, int dtype, bool ln, int64_t chunk_rows, const DevInfo &d) {
    HostPlan h;
    const size_t rowb = (size_t)N * elem_bytes(dtype);
    int64_t R = chunk_rows > 0 ? chunk_rows : (int64_t)(kHostChunkBytes / rowb);
    if (R < 1) R = 1;
    if (R > M) R = M;
    h.R = R;
    for (int64_t r0 = 0; r0 < M; ++h.nchunks) {
        const int64_t want = host_chunk_rows(R, h.nchunks);
        const int64_t rows = M - r0 < want ? M - r0 : want;
        h.Gtot += grid_rows(rows, d);
        r0 += rows;
    }
    const int nst = ln ? 2 : 1;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, 256);
        return at;
    };
    h.gam = take((size_t)N * elem_bytes(dtype));
    h.st = take((size_t)M * 4 * nst);  // rstd [M], then mean [M]
    for (int b = 0; b < kHostBufs; ++b) {
        h.x[b] = take((size_t)R * rowb);
        h.dy[b] = take((size_t)R * rowb);
        h.dx[b] = take((size_t)R * rowb);
    }
    h.grad = take((size_t)N * 4 * nst);
    h.part = take((size_t)h.Gtot * partial_ld(N) * 4 * nst);
    h.total = off + 256;  // the base is aligned up to 256 bytes inside the buffer
    return h;
}

// two internal streams per device (copies in, copies out), created on first use
struct HostStreams {
    cudaStream_t in = nullptr, out = nullptr;
};
HostStreams g_host_streams[kMaxDevices];
std::mutex g_host_streams_mu;

// After a failed enqueue part-way through a host-buffer call: the caller's
// stream still waits for everything the internal streams were given, so the
// caller may reuse or free its buffers in stream order.  Best effort: errors
// here are dropped, the call already reports its own.
void join_internal_streams(const HostStreams &hs, cudaEvent_t e_in, cudaEvent_t e_out, cudaStream_t s) {
    if (cudaEventRecord(e_in, hs.in) == cudaSuccess) cudaStreamWaitEvent(s, e_in, 0);
    if (cudaEventRecord(e_out, hs.out) == cudaSuccess) cudaStreamWaitEvent(s, e_out, 0);
    cudaGetLastError();
}

int host_streams(HostStreams *hs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GBN_ECUDA;
    std::lock_guard<std::mutex> lock(g_host_streams_mu);
    HostStreams &h = g_host_streams[dev];
    if (!h.in) {
        cudaStream_t a = nullptr, b = nullptr;
        if (cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking) != cudaSuccess) {
            if (a) cudaStreamDestroy(a);
            cudaGetLastError();
            return GBN_ECUDA;
        }
        h.in = a;
        h.out = b;
    }
    *hs = h;
    return GBN_OK;
}

int bwd_host_impl(bool ln, const void *dy, const void *x, const void *gamma, const float *mean, const float *rstd,
                  void *dx, float *dgamma, float *dbeta, int64_t M, int64_t N, int dtype, void *workspace,
                  size_t workspace_bytes_given, const Opts &ho, cudaStream_t s) {
    int st = check_shape(M, N, dtype);
    if (st != GBN_OK) return st;
    if (!dgamma || (ln && !dbeta)) return GBN_EINVAL;
    if (M == 0) {  // nothing is enqueued: the host outputs are written now
        memset(dgamma, 0, (size_t)N * 4);
        if (ln) memset(dbeta, 0, (size_t)N * 4);
        return GBN_OK;
    }
    if (!dy || !x || !gamma || !rstd || (ln && !mean) || !dx || !workspace) return GBN_EINVAL;
    DevInfo d;
    if ((st = device_info(&d)) != GBN_OK) return st;
    const HostPlan h = host_plan(M, N, dtype, ln, ho.host_chunk, d);
    if (workspace_bytes_given < h.total) return GBN_EWORKSPACE;
    HostStreams hs;
    if ((st = host_streams(&hs)) != GBN_OK) return st;
    unsigned char *base = reinterpret_cast<unsigned char *>(workspace_partials(workspace));
    const size_t es = elem_bytes(dtype), rowb = (size_t)N * es;
    const int ldp = partial_ld(N);
    float *grad = reinterpret_cast<float *>(base + h.grad);
    float *part = reinterpret_cast<float *>(base + h.part);

    constexpr int B = kHostBufs;
    cudaEvent_t ev[2 + 3 * B] = {};
    for (auto &e : ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            for (auto &f : ev)
                if (f) cudaEventDestroy(f);
            cudaGetLastError();
            return GBN_ECUDA;
        }
    cudaEvent_t start = ev[0], dx_out = ev[1];
    cudaEvent_t *loaded = ev + 2, *computed = ev + 2 + B, *unloaded = ev + 2 + 2 * B;
    const auto chk = [](cudaError_t e) { return e == cudaSuccess; };
    float *st_r = reinterpret_cast<float *>(base + h.st);
    float *st_m = st_r + M;
    bool ok = chk(cudaEventRecord(start, s)) && chk(cudaStreamWaitEvent(hs.in, start, 0)) &&
              chk(cudaStreamWaitEvent(hs.out, start, 0)) &&
              chk(cudaMemcpyAsync(base + h.gam, gamma, rowb, cudaMemcpyHostToDevice, hs.in)) &&
              chk(cudaMemcpyAsync(st_r, rstd, (size_t)M * 4, cudaMemcpyHostToDevice, hs.in)) &&
              (!ln || chk(cudaMemcpyAsync(st_m, mean, (size_t)M * 4, cudaMemcpyHostToDevice, hs.in)));
    Opts o = ho;
    o.ld_x = o.ld_dy = o.ld_out = N;
    int64_t goff = 0, r0 = 0;
    for (int64_t i = 0; ok && i < h.nchunks; r0 += host_chunk_rows(h.R, i), ++i) {
        const int b = static_cast<int>(i % B);
        const int64_t want = host_chunk_rows(h.R, i), rows = M - r0 < want ? M - r0 : want;
        // in: the buffers are free once chunk i-B's kernel has read them
        ok = (i < B || chk(cudaStreamWaitEvent(hs.in, computed[b], 0))) &&
             chk(cudaMemcpyAsync(base + h.x[b], static_cast<const unsigned char *>(x) + r0 * rowb, rows * rowb,
                                 cudaMemcpyHostToDevice, hs.in)) &&
             chk(cudaMemcpyAsync(base + h.dy[b], static_cast<const unsigned char *>(dy) + r0 * rowb, rows * rowb,
                                 cudaMemcpyHostToDevice, hs.in)) &&
             chk(cudaEventRecord(loaded[b], hs.in));
        // compute: dx's buffer is free once chunk i-B's dx has been copied out
        ok = ok && chk(cudaStreamWaitEvent(s, loaded[b], 0)) &&
             (i < B || chk(cudaStreamWaitEvent(s, unloaded[b], 0)));
        if (ok) {
            const int G = grid_rows(rows, d);
            st = bwd_rows_impl(ln, base + h.dy[b], base + h.x[b], base + h.gam, ln ? st_m + r0 : nullptr, st_r + r0,
                               base + h.dx[b], rows, N, dtype, nullptr, 0, o, s, -1.f, nullptr, nullptr,
                               part + (size_t)goff * ldp, ln ? part + (size_t)(h.Gtot + goff) * ldp : nullptr);
            goff += G;
            ok = st == GBN_OK && chk(cudaEventRecord(computed[b], s));
        }
        // out
        ok = ok && chk(cudaStreamWaitEvent(hs.out, computed[b], 0)) &&
             chk(cudaMemcpyAsync(static_cast<unsigned char *>(dx) + r0 * rowb, base + h.dx[b], rows * rowb,
                                 cudaMemcpyDeviceToHost, hs.out)) &&
             chk(cudaEventRecord(unloaded[b], hs.out));
    }
    if (ok) {
        ok = chk(launch_colsum(part, static_cast<int>(h.Gtot), ldp, static_cast<int>(N), grad,
                               ln ? grad + N : nullptr, GBN_F32, false, colsum_small(dtype, N, d), d.sms, s)) &&
             chk(cudaMemcpyAsync(dgamma, grad, (size_t)N * 4, cudaMemcpyDeviceToHost, s)) &&
             (!ln || chk(cudaMemcpyAsync(dbeta, grad + N, (size_t)N * 4, cudaMemcpyDeviceToHost, s))) &&
             chk(cudaEventRecord(dx_out, hs.out)) && chk(cudaStreamWaitEvent(s, dx_out, 0));
    }
    if (!ok) join_internal_streams(hs, start, dx_out, s);
    for (auto &e : ev) cudaEventDestroy(e);  // released once the work recorded on them is done
    if (!ok) {
        cudaGetLastError();
        return st != GBN_OK ? st : GBN_ECUDA;
    }
    return GBN_OK;
}

// Activation backward from host buffers: the same pipeline as the norm's
// (copies in on one internal stream, the kernel on the caller's stream,
// copies out on the other, three device buffers per tensor), over chunks of
// elements: about kHostChunkBytes of each tensor after the same ramp.
struct ActHostPlan {
    int64_t R = 0, nchunks = 0;
    size_t dy[kHostBufs], pre[kHostBufs], dx[kHostBufs], total = 0;
};

// chunk: elements per chunk after the ramp, 0 for about kHostChunkBytes of
// each tensor
ActHostPlan act_host_plan(int64_t n, int dtype, int64_t chunk) {
    ActHostPlan h;
    const size_t es = elem_bytes(dtype);
    int64_t R = chunk > 0 ? chunk : (int64_t)(kHostChunkBytes / es);
    if (R > n) R = n;
    if (R < 1) R = 1;
    h.R = R;
    for (int64_t e0 = 0; e0 < n; ++h.nchunks) e0 += host_chunk_rows(R, h.nchunks);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, 256);
        return at;
    };
    for (int b = 0; b < kHostBufs; ++b) {
        h.dy[b] = take((size_t)R * es);
        h.pre[b] = take((size_t)R * es);
        h.dx[b] = take((size_t)R * es);
    }
    h.total = off + 256;
    return h;
}

int act_host_impl(int act, const void *dy, const void *preact, void *dx, int64_t n, int dtype, void *workspace,
                  size_t workspace_bytes_given, const Opts &ho, cudaStream_t s) {
    if (!valid_dtype(dtype)) return GBN_EDTYPE;
    if (n < 0) return GBN_EINVAL;
    if (n == 0) return GBN_OK;
    if (!dy || !preact || !dx || !workspace) return GBN_EINVAL;
    DevInfo d;
    int st = device_info(&d);
    if (st != GBN_OK) return st;
    const ActHostPlan h = act_host_plan(n, dtype, ho.host_chunk);
    if (workspace_bytes_given < h.total) return GBN_EWORKSPACE;
    HostStreams hs;
    if ((st = host_streams(&hs)) != GBN_OK) return st;
    unsigned char *base = reinterpret_cast<unsigned char *>(workspace_partials(workspace));
    const size_t es = elem_bytes(dtype);
    constexpr int B = kHostBufs;
    cudaEvent_t ev[2 + 3 * B] = {};
    for (auto &e : ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            for (auto &f : ev)
                if (f) cudaEventDestroy(f);
            cudaGetLastError();
            return GBN_ECUDA;
        }
    cudaEvent_t start = ev[0], out_done = ev[1];
    cudaEvent_t *loaded = ev + 2, *computed = ev + 2 + B, *unloaded = ev + 2 + 2 * B;
    const auto chk = [](cudaError_t e) { return e == cudaSuccess; };
    bool ok = chk(cudaEventRecord(start, s)) && chk(cudaStreamWaitEvent(hs.in, start, 0)) &&
              chk(cudaStreamWaitEvent(hs.out, start, 0));
    int64_t e0 = 0;
    for (int64_t i = 0; ok && i < h.nchunks; e0 += host_chunk_rows(h.R, i), ++i) {
        const int b = static_cast<int>(i % B);
        const int64_t want = host_chunk_rows(h.R, i), cnt = n - e0 < want ? n - e0 : want;
        const size_t off = (size_t)e0 * es, bytes = (size_t)cnt * es;
        ok = (i < B || chk(cudaStreamWaitEvent(hs.in, computed[b], 0))) &&
             chk(cudaMemcpyAsync(base + h.dy[b], static_cast<const unsigned char *>(dy) + off, bytes,
                                 cudaMemcpyHostToDevice, hs.in)) &&
             chk(cudaMemcpyAsync(base + h.pre[b], static_cast<const unsigned char *>(preact) + off, bytes,
                                 cudaMemcpyHostToDevice, hs.in)) &&
             chk(cudaEventRecord(loaded[b], hs.in)) && chk(cudaStreamWaitEvent(s, loaded[b], 0)) &&
             (i < B || chk(cudaStreamWaitEvent(s, unloaded[b], 0))) &&
             chk(launch_act_bwd(act, dtype, base + h.dy[b], base + h.pre[b], base + h.dx[b], cnt, d.sms, d.err, s)) &&
             chk(cudaEventRecord(computed[b], s)) && chk(cudaStreamWaitEvent(hs.out, computed[b], 0)) &&
             chk(cudaMemcpyAsync(static_cast<unsigned char *>(dx) + off, base + h.dx[b], bytes,
                                 cudaMemcpyDeviceToHost, hs.out)) &&
             chk(cudaEventRecord(unloaded[b], hs.out));
    }
    ok = ok && chk(cudaEventRecord(out_done, hs.out)) && chk(cudaStreamWaitEvent(s, out_done, 0));
    if (!ok) join_internal_streams(hs, start, out_done, s);
    for (auto &e : ev) cudaEventDestroy(e);  // released once the work recorded on them is done
    if (!ok) {
        cudaGetLastError();
        return GBN_ECUDA;
    }
    return GBN_OK;
}

}  // namespace
}  // namespace gbn

using namespace gbn;

extern "C" {

size_t gbn_bwd_workspace_bytes(int64_t M, int64_t N, int dtype, int has_beta) {
    if (check_shape(M, N, dtype) != GBN_OK || M <= 0) return 0;
    DevInfo d;
    if (device_info(&d) != GBN_OK) return 0;
    return workspace_bytes(M, N, has_beta != 0, d);
}

int ln_fwd_ex(const void *x, const void *gamma, const void *beta, void *y, float *mean, float *rstd, float eps,
              int64_t M, int64_t N, int dtype, const gbn_options *opt, cudaStream_t stream) {
    Opts o;
    int st = check_shape(M, N, dtype);
    if (st == GBN_OK) st = resolve_options(opt, N, dtype, &o);
    if (st != GBN_OK) return st;
    return fwd_impl(true, x, gamma, beta, y, mean, rstd, eps, M, N, dtype, o, stream);
}

int rms_fwd_ex(const void *x, const void *gamma, void *y, float *rstd, float eps, int64_t M, int64_t N, int dtype,
               const gbn_options *opt, cudaStream_t stream) {
    Opts o;
    int st = check_shape(M, N, dtype);
    if (st == GBN_OK) st = resolve_options(opt, N, dtype, &o);
    if (st != GBN_OK) return st;
    return fwd_impl(false, x, gamma, nullptr, y, nullptr, rstd, eps, M, N, dtype, o, stream);
}

int ln_fwd(const void *x, const void *gamma, const void *beta, void *y, float *mean, float *rstd, float eps,
           int64_t M, int64_t N, int dtype, cudaStream_t stream) {
    return ln_fwd_ex(x, gamma, beta, y, mean, rstd, eps, M, N, dtype, nullptr, stream);
}

int rms_fwd(const void *x, const void *gamma, void *y, float *rstd, float eps, int64_t M, int64_t N, int dtype,
            cudaStream_t stream) {
    return rms_fwd_ex(x, gamma, y, rstd, eps, M, N, dtype, nullptr, stream);
}

int ln_bwd_rows(const void *dy, const void *x, const void *gamma, const float *mean, const float *rstd, void *dx,
                int64_t M, int64_t N, int dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    Opts o;
    o.ld_x = o.ld_dy = o.ld_out = N;
    return bwd_rows_impl(true, dy, x, gamma, mean, rstd, dx, M, N, dtype, workspace, workspace_bytes, o, stream);
}

int rms_bwd_rows(const void *dy, const void *x, const void *gamma, const float *rstd, void *dx, int64_t M,
                 int64_t N, int dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    Opts o;
    o.ld_x = o.ld_dy = o.ld_out = N;
    return bwd_rows_impl(false, dy, x, gamma, nullptr, rstd, dx, M, N, dtype, workspace, workspace_bytes, o,
                         stream);
}

int gbn_bwd_reduce(const void *workspace, size_t workspace_bytes, int64_t M, int64_t N, int dtype, int has_beta,
                   float *dgamma, float *dbeta, cudaStream_t stream) {
    return reduce_impl(workspace, workspace_bytes, M, N, dtype, has_beta != 0, dgamma, dbeta, Opts(), stream);
}

int ln_bwd_ex(const void *dy, const void *x, const void *gamma, const float *mean, const float *rstd, void *dx,
              void *dgamma, void *dbeta, float eps, int64_t M, int64_t N, int dtype, void *workspace,
              size_t workspace_bytes, const gbn_options *opt, cudaStream_t stream) {
    Opts o;
    int st = check_shape(M, N, dtype);
    if (st == GBN_OK) st = resolve_options(opt, N, dtype, &o);
    if (st != GBN_OK) return st;
    if (M > 0 && (!dgamma || !dbeta)) return GBN_EINVAL;
    // no saved statistics: recompute them from x with eps
    const bool recompute = !mean && !rstd;
    if (recompute && (!(eps >= 0.f) || !isfinite(eps))) return GBN_EINVAL;
    if (recompute && o.reduce_mode == GBN_REDUCE_COLWALK) return GBN_EINVAL;
    if (M > 0 && o.reduce_mode == GBN_REDUCE_ATOMIC && !o.accumulate) {
        st = cuda_status(cudaMemsetAsync(dgamma, 0, (size_t)N * 4, stream));
        if (st == GBN_OK) st = cuda_status(cudaMemsetAsync(dbeta, 0, (size_t)N * 4, stream));
        if (st != GBN_OK) return st;
    }
    st = bwd_rows_impl(true, dy, x, gamma, mean, rstd, dx, M, N, dtype, workspace, workspace_bytes, o, stream,
                       recompute ? eps : -1.f, static_cast<float *>(dgamma), static_cast<float *>(dbeta));
    if (st != GBN_OK || (M > 0 && o.reduce_mode != GBN_REDUCE_PARTIALS)) return st;
    return reduce_impl(workspace, workspace_bytes, M, N, dtype, true, dgamma, dbeta, o, stream);
}

int rms_bwd_ex(const void *dy, const void *x, const void *gamma, const float *rstd, void *dx, void *dgamma,
               float eps, int64_t M, int64_t N, int dtype, void *workspace, size_t workspace_bytes,
               const gbn_options *opt, cudaStream_t stream) {
    Opts o;
    int st = check_shape(M, N, dtype);
    if (st == GBN_OK) st = resolve_options(opt, N, dtype, &o);
    if (st != GBN_OK) return st;
    if (M > 0 && !dgamma) return GBN_EINVAL;
    // no saved rstd: recompute it from x with eps
    const bool recompute = !rstd;
    if (recompute && (!(eps >= 0.f) || !isfinite(eps))) return GBN_EINVAL;
    if (recompute && o.reduce_mode == GBN_REDUCE_COLWALK) return GBN_EINVAL;
    if (M > 0 && o.reduce_mode == GBN_REDUCE_ATOMIC && !o.accumulate) {
        st = cuda_status(cudaMemsetAsync(dgamma, 0, (size_t)N * 4, stream));
        if (st != GBN_OK) return st;
    }
    st = bwd_rows_impl(false, dy, x, gamma, nullptr, rstd, dx, M, N, dtype, workspace, workspace_bytes, o, stream,
                       recompute ? eps : -1.f, static_cast<float *>(dgamma));
    if (st != GBN_OK || (M > 0 && o.reduce_mode != GBN_REDUCE_PARTIALS)) return st;
    return reduce_impl(workspace, workspace_bytes, M, N, dtype, false, dgamma, nullptr, o, stream);
}

int ln_bwd(const void *dy, const void *x, const void *gamma, const float *mean, const float *rstd, void *dx,
           float *dgamma, float *dbeta, float eps, int64_t M, int64_t N, int dtype, void *workspace,
           size_t workspace_bytes, cudaStream_t stream) {
    return ln_bwd_ex(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, eps, M, N, dtype, workspace, workspace_bytes,
                     nullptr, stream);
}

int rms_bwd(const void *dy, const void *x, const void *gamma, const float *rstd, void *dx, float *dgamma, float eps,
            int64_t M, int64_t N, int dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return rms_bwd_ex(dy, x, gamma, rstd, dx, dgamma, eps, M, N, dtype, workspace, workspace_bytes, nullptr,
                      stream);
}

int act_bwd_impl(int act, const void *dy, const void *preact, void *dx, int64_t n, int dtype, cudaStream_t s) {
    if (!valid_dtype(dtype)) return GBN_EDTYPE;
    if (n < 0) return GBN_EINVAL;
    if (n == 0) return GBN_OK;
    if (!dy || !preact || !dx) return GBN_EINVAL;
    DevInfo d;
    int st = device_info(&d);
    if (st != GBN_OK) return st;
    return cuda_status(launch_act_bwd(act, dtype, dy, preact, dx, n, d.sms, d.err, s));
}

int silu_bwd(const void *dy, const void *preact, void *dx, int64_t n, int dtype, cudaStream_t stream) {
    return act_bwd_impl(kActSilu, dy, preact, dx, n, dtype, stream);
}

int gelu_bwd(const void *dy, const void *preact, void *dx, int64_t n, int dtype, cudaStream_t stream) {
    return act_bwd_impl(kActGelu, dy, preact, dx, n, dtype, stream);
}

size_t gbn_bwd_host_workspace_bytes_ex(int64_t M, int64_t N, int dtype, int has_beta, const gbn_options *opt) {
    Opts o;
    if (check_shape(M, N, dtype) != GBN_OK || M <= 0 || resolve_host_options(opt, &o) != GBN_OK) return 0;
    DevInfo d;
    if (device_info(&d) != GBN_OK) return 0;
    return host_plan(M, N, dtype, has_beta != 0, o.host_chunk, d).total;
}

size_t gbn_bwd_host_workspace_bytes(int64_t M, int64_t N, int dtype, int has_beta) {
    return gbn_bwd_host_workspace_bytes_ex(M, N, dtype, has_beta, nullptr);
}

int ln_bwd_host_ex(const void *dy, const void *x, const void *gamma, const float *mean, const float *rstd, void *dx,
                   float *dgamma, float *dbeta, int64_t M, int64_t N, int dtype, void *workspace,
                   size_t workspace_bytes, const gbn_options *opt, cudaStream_t stream) {
    Opts o;
    const int st = resolve_host_options(opt, &o);
    if (st != GBN_OK) return st;
    return bwd_host_impl(true, dy, x, gamma, mean, rstd, dx, dgamma, dbeta, M, N, dtype, workspace,
                         workspace_bytes, o, stream);
}

int rms_bwd_host_ex(const void *dy, const void *x, const void *gamma, const float *rstd, void *dx, float *dgamma,
                    int64_t M, int64_t N, int dtype, void *workspace, size_t workspace_bytes,
                    const gbn_options *opt, cudaStream_t stream) {
    Opts o;
    const int st = resolve_host_options(opt, &o);
    if (st != GBN_OK) return st;
    return bwd_host_impl(false, dy, x, gamma, nullptr, rstd, dx, dgamma, nullptr, M, N, dtype, workspace,
                         workspace_bytes, o, stream);
}

int ln_bwd_host(const void *dy, const void *x, const void *gamma, const float *mean, const float *rstd, void *dx,
                float *dgamma, float *dbeta, int64_t M, int64_t N, int dtype, void *workspace,
                size_t workspace_bytes, cudaStream_t stream) {
    return ln_bwd_host_ex(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, M, N, dtype, workspace, workspace_bytes,
                          nullptr, stream);
}

int rms_bwd_host(const void *dy, const void *x, const void *gamma, const float *rstd, void *dx, float *dgamma,
                 int64_t M, int64_t N, int dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return rms_bwd_host_ex(dy, x, gamma, rstd, dx, dgamma, M, N, dtype, workspace, workspace_bytes, nullptr,
                           stream);
}

size_t gbn_act_host_workspace_bytes_ex(int64_t n, int dtype, const gbn_options *opt) {
    Opts o;
    if (!valid_dtype(dtype) || n <= 0 || resolve_host_options(opt, &o) != GBN_OK) return 0;
    return act_host_plan(n, dtype, o.host_chunk).total;
}

size_t gbn_act_host_workspace_bytes(int64_t n, int dtype) { return gbn_act_host_workspace_bytes_ex(n, dtype, nullptr); }

int silu_bwd_host_ex(const void *dy, const void *preact, void *dx, int64_t n, int dtype, void *workspace,
                     size_t workspace_bytes, const gbn_options *opt, cudaStream_t stream) {
    Opts o;
    const int st = resolve_host_options(opt, &o);
    if (st != GBN_OK) return st;
    return act_host_impl(kActSilu, dy, preact, dx, n, dtype, workspace, workspace_bytes, o, stream);
}

int gelu_bwd_host_ex(const void *dy, const void *preact, void *dx, int64_t n, int dtype, void *workspace,
                     size_t workspace_bytes, const gbn_options *opt, cudaStream_t stream) {
    Opts o;
    const int st = resolve_host_options(opt, &o);
    if (st != GBN_OK) return st;
    return act_host_impl(kActGelu, dy, preact, dx, n, dtype, workspace, workspace_bytes, o, stream);
}

int silu_bwd_host(const void *dy, const void *preact, void *dx, int64_t n, int dtype, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
    return silu_bwd_host_ex(dy, preact, dx, n, dtype, workspace, workspace_bytes, nullptr, stream);
}

int gelu_bwd_host(const void *dy, const void *preact, void *dx, int64_t n, int dtype, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
    return gelu_bwd_host_ex(dy, preact, dx, n, dtype, workspace, workspace_bytes, nullptr, stream);
}

int gbn_bwd_plan(int64_t M, int64_t N, int dtype, int has_beta, int *G, int *staged) {
    int st = check_shape(M, N, dtype);
    if (st != GBN_OK) return st;
    DevInfo d;
    if ((st = device_info(&d)) != GBN_OK) return st;
    const int g = grid_rows(M, d);
    if (G) *G = g;
    if (staged) {
        *staged = 0;
        if (M > 0 && ws_plan(has_beta != 0, dtype, N, stat_rows_of(M, g), d).ok)
            *staged = 2;
        else if (M > 0 && staged_plan(true, has_beta != 0, dtype, M, N, g, d).ok)
            *staged = 1;
    }
    return GBN_OK;
}

int gbn_device_error(int clear) {
    int v = 0;
    if (read_error_flag(&v, clear != 0) != cudaSuccess) {
        cudaGetLastError();
        return -GBN_ECUDA;
    }
    return v;
}

const char *gbn_status_string(int status) {
    switch (status) {
        case GBN_OK: return "ok";
        case GBN_EINVAL: return "invalid argument (null pointer, bad M, N or eps)";
        case GBN_EDTYPE: return "unknown dtype";
        case GBN_EWORKSPACE: return "workspace smaller than gbn_bwd_workspace_bytes()";
        case GBN_ECUDA: return "CUDA launch or query failed";
        case GBN_EDEVICE: return "a kernel gave up on a bounded wait";
        case GBN_ESCRATCH: return "problem needs more workspace than rms_bwd_noalloc's static scratch holds";
    }
    return "unknown status";
}

}  // extern "C"
