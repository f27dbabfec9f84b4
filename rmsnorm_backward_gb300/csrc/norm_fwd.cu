// norm_fwd.cu -- LayerNorm / RMSNorm forward kernels for sm_103a.
//
// Definition followed: "Norm backward in Triton -- the dγ/dβ reduction",
// section "The gradients" (forward line and RMSNorm paragraph), with the
// variance taken as in "05: Layer norm", kernel ln_fwd: the biased variance of
// the row centred on its mean, computed after the mean (two passes), eps
// under the root.  The forward saves the per-row mean (LayerNorm) and rstd
// for the backward ("Norm & activation backward", section "Half one").
//
// Two kernels:
//  * staged: one persistent CTA per SM.  The CTA's rows are split over
//    "slots" (groups of tpr threads); each slot streams its rows through a
//    ring of shared-memory stages filled by 1-D bulk (TMA) copies that
//    complete on mbarriers.  A thread keeps its 16-byte vectors of the row
//    in registers, so both passes of the two-pass variance read on-chip
//    data and x leaves HBM exactly once.
//  * plain: any N and alignment; a CTA walks a row three times with scalar
//    loads (mean, centred squares, output), the later passes hitting L1/L2.
#include "gbn_device.cuh"
#include "gbn_launch.h"

namespace gbn {

template <typename T, bool LN, int NV, bool HOLD>
__global__ void __launch_bounds__(kRingThreads, 1) fwd_staged_kernel(const FwdParams p) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int E = NV * V;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int tpr = p.tpr;
    const int slots = blockDim.x / tpr;
    const int slot = tid / tpr;
    const int ts = tid - slot * tpr;
    const int W = tpr >> 5;
    const int warp = ts >> 5;
    const int lane = tid & 31;
    const int N = p.N;
    const int nvec = N / V;
    const int S = p.stages;
    const uint32_t rowb = static_cast<uint32_t>(N) * sizeof(T);

    const RingLayout L = ring_layout(false, LN, sizeof(T), N, tpr, S, p.stat_rows, blockDim.x);
    unsigned char *ring = smem + L.ring_off + (size_t)slot * S * rowb;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bar_off) + slot * S;
    float *red = reinterpret_cast<float *>(smem + L.red_off) + slot * 4 * W * 2;
    volatile int *flag = reinterpret_cast<int *>(smem + L.flag_off) + slot;

    int64_t row0;
    int nrows;
    block_rows(p.M, p.G, blockIdx.x, row0, nrows);
    const int ns = slot < nrows ? (nrows - slot + slots - 1) / slots : 0;

    if (tid == 0) {
        uint64_t *all = reinterpret_cast<uint64_t *>(smem + L.bar_off);
        for (int i = 0; i < slots * S; ++i) mbar_init(&all[i], 1);
        fence_barrier_init();
    }
    if (ts == 0) *flag = 0;
    __syncthreads();

    const uint64_t pol = policy_evict_first();
    const T *xg = static_cast<const T *>(p.x);
    auto issue = [&](int k) {
        const int st = k % S;
        const int64_t row = row0 + slot + (int64_t)k * slots;
        mbar_arrive_expect_tx(&bar[st], rowb);
        bulk_load(ring + (size_t)st * rowb, xg + row * N, rowb, &bar[st], pol);
    };
    int issued = 0;
    if (ts == 0) {
        for (; issued < S && issued < ns; ++issued) issue(issued);
    }

    // gamma / beta: unpacked once (HOLD) or kept as raw vectors
    float gam[HOLD ? E : 1], bet[HOLD && LN ? E : 1];
    uint4 graw[HOLD ? 1 : NV], braw[HOLD ? 1 : NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int v = ts + j * tpr;
        uint4 g = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        if (v < nvec) {
            g = ld_global_nc_v4(static_cast<const T *>(p.gamma) + (size_t)v * V);
            if (LN) b = ld_global_nc_v4(static_cast<const T *>(p.beta) + (size_t)v * V);
        }
        if constexpr (HOLD) {
            Tr::unpack(g, gam + j * V);
            if constexpr (LN) Tr::unpack(b, bet + j * V);
        } else {
            graw[j] = g;
            braw[j] = b;
        }
    }
    const float fn = static_cast<float>(N);

    int k = 0;
    for (; k < ns; ++k) {
        const int st = k % S;
        const bool timed_out = !mbar_wait_bounded(&bar[st], (k / S) & 1);
        if (timed_out) record_error(p.err, kErrWaitFull);
        const unsigned char *sx = ring + (size_t)st * rowb;
        // the row, in registers: fp32 values (HOLD) or raw vectors
        float xf[HOLD ? E : 1];
        uint4 xr[HOLD ? 1 : NV];
        float sum[1] = {0.f};
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int v = ts + j * tpr;
            const uint4 raw = v < nvec ? *reinterpret_cast<const uint4 *>(sx + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
            float f[V];
            Tr::unpack(raw, f);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                sum[0] = LN ? sum[0] + f[e] : fmaf(f[e], f[e], sum[0]);
                if constexpr (HOLD) xf[j * V + e] = f[e];
            }
            if constexpr (!HOLD) xr[j] = raw;
        }
        const bool abort = slot_reduce<1>(sum, red + (k & 1) * 2 * W * 2, flag, timed_out, W, warp, lane, 1 + slot, tpr);
        if (abort) break;
        // the slot has the row in registers: refill its stage
        if (ts == 0 && issued < ns) {
            fence_proxy_async();
            issue(issued++);
        }
        float mu = 0.f, rs;
        if constexpr (LN) {
            mu = sum[0] / fn;
            float sq[1] = {0.f};
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                float f[V];
                if constexpr (HOLD) {
#pragma unroll
                    for (int e = 0; e < V; ++e) f[e] = xf[j * V + e];
                } else {
                    Tr::unpack(xr[j], f);
                }
                const bool live = ts + j * tpr < nvec;
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float d = live ? f[e] - mu : 0.f;
                    sq[0] = fmaf(d, d, sq[0]);
                }
            }
            slot_reduce<1>(sq, red + ((k & 1) * 2 + 1) * W * 2, flag, false, W, warp, lane, 1 + slot, tpr);
            rs = 1.0f / sqrtf(sq[0] / fn + p.eps);
        } else {
            rs = 1.0f / sqrtf(sum[0] / fn + p.eps);
        }
        const int64_t row = row0 + slot + (int64_t)k * slots;
        T *yrow = static_cast<T *>(p.y) + row * N;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int v = ts + j * tpr;
            if (v < nvec) {
                float f[V], g[V], b[V], o[V];
                if constexpr (HOLD) {
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        f[e] = xf[j * V + e];
                        g[e] = gam[j * V + e];
                        b[e] = LN ? bet[j * V + e] : 0.f;
                    }
                } else {
                    Tr::unpack(xr[j], f);
                    Tr::unpack(graw[j], g);
                    if constexpr (LN) Tr::unpack(braw[j], b);
                }
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float xhat = LN ? (f[e] - mu) * rs : f[e] * rs;
                    o[e] = LN ? fmaf(g[e], xhat, b[e]) : g[e] * xhat;
                }
                st_global_cs_v4(yrow + (size_t)v * V, Tr::pack(o));
            }
        }
        if (ts == 0) {
            p.rstd[row] = rs;
            if (LN) p.mean[row] = mu;
        }
    }
    // after a wait ran out: let the copies this slot still has in flight land
    // (bounded) before the CTA exits
    if (ts == 0) {
        for (int kk = k; kk < issued; ++kk) {
            if (!mbar_wait_bounded(&bar[kk % S], (kk / S) & 1, 100000000ull)) {
                record_error(p.err, kErrDrain);
                break;
            }
        }
    }
}

template <typename T, bool LN>
__global__ void __launch_bounds__(kGenericThreads) fwd_plain_kernel(const FwdParams p) {
    using Tr = Traits<T>;
    __shared__ float sm[kGenericThreads / 32];
    const int N = p.N;
    const float fn = static_cast<float>(N);
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
        const T *xr = static_cast<const T *>(p.x) + row * N;
        float mu = 0.f;
        if (LN) {
            float s = 0.f;
            for (int j = threadIdx.x; j < N; j += blockDim.x) s += Tr::load1(xr + j);
            mu = block_sum(s, sm) / fn;
        }
        float q = 0.f;
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            const float d = Tr::load1(xr + j) - mu;
            q = fmaf(d, d, q);
        }
        const float rs = 1.0f / sqrtf(block_sum(q, sm) / fn + p.eps);
        T *yr = static_cast<T *>(p.y) + row * N;
        const T *g = static_cast<const T *>(p.gamma);
        const T *b = static_cast<const T *>(p.beta);
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            const float xhat = (Tr::load1(xr + j) - mu) * rs;
            const float gj = Tr::load1(g + j);
            Tr::store1(yr + j, LN ? fmaf(gj, xhat, Tr::load1(b + j)) : gj * xhat);
        }
        if (threadIdx.x == 0) {
            p.rstd[row] = rs;
            if (LN) p.mean[row] = mu;
        }
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
namespace {

template <typename K>
cudaError_t allow_smem(K kernel) {
    // the opt-in limit is set once per kernel and device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
}

template <typename T, bool LN, int NV, bool HOLD>
cudaError_t fwd_staged_t(const FwdParams &p, size_t smem, cudaStream_t s) {
    static thread_local int set_for_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (set_for_dev != dev) {
        e = allow_smem(fwd_staged_kernel<T, LN, NV, HOLD>);
        if (e != cudaSuccess) return e;
        set_for_dev = dev;
    }
    fwd_staged_kernel<T, LN, NV, HOLD><<<p.G, kRingThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// held-register variants up to 16 elements per thread, raw-vector ones beyond
template <typename T, bool LN>
cudaError_t fwd_staged_nv(int nv, const FwdParams &p, size_t smem, cudaStream_t s) {
    constexpr int V = Traits<T>::kVec;
    if (nv * V <= 16) {
        switch (nv) {
            case 1: return fwd_staged_t<T, LN, 1, true>(p, smem, s);
            case 2: return fwd_staged_t<T, LN, 2, true>(p, smem, s);
            case 3: if constexpr (3 * V <= 16) return fwd_staged_t<T, LN, 3, true>(p, smem, s); break;
            case 4: if constexpr (4 * V <= 16) return fwd_staged_t<T, LN, 4, true>(p, smem, s); break;
        }
        return cudaErrorInvalidValue;
    }
    if constexpr (V == 8) {
        switch (nv) {
            case 3: return fwd_staged_t<T, LN, 3, false>(p, smem, s);
            case 4: return fwd_staged_t<T, LN, 4, false>(p, smem, s);
        }
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t fwd_staged_ln(bool ln, int nv, const FwdParams &p, size_t smem, cudaStream_t s) {
    return ln ? fwd_staged_nv<T, true>(nv, p, smem, s) : fwd_staged_nv<T, false>(nv, p, smem, s);
}

template <typename T>
cudaError_t fwd_plain_ln(bool ln, const FwdParams &p, cudaStream_t s) {
    if (ln)
        fwd_plain_kernel<T, true><<<p.G, kGenericThreads, 0, s>>>(p);
    else
        fwd_plain_kernel<T, false><<<p.G, kGenericThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_staged(int dtype, bool ln, int nv, const FwdParams &p, size_t smem, cudaStream_t s) {
    switch (dtype) {
        case 0: return fwd_staged_ln<float>(ln, nv, p, smem, s);
        case 1: return fwd_staged_ln<__half>(ln, nv, p, smem, s);
        case 2: return fwd_staged_ln<__nv_bfloat16>(ln, nv, p, smem, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_plain(int dtype, bool ln, const FwdParams &p, cudaStream_t s) {
    switch (dtype) {
        case 0: return fwd_plain_ln<float>(ln, p, s);
        case 1: return fwd_plain_ln<__half>(ln, p, s);
        case 2: return fwd_plain_ln<__nv_bfloat16>(ln, p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbn
