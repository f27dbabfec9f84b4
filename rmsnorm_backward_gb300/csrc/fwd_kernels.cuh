// fwd_kernels.cuh -- LayerNorm / RMSNorm forward kernel templates for
// sm_103a, instantiated once per storage dtype in fwd_f32.cu, fwd_f16.cu and
// fwd_bf16.cu.
//
// Definition followed: "Norm backward in Triton -- the dγ/dβ reduction",
// section "The gradients" (forward line and RMSNorm paragraph), with the
// variance taken as in "05: Layer norm", kernel ln_fwd: the biased variance of
// the row centred on its mean, computed after the mean (two passes), eps
// under the root.  The forward saves the per-row mean (LayerNorm) and rstd
// for the backward ("Norm & activation backward", section "Half one").
//
// Kernels:
//  * fwd_staged_kernel: one persistent CTA per SM.  The CTA's rows are split
//    over slots of tpr threads; each slot streams its rows through a ring of
//    shared-memory stages filled by 1-D bulk (TMA) copies that complete on
//    mbarriers.  A thread keeps its part of the row in registers (fp32 when
//    it owns <= 16 elements, raw vectors otherwise), so both passes of the
//    two-pass variance read on-chip data and x leaves HBM once.
//  * fwd_plain_kernel: any N and alignment; a CTA walks a row three times
//    with scalar loads (mean, centred squares, output), the later passes
//    hitting L1/L2.
#pragma once

#include <atomic>

#include "bwd_kernels.cuh"  // ensure_smem_optin
#include "gbn_device.cuh"
#include "gbn_launch.h"

namespace gbn {

template <typename T, bool LN, int NV, bool FULL>
__global__ void __launch_bounds__(kRingThreads, 1) fwd_staged_kernel(const FwdParams p) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int E = NV * V;
    constexpr bool HOLD = E <= 16;
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
    const uint32_t vstride = static_cast<uint32_t>(tpr) * 16;

    const RingLayout L = ring_layout(false, LN, sizeof(T), N, tpr, S, p.stat_rows, blockDim.x);
    unsigned char *ring = smem + L.ring_off + (size_t)slot * S * rowb;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bar_off) + slot * S;
    float *red = reinterpret_cast<float *>(smem + L.red_off) + slot * 4 * 2 * kRedStride;
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

    const size_t row_step = (size_t)slots * p.ld_y;
    const size_t xrow_step = (size_t)slots * p.ld_x;
    const T *px = static_cast<const T *>(p.x) + (row0 + slot) * p.ld_x;
    int issued = 0, pst = 0;
    auto issue = [&]() {
        mbar_arrive_expect_tx(&bar[pst], rowb);
        bulk_load_nohint(ring + (size_t)pst * rowb, px, rowb, &bar[pst]);
        px += xrow_step;
        if (++pst == S) pst = 0;
        ++issued;
    };
    if (ts == 0) {
        while (issued < S && issued < ns) issue();
    }

    // gamma / beta: unpacked once (HOLD) or kept as raw vectors
    float gam[HOLD ? E : 1], bet[HOLD && LN ? E : 1];
    uint4 graw[HOLD ? 1 : NV], braw[HOLD ? 1 : NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int v = ts + j * tpr;
        uint4 g = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        if (FULL || v < nvec) {
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
    const float inv_n = 1.0f / static_cast<float>(N);
    T *yrow = static_cast<T *>(p.y) + (row0 + slot) * p.ld_y + (size_t)ts * V;
    int64_t row = row0 + slot;
    RingPos pos;

    int k = 0;
    for (; k < ns; ++k) {
        const bool timed_out = !mbar_wait_bounded(&bar[pos.stage], pos.parity);
        if (timed_out) record_error(p.err, kErrWaitFull);
        const unsigned char *sx = ring + (size_t)pos.stage * rowb + (size_t)ts * 16;
        // the row, in registers: fp32 values (HOLD) or raw vectors
        float xf[HOLD ? E : 1];
        uint4 xr[HOLD ? 1 : NV];
        float sum[1] = {0.f};
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const uint4 raw = (FULL || ts + j * tpr < nvec) ? *reinterpret_cast<const uint4 *>(sx + j * vstride)
                                                            : make_uint4(0, 0, 0, 0);
            float f[V];
            Tr::unpack(raw, f);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                sum[0] = LN ? sum[0] + f[e] : fmaf(f[e], f[e], sum[0]);
                if constexpr (HOLD) xf[j * V + e] = f[e];
            }
            if constexpr (!HOLD) xr[j] = raw;
        }
        const bool abort = slot_reduce<1>(sum, red + (k & 1) * 2 * 2 * kRedStride, flag, timed_out, W, warp, lane,
                                          1 + slot, tpr);
        if (abort) break;
        // the slot has the row in registers: refill its stage
        if (ts == 0 && issued < ns) {
            fence_proxy_async();
            issue();
        }
        float mu = 0.f, rs;
        if constexpr (LN) {
            mu = sum[0] * inv_n;
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
                const bool live = FULL || ts + j * tpr < nvec;
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float d = live ? f[e] - mu : 0.f;
                    sq[0] = fmaf(d, d, sq[0]);
                }
            }
            slot_reduce<1>(sq, red + ((k & 1) * 2 + 1) * 2 * kRedStride, flag, false, W, warp, lane, 1 + slot, tpr);
            rs = 1.0f / sqrtf(sq[0] * inv_n + p.eps);
        } else {
            rs = 1.0f / sqrtf(sum[0] * inv_n + p.eps);
        }
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if (FULL || ts + j * tpr < nvec) {
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
                st_global_cs_v4(yrow + (size_t)j * tpr * V, Tr::pack(o));
            }
        }
        if (ts == 0) {
            p.rstd[row] = rs;
            if (LN) p.mean[row] = mu;
        }
        yrow += row_step;
        row += slots;
        pos.next(S);
    }
    // after a wait ran out: let the copies this slot still has in flight land
    // (bounded) before the CTA exits
    if (ts == 0) {
        for (int kk = k; kk < issued; ++kk) {
            if (!mbar_wait_bounded(&bar[kk % S], (kk / S) & 1, kDrainNs)) {
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
    const float inv_n = 1.0f / static_cast<float>(N);
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
        const T *xr = static_cast<const T *>(p.x) + row * p.ld_x;
        float mu = 0.f;
        if (LN) {
            float s = 0.f;
            for (int j = threadIdx.x; j < N; j += blockDim.x) s += Tr::load1(xr + j);
            mu = block_sum(s, sm) * inv_n;
        }
        float q = 0.f;
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            const float d = Tr::load1(xr + j) - mu;
            q = fmaf(d, d, q);
        }
        const float rs = 1.0f / sqrtf(block_sum(q, sm) * inv_n + p.eps);
        T *yr = static_cast<T *>(p.y) + row * p.ld_y;
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

template <typename T, bool LN, int NV, bool FULL>
cudaError_t fwd_staged_launch(const FwdParams &p, size_t smem, cudaStream_t s) {
    static std::atomic<uint64_t> done{0};
    cudaError_t e = ensure_smem_optin(fwd_staged_kernel<T, LN, NV, FULL>, done);
    if (e != cudaSuccess) return e;
    fwd_staged_kernel<T, LN, NV, FULL><<<p.G, kRingThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename T, bool LN>
cudaError_t fwd_staged_nv(int nv, bool full, const FwdParams &p, size_t smem, cudaStream_t s) {
    switch (nv) {
        case 1: return full ? fwd_staged_launch<T, LN, 1, true>(p, smem, s) : fwd_staged_launch<T, LN, 1, false>(p, smem, s);
        case 2: return full ? fwd_staged_launch<T, LN, 2, true>(p, smem, s) : fwd_staged_launch<T, LN, 2, false>(p, smem, s);
        case 3: return full ? fwd_staged_launch<T, LN, 3, true>(p, smem, s) : fwd_staged_launch<T, LN, 3, false>(p, smem, s);
        case 4: return full ? fwd_staged_launch<T, LN, 4, true>(p, smem, s) : fwd_staged_launch<T, LN, 4, false>(p, smem, s);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t fwd_staged_dispatch(bool ln, int nv, bool full, const FwdParams &p, size_t smem, cudaStream_t s) {
    return ln ? fwd_staged_nv<T, true>(nv, full, p, smem, s) : fwd_staged_nv<T, false>(nv, full, p, smem, s);
}

template <typename T>
cudaError_t fwd_plain_dispatch(bool ln, const FwdParams &p, cudaStream_t s) {
    if (ln)
        fwd_plain_kernel<T, true><<<p.G, kGenericThreads, 0, s>>>(p);
    else
        fwd_plain_kernel<T, false><<<p.G, kGenericThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gbn
