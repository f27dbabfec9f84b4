// bwd_kernels.cuh -- LayerNorm / RMSNorm backward kernel templates for
// sm_103a, instantiated once per storage dtype in bwd_f32.cu, bwd_f16.cu and
// bwd_bf16.cu.
//
// Definition followed: "Norm backward in Triton -- the dγ/dβ reduction",
// section "The gradients": with dyhat = dy*gamma,
//   dx = rstd*(dyhat - mean(dyhat) - xhat*mean(dyhat*xhat))   (RMSNorm: no
//   mean(dyhat) term), dgamma = sum over rows of dy*xhat, dbeta = sum of dy.
// xhat is recomputed from the saved per-row mean / rstd, never stored
// ("Norm & activation backward", section "Half one").  dgamma / dbeta use the
// disjoint-row-block scheme of "Norm backward in Triton", section "The hard
// half": each CTA owns a contiguous block of rows, accumulates its partial
// sums in registers and stores one partial row (no atomics); colsum_kernel
// (norm_bwd.cu) then sums the partial rows per column in a fixed order.
//
// Kernels:
//  * bwd_staged_kernel: one persistent CTA per SM; its rows are spread over
//    slots of tpr threads.  Each slot streams x and dy rows through a ring of
//    shared-memory stages filled by 1-D bulk (TMA) copies completing on
//    mbarriers.  A thread owns NV fixed 16-byte column vectors.  Pass 1
//    reads its vectors from the stage and forms the two in-row sums (warp
//    shuffles plus one named barrier) and the per-column fp32 accumulators of
//    dy*xhat and dy; pass 2 writes dx with 16-byte streaming stores, from
//    values held in registers (xhat and dyhat up to 16 elements per thread;
//    raw x and dyhat up to 32 for RMSNorm, gamma then staged in shared
//    memory) or by re-reading the stage (wider rows).  The slot's barrier also shows that
//    every thread is done with a stage, so the stage is refilled right away
//    (held) or one row later (re-read).  At the end the slots' accumulators
//    are added in slot order in shared memory and the CTA stores its
//    partial row.
//  * bwd_plain_kernel: any N and alignment, scalar loads, the CTA's own
//    partial row in global memory as the accumulator.
#pragma once

#include <atomic>

#include "gbn_device.cuh"
#include "gbn_launch.h"

namespace gbn {

// This CTA's partial row(s) of dgamma / dbeta from the threads' register
// accumulators (a thread owns vectors ts, ts + tpr, ...).  Several slots add
// their accumulators in slot order in shared memory (`comb`, the ring area,
// free once every slot is done with its stages).  With p.atom_g set (the
// atomics ablation) the sums go into dgamma / dbeta with fp32 atomics.
template <typename T, bool LN, int NV, bool FULL>
__device__ __forceinline__ void bwd_store_partials(const BwdParams &p, const float *acc_g, const float *acc_b,
                                                   unsigned char *comb_area, int slots, int slot, int ts, int tpr,
                                                   int nvec) {
    constexpr int V = Traits<T>::kVec;
    const int tid = threadIdx.x;
    const int N = p.N;
    const int ldp = p.ldp;
    const bool atomic = p.atom_g != nullptr;  // reduction ablation
    float *pg = atomic ? p.atom_g : p.part + (size_t)blockIdx.x * ldp;
    float *pb = atomic ? p.atom_b : (p.part_b ? p.part_b : p.part + (size_t)p.G * ldp) + (size_t)blockIdx.x * ldp;
    auto put = [atomic](float *dst, const float4 &v) {
        if (atomic) {
            atomicAdd(dst, v.x);
            atomicAdd(dst + 1, v.y);
            atomicAdd(dst + 2, v.z);
            atomicAdd(dst + 3, v.w);
        } else {
            *reinterpret_cast<float4 *>(dst) = v;
        }
    };
    if (slots == 1) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int v = ts + j * tpr;
            if (FULL || v < nvec) {
#pragma unroll
                for (int e = 0; e < V; e += 4) {
                    put(pg + (size_t)v * V + e,
                        make_float4(acc_g[j * V + e], acc_g[j * V + e + 1], acc_g[j * V + e + 2], acc_g[j * V + e + 3]));
                    if constexpr (LN)
                        put(pb + (size_t)v * V + e, make_float4(acc_b[j * V + e], acc_b[j * V + e + 1],
                                                                acc_b[j * V + e + 2], acc_b[j * V + e + 3]));
                }
            }
        }
    } else {
        __syncthreads();  // every slot is done with its ring stages
        float *comb = reinterpret_cast<float *>(comb_area);
        float *comb_g = comb + (size_t)slot * ldp;
        float *comb_b = comb + ((size_t)slots + slot) * ldp;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int v = ts + j * tpr;
            if (FULL || v < nvec) {
#pragma unroll
                for (int e = 0; e < V; e += 4) {
                    *reinterpret_cast<float4 *>(comb_g + (size_t)v * V + e) = make_float4(
                        acc_g[j * V + e], acc_g[j * V + e + 1], acc_g[j * V + e + 2], acc_g[j * V + e + 3]);
                    if constexpr (LN)
                        *reinterpret_cast<float4 *>(comb_b + (size_t)v * V + e) = make_float4(
                            acc_b[j * V + e], acc_b[j * V + e + 1], acc_b[j * V + e + 2], acc_b[j * V + e + 3]);
                }
            }
        }
        __syncthreads();
        for (int c = tid * 4; c < N; c += blockDim.x * 4) {
            float4 a = *reinterpret_cast<const float4 *>(comb + c);
            for (int s2 = 1; s2 < slots; ++s2) {
                const float4 b = *reinterpret_cast<const float4 *>(comb + (size_t)s2 * ldp + c);
                a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
            }
            put(pg + c, a);
            if constexpr (LN) {
                const float *cb = comb + (size_t)slots * ldp;
                float4 d = *reinterpret_cast<const float4 *>(cb + c);
                for (int s2 = 1; s2 < slots; ++s2) {
                    const float4 b = *reinterpret_cast<const float4 *>(cb + (size_t)s2 * ldp + c);
                    d.x += b.x; d.y += b.y; d.z += b.z; d.w += b.w;
                }
                put(pb + c, d);
            }
        }
    }
}

template <typename T, bool LN, int NV, bool FULL, bool RECOMP>
__global__ void __launch_bounds__(kRingThreads, 1) bwd_staged_kernel(const BwdParams p) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int E = NV * V;                         // elements a thread owns per row
    constexpr int MODE = bwd_hold_mode(LN, E);        // what pass 2 finds in registers
    constexpr bool HOLD = MODE != kReread;            // the stage is free after pass 1
    constexpr bool GSMEM = bwd_gamma_smem(LN, E);     // gamma read from shared memory (fp32)
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
    const uint32_t stage_bytes = 2 * rowb;
    const uint32_t vstride = static_cast<uint32_t>(tpr) * 16;  // bytes between a thread's vectors

    const RingLayout L = ring_layout(true, LN, sizeof(T), N, tpr, S, p.stat_rows, blockDim.x, GSMEM);
    unsigned char *ring = smem + L.ring_off + (size_t)slot * S * stage_bytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bar_off) + slot * S;
    float *gam_s = reinterpret_cast<float *>(smem + L.gam_off);
    float *st_rstd = reinterpret_cast<float *>(smem + L.stat_off);
    float *st_mean = st_rstd + p.stat_rows;
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

    // producer (thread 0 of the slot): the slot's rows in order
    const size_t row_step = (size_t)slots * p.ld_dx;
    int issued = 0, pst = 0;
    auto issue = [&]() {
        const int64_t row = row0 + slot + (int64_t)issued * slots;
        unsigned char *dst = ring + (size_t)pst * stage_bytes;
        mbar_arrive_expect_tx(&bar[pst], stage_bytes);
        bulk_load_nohint(dst, static_cast<const T *>(p.x) + row * p.ld_x, rowb, &bar[pst]);
        bulk_load_nohint(dst + rowb, static_cast<const T *>(p.dy) + row * p.ld_dy, rowb, &bar[pst]);
        if (++pst == S) pst = 0;
        ++issued;
    };
    if (ts == 0) {
        while (issued < S && issued < ns) issue();
    }

    // this CTA's saved statistics, staged once (RECOMP: none were saved)
    if constexpr (!RECOMP) {
        for (int i = tid; i < nrows; i += blockDim.x) {
            st_rstd[i] = p.rstd[row0 + i];
            if (LN) st_mean[i] = p.mean[row0 + i];
        }
    }
    // gamma: unpacked into registers (kHoldAll), unpacked into shared memory
    // (kHoldX), or kept as raw vectors (kReread)
    constexpr bool GREG = HOLD && !GSMEM;
    float gam[GREG ? E : 1];
    uint4 graw[HOLD ? 1 : NV];
    if constexpr (GSMEM) {
        for (int v = tid; v < nvec; v += blockDim.x) {
            float f[V];
            Tr::unpack(ld_global_nc_v4(static_cast<const T *>(p.gamma) + (size_t)v * V), f);
#pragma unroll
            for (int e = 0; e < V; e += 4)
                *reinterpret_cast<float4 *>(gam_s + (size_t)v * V + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int v = ts + j * tpr;
            const uint4 g = (FULL || v < nvec) ? ld_global_nc_v4(static_cast<const T *>(p.gamma) + (size_t)v * V)
                                               : make_uint4(0, 0, 0, 0);
            if constexpr (GREG)
                Tr::unpack(g, gam + j * V);
            else
                graw[j] = g;
        }
    }
    float acc_g[E], acc_b[LN ? E : 1];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        acc_g[e] = 0.f;
        if constexpr (LN) acc_b[e] = 0.f;
    }
    __syncthreads();
    griddep_launch_dependents();

    const float inv_n = 1.0f / static_cast<float>(N);
    T *dxrow = static_cast<T *>(p.dx) + (row0 + slot) * p.ld_dx + (size_t)ts * V;
    RingPos pos;
    int k = 0;
    for (; k < ns; ++k) {
        const bool timed_out = !mbar_wait_bounded(&bar[pos.stage], pos.parity, p.wait_ns);
        if (timed_out) record_error(p.err, kErrWaitFull);
        if constexpr (RECOMP && MODE == kHoldAll) {
            // No saved statistics, row held in registers: x and dy in fp32.
            // RMSNorm: sum(x^2) and sum(dyhat*x) in one exchange give rstd and
            // c2 = rstd*sum(dyhat*x)/N.  LayerNorm: sum(x) first (the mean),
            // then sum((x-mean)^2), sum(dyhat), sum(dyhat*(x-mean)) in one
            // exchange.  dgamma / dbeta accumulate in pass 2, once rstd is known.
            const unsigned char *sx = ring + (size_t)pos.stage * stage_bytes + (size_t)ts * 16;
            float xv[E], dv[E];
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (FULL || ts + j * tpr < nvec) {
                    Tr::unpack(*reinterpret_cast<const uint4 *>(sx + j * vstride), xv + j * V);
                    Tr::unpack(*reinterpret_cast<const uint4 *>(sx + rowb + j * vstride), dv + j * V);
                } else {
#pragma unroll
                    for (int e = 0; e < V; ++e) xv[j * V + e] = dv[j * V + e] = 0.f;
                }
            }
            float mu = 0.f;
            if constexpr (LN) {
                float m[1] = {0.f};
#pragma unroll
                for (int e = 0; e < E; ++e) m[0] += xv[e];
                if (slot_reduce<1>(m, red + 6 * kRedStride, flag, timed_out, W, warp, lane, 1 + slot, tpr)) break;
                mu = m[0] * inv_n;
            }
            float r[LN ? 3 : 2];  // sum((x-mean)^2), [sum(dyhat)], sum(dyhat*(x-mean))
#pragma unroll
            for (int q = 0; q < (LN ? 3 : 2); ++q) r[q] = 0.f;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const bool live = FULL || ts + j * tpr < nvec;
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float d = live ? xv[j * V + e] - mu : 0.f;
                    const float dyhat = dv[j * V + e] * gam[j * V + e];
                    r[0] = fmaf(d, d, r[0]);
                    if constexpr (LN) r[1] += dyhat;
                    r[LN ? 2 : 1] = fmaf(dyhat, d, r[LN ? 2 : 1]);
                }
            }
            const bool abort = slot_reduce<LN ? 3 : 2>(r, red + (k & 1) * 3 * kRedStride, flag, LN ? false : timed_out,
                                                       W, warp, lane, 1 + slot, tpr);
            if (abort) break;
            if (ts == 0 && issued < ns) {  // the row is in registers: refill its stage
                fence_proxy_async();
                issue();
            }
            const float rs = 1.0f / sqrtf(r[0] * inv_n + p.eps);
            const float a = -rs * (rs * (r[LN ? 2 : 1] * inv_n));
            const float b = LN ? -rs * (r[1] * inv_n) : 0.f;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (FULL || ts + j * tpr < nvec) {
                    float o[V];
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float xhat = (xv[j * V + e] - mu) * rs;
                        const float dyv = dv[j * V + e];
                        acc_g[j * V + e] = fmaf(dyv, xhat, acc_g[j * V + e]);
                        if constexpr (LN) acc_b[j * V + e] += dyv;
                        o[e] = fmaf(dyv * gam[j * V + e], rs, LN ? fmaf(xhat, a, b) : xhat * a);
                    }
                    st_global_cs_v4(dxrow + (size_t)j * tpr * V, Tr::pack(o));
                }
            }
            dxrow += row_step;
            pos.next(S);
            continue;
        }
        if constexpr (RECOMP && !LN && MODE == kHoldX) {
            // RMSNorm with no saved statistics, x held as raw vectors: pass 1
            // forms sum(x^2) and sum(dyhat*x) together (one exchange gives
            // rstd and c2 = rstd*sum(dyhat*x)/N) and holds dy itself; pass 2
            // adds dy*xhat into the dgamma accumulators and writes dx =
            // dy*gamma*rstd + x*(rstd*a), gamma from shared memory
            const unsigned char *sx = ring + (size_t)pos.stage * stage_bytes + (size_t)ts * 16;
            const unsigned char *sdy = sx + rowb;
            uint4 xr[NV];
            float dyv[E];
            float r[2] = {0.f, 0.f};  // sum(x^2), sum(dyhat*x)
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                float xf[V], gl[V];
                if (FULL || ts + j * tpr < nvec) {
                    xr[j] = *reinterpret_cast<const uint4 *>(sx + j * vstride);
                    Tr::unpack(xr[j], xf);
                    Tr::unpack(*reinterpret_cast<const uint4 *>(sdy + j * vstride), dyv + j * V);
                    const float *gs = gam_s + (size_t)(ts + j * tpr) * V;
#pragma unroll
                    for (int e = 0; e < V; e += 4) {
                        const float4 t = *reinterpret_cast<const float4 *>(gs + e);
                        gl[e] = t.x, gl[e + 1] = t.y, gl[e + 2] = t.z, gl[e + 3] = t.w;
                    }
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        r[0] = fmaf(xf[e], xf[e], r[0]);
                        r[1] = fmaf(dyv[j * V + e] * gl[e], xf[e], r[1]);
                    }
                } else {
                    xr[j] = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int e = 0; e < V; ++e) dyv[j * V + e] = 0.f;
                }
            }
            if (slot_reduce<2>(r, red + (k & 1) * 2 * kRedStride, flag, timed_out, W, warp, lane, 1 + slot, tpr))
                break;
            if (ts == 0 && issued < ns) {  // the row is in registers: refill its stage
                fence_proxy_async();
                issue();
            }
            const float rs = 1.0f / sqrtf(r[0] * inv_n + p.eps);
            const float ax = (-rs * (rs * (r[1] * inv_n))) * rs;  // xhat*a = x*(rstd*a)
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (FULL || ts + j * tpr < nvec) {
                    float xf[V], o[V];
                    Tr::unpack(xr[j], xf);
                    const float *gs = gam_s + (size_t)(ts + j * tpr) * V;
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float dyv_e = dyv[j * V + e];
                        acc_g[j * V + e] = fmaf(dyv_e, xf[e] * rs, acc_g[j * V + e]);
                        o[e] = fmaf(dyv_e * gs[e], rs, xf[e] * ax);
                    }
                    st_global_cs_v4(dxrow + (size_t)j * tpr * V, Tr::pack(o));
                }
            }
            dxrow += row_step;
            pos.next(S);
            continue;
        }
        const int i = slot + k * slots;
        const unsigned char *sx = ring + (size_t)pos.stage * stage_bytes + (size_t)ts * 16;
        const unsigned char *sdy = sx + rowb;
        float rs, mu = 0.f;
        if constexpr (RECOMP) {
            // the statistics from the staged row, as the forward forms them:
            // mean, then the centred squares (LayerNorm), or the mean square
            float q[1] = {0.f};
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (FULL || ts + j * tpr < nvec) {
                    float f[V];
                    Tr::unpack(*reinterpret_cast<const uint4 *>(sx + j * vstride), f);
#pragma unroll
                    for (int e = 0; e < V; ++e) q[0] = LN ? q[0] + f[e] : fmaf(f[e], f[e], q[0]);
                }
            }
            if (slot_reduce<1>(q, red + 4 * kRedStride, flag, timed_out, W, warp, lane, 1 + slot, tpr)) break;
            if constexpr (LN) {
                mu = q[0] * inv_n;
                float c[1] = {0.f};
#pragma unroll
                for (int j = 0; j < NV; ++j) {
                    if (FULL || ts + j * tpr < nvec) {
                        float f[V];
                        Tr::unpack(*reinterpret_cast<const uint4 *>(sx + j * vstride), f);
#pragma unroll
                        for (int e = 0; e < V; ++e) {
                            const float d = f[e] - mu;
                            c[0] = fmaf(d, d, c[0]);
                        }
                    }
                }
                slot_reduce<1>(c, red + 5 * kRedStride, flag, false, W, warp, lane, 1 + slot, tpr);
                rs = 1.0f / sqrtf(c[0] * inv_n + p.eps);
            } else {
                rs = 1.0f / sqrtf(q[0] * inv_n + p.eps);
            }
        } else {
            rs = st_rstd[i];
            mu = LN ? st_mean[i] : 0.f;
        }
        // pass 1
        float xh[MODE == kHoldAll ? E : 1], dh[HOLD ? E : 1];
        uint4 xraw[MODE == kHoldX ? NV : 1];
        float s[2] = {0.f, 0.f};  // sum(dyhat), sum(dyhat*xhat)
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float xf[V], df[V], gl[V];
            if (FULL || ts + j * tpr < nvec) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(sx + j * vstride);
                if constexpr (MODE == kHoldX) xraw[j] = xv;
                Tr::unpack(xv, xf);
                Tr::unpack(*reinterpret_cast<const uint4 *>(sdy + j * vstride), df);
            } else {
                if constexpr (MODE == kHoldX) xraw[j] = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int e = 0; e < V; ++e) xf[e] = df[e] = 0.f;
            }
            if constexpr (!HOLD) Tr::unpack(graw[j], gl);
            if constexpr (GSMEM) {
                const float *gs = gam_s + (size_t)(ts + j * tpr) * V;
#pragma unroll
                for (int e = 0; e < V; e += 4) {
                    const float4 t = (FULL || ts + j * tpr < nvec) ? *reinterpret_cast<const float4 *>(gs + e)
                                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                    gl[e] = t.x; gl[e + 1] = t.y; gl[e + 2] = t.z; gl[e + 3] = t.w;
                }
            }
#pragma unroll
            for (int e = 0; e < V; ++e) {
                const float g = GREG ? gam[j * V + e] : gl[e];
                const float xhat = LN ? (xf[e] - mu) * rs : xf[e] * rs;
                const float dyhat = df[e] * g;
                if constexpr (LN) s[0] += dyhat;
                s[1] = fmaf(dyhat, xhat, s[1]);
                acc_g[j * V + e] = fmaf(df[e], xhat, acc_g[j * V + e]);
                if constexpr (LN) acc_b[j * V + e] += df[e];
                if constexpr (MODE == kHoldAll) xh[j * V + e] = xhat;
                if constexpr (HOLD) dh[j * V + e] = dyhat;
            }
        }
        const bool abort = slot_reduce<2>(s, red + (k & 1) * 2 * kRedStride, flag, timed_out, W, warp, lane,
                                          1 + slot, tpr);
        if (abort) break;
        // HOLD: the slot is done with this stage; otherwise it re-reads this
        // stage in pass 2 and the previous stage is the one now free
        if (ts == 0 && issued < ns && (HOLD || k > 0)) {
            fence_proxy_async();
            issue();
        }
        // pass 2: dx = rstd*(dyhat - c1 - xhat*c2) = dyhat*rstd + xhat*a + b
        const float a = -rs * (s[1] * inv_n);
        const float b = LN ? -rs * (s[0] * inv_n) : 0.f;
        const float ax = a * rs;  // kHoldX (RMSNorm): xhat*a = x*(rstd*a)
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if (FULL || ts + j * tpr < nvec) {
                float o[V];
                if constexpr (MODE == kHoldAll) {
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        o[e] = fmaf(dh[j * V + e], rs, LN ? fmaf(xh[j * V + e], a, b) : xh[j * V + e] * a);
                } else if constexpr (MODE == kHoldX) {
                    float xf[V];
                    Tr::unpack(xraw[j], xf);
#pragma unroll
                    for (int e = 0; e < V; ++e) o[e] = fmaf(dh[j * V + e], rs, xf[e] * ax);
                } else {
                    float xf[V], df[V], gl[V];
                    Tr::unpack(*reinterpret_cast<const uint4 *>(sx + j * vstride), xf);
                    Tr::unpack(*reinterpret_cast<const uint4 *>(sdy + j * vstride), df);
                    Tr::unpack(graw[j], gl);
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float xhat = LN ? (xf[e] - mu) * rs : xf[e] * rs;
                        o[e] = fmaf(df[e] * gl[e], rs, LN ? fmaf(xhat, a, b) : xhat * a);
                    }
                }
                st_global_cs_v4(dxrow + (size_t)j * tpr * V, Tr::pack(o));
            }
        }
        dxrow += row_step;
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

    bwd_store_partials<T, LN, NV, FULL>(p, acc_g, acc_b, smem + L.ring_off, slots, slot, ts, tpr, nvec);
}

template <typename T, bool LN>
__global__ void __launch_bounds__(kGenericThreads) bwd_plain_kernel(const BwdParams p) {
    using Tr = Traits<T>;
    __shared__ float sm[kGenericThreads / 32];
    const int N = p.N;
    const float inv_n = 1.0f / static_cast<float>(N);
    int64_t row0;
    int nrows;
    block_rows(p.M, p.G, blockIdx.x, row0, nrows);
    float *pg = p.part + (size_t)blockIdx.x * p.ldp;
    float *pb = (p.part_b ? p.part_b : p.part + (size_t)p.G * p.ldp) + (size_t)blockIdx.x * p.ldp;
    griddep_launch_dependents();
    // column j is always handled by thread j % blockDim.x: a fixed order per column
    for (int j = threadIdx.x; j < N; j += blockDim.x) {
        pg[j] = 0.f;
        if (LN) pb[j] = 0.f;
    }
    const T *g = static_cast<const T *>(p.gamma);
    for (int i = 0; i < nrows; ++i) {
        const int64_t row = row0 + i;
        const T *xr = static_cast<const T *>(p.x) + row * p.ld_x;
        const T *dyr = static_cast<const T *>(p.dy) + row * p.ld_dy;
        float rs, mu = 0.f;
        if (p.rstd) {
            rs = p.rstd[row];
            mu = LN ? p.mean[row] : 0.f;
        } else {
            // no saved statistics: the forward's two passes over the row
            if (LN) {
                float t = 0.f;
                for (int j = threadIdx.x; j < N; j += blockDim.x) t += Tr::load1(xr + j);
                mu = block_sum(t, sm) * inv_n;
            }
            float q = 0.f;
            for (int j = threadIdx.x; j < N; j += blockDim.x) {
                const float d = Tr::load1(xr + j) - mu;
                q = fmaf(d, d, q);
            }
            rs = 1.0f / sqrtf(block_sum(q, sm) * inv_n + p.eps);
        }
        float s1 = 0.f, s2 = 0.f;
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            const float xhat = (Tr::load1(xr + j) - mu) * rs;
            const float dyhat = Tr::load1(dyr + j) * Tr::load1(g + j);
            s1 += dyhat;
            s2 = fmaf(dyhat, xhat, s2);
        }
        const float a = -rs * (block_sum(s2, sm) * inv_n);
        const float b = LN ? -rs * (block_sum(s1, sm) * inv_n) : 0.f;
        T *dxr = static_cast<T *>(p.dx) + row * p.ld_dx;
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            const float xhat = (Tr::load1(xr + j) - mu) * rs;
            const float dy = Tr::load1(dyr + j);
            const float dyhat = dy * Tr::load1(g + j);
            Tr::store1(dxr + j, fmaf(dyhat, rs, fmaf(xhat, a, b)));
            pg[j] = fmaf(dy, xhat, pg[j]);
            if (LN) pb[j] += dy;
        }
    }
    if (p.atom_g) {  // reduction ablation: add the CTA's partial row with atomics
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            atomicAdd(p.atom_g + j, pg[j]);
            if (LN) atomicAdd(p.atom_b + j, pb[j]);
        }
    }
}

// Reduction ablation after the column-walk design of "05: Layer norm"
// (kernel ln_bwd_dwdb): CTA b owns columns [32b, 32b + 32) and reads x and
// dy again, row by row; lane q of row-lane l adds rows l, l+32, ... of
// column 32b + q in order, then the 32 row-lane sums are added in order.
// Deterministic; costs a second read of x and dy.
template <typename T, bool LN, bool ACC>
__global__ void __launch_bounds__(1024) colwalk_kernel(const BwdParams p, float *__restrict__ dgamma,
                                                       float *__restrict__ dbeta) {
    using Tr = Traits<T>;
    __shared__ float sg[32][33], sb[32][33];
    const int q = threadIdx.x & 31, lane_row = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + q;
    float ag = 0.f, ab = 0.f;
    if (c < p.N) {
        const T *x = static_cast<const T *>(p.x) + c;
        const T *dy = static_cast<const T *>(p.dy) + c;
        int64_t r = lane_row;
        for (; r + 7 * 32 < p.M; r += 8 * 32) {
            float xv[8], dv[8], rs[8], mu[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t rr = r + u * 32;
                xv[u] = Tr::load1(x + rr * p.ld_x);
                dv[u] = Tr::load1(dy + rr * p.ld_dy);
                rs[u] = p.rstd[rr];
                mu[u] = LN ? p.mean[rr] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                ag = fmaf(dv[u], (xv[u] - mu[u]) * rs[u], ag);
                if (LN) ab += dv[u];
            }
        }
        for (; r < p.M; r += 32) {
            const float xv = Tr::load1(x + r * p.ld_x), dv = Tr::load1(dy + r * p.ld_dy);
            ag = fmaf(dv, (xv - (LN ? p.mean[r] : 0.f)) * p.rstd[r], ag);
            if (LN) ab += dv;
        }
    }
    sg[lane_row][q] = ag;
    sb[lane_row][q] = ab;
    __syncthreads();
    if (lane_row == 0 && c < p.N) {
        float tg = sg[0][q], tb = sb[0][q];
        for (int l = 1; l < 32; ++l) {
            tg += sg[l][q];
            tb += sb[l][q];
        }
        dgamma[c] = ACC ? dgamma[c] + tg : tg;
        if (LN) dbeta[c] = ACC ? dbeta[c] + tb : tb;
    }
}

template <typename T>
cudaError_t colwalk_dispatch(bool ln, const BwdParams &p, float *dg, float *db, bool acc, cudaStream_t s) {
    const dim3 grid((p.N + 31) / 32);
    if (ln)
        acc ? colwalk_kernel<T, true, true><<<grid, 1024, 0, s>>>(p, dg, db)
            : colwalk_kernel<T, true, false><<<grid, 1024, 0, s>>>(p, dg, db);
    else
        acc ? colwalk_kernel<T, false, true><<<grid, 1024, 0, s>>>(p, dg, db)
            : colwalk_kernel<T, false, false><<<grid, 1024, 0, s>>>(p, dg, db);
    return cudaGetLastError();
}

// Sets the opt-in dynamic shared-memory limit of `kernel` once per device.
template <typename T, bool LN, int NV, bool FULL, bool RECOMP>
cudaError_t bwd_staged_launch_r(const BwdParams &p, size_t smem, cudaStream_t s) {
    static std::atomic<uint64_t> done{0};
    cudaError_t e = ensure_smem_optin(bwd_staged_kernel<T, LN, NV, FULL, RECOMP>, done);
    if (e != cudaSuccess) return e;
    bwd_staged_kernel<T, LN, NV, FULL, RECOMP><<<p.G, kRingThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// recompute: no saved statistics (p.rstd == nullptr); the row's statistics
// are formed from the staged x with p.eps
template <typename T, bool LN, int NV, bool FULL>
cudaError_t bwd_staged_launch(const BwdParams &p, size_t smem, cudaStream_t s) {
    return p.rstd ? bwd_staged_launch_r<T, LN, NV, FULL, false>(p, smem, s)
                  : bwd_staged_launch_r<T, LN, NV, FULL, true>(p, smem, s);
}

template <typename T, bool LN>
cudaError_t bwd_staged_nv(int nv, bool full, const BwdParams &p, size_t smem, cudaStream_t s) {
    switch (nv) {
        case 1: return full ? bwd_staged_launch<T, LN, 1, true>(p, smem, s) : bwd_staged_launch<T, LN, 1, false>(p, smem, s);
        case 2: return full ? bwd_staged_launch<T, LN, 2, true>(p, smem, s) : bwd_staged_launch<T, LN, 2, false>(p, smem, s);
        case 3: return full ? bwd_staged_launch<T, LN, 3, true>(p, smem, s) : bwd_staged_launch<T, LN, 3, false>(p, smem, s);
        case 4: return full ? bwd_staged_launch<T, LN, 4, true>(p, smem, s) : bwd_staged_launch<T, LN, 4, false>(p, smem, s);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t bwd_staged_dispatch(bool ln, int nv, bool full, const BwdParams &p, size_t smem, cudaStream_t s) {
    return ln ? bwd_staged_nv<T, true>(nv, full, p, smem, s) : bwd_staged_nv<T, false>(nv, full, p, smem, s);
}

template <typename T>
cudaError_t bwd_plain_dispatch(bool ln, const BwdParams &p, cudaStream_t s) {
    if (ln)
        bwd_plain_kernel<T, true><<<p.G, kGenericThreads, 0, s>>>(p);
    else
        bwd_plain_kernel<T, false><<<p.G, kGenericThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gbn
