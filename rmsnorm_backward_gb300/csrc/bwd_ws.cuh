// bwd_ws.cuh -- warp-specialised LayerNorm / RMSNorm backward for sm_103a,
// for rows that split into 16 warps x 32 lanes x 1-2 16-byte vectors.  Same
// definition as bwd_kernels.cuh ("Norm backward in Triton -- the dγ/dβ
// reduction", section "The gradients"; xhat recomputed from the saved mean /
// rstd, or, with no saved statistics, the statistics themselves formed from
// the staged row: "Norm & activation backward", section "Half one"; the
// per-CTA partial rows of "The hard half").
//
// One persistent CTA per SM owns a contiguous block of rows, streamed
// through a ring of S shared-memory stages (x row, dy row) by 1-D bulk
// copies.  The row's reductions and its elementwise output run in different
// warps, so no warp waits for a peer's share of a row:
//  * warp 0, lane 0 (producer): copies gamma first (mbarrier `gbar`), then
//    issues row k into stage k mod S once every output warp has released row
//    k - S (mbarrier `consumed`, one arrival per output warp); the two
//    copies of a row complete the stage's `full` mbarrier.  It starts as
//    soon as the barriers exist, so HBM is busy from the kernel's start.
//  * the other warps meanwhile stage the CTA's saved statistics in shared
//    memory (one named barrier among them).
//  * kSumWarps sum warps: sum warp j takes whole rows j, j + kSumWarps, ...
//    (several rows in flight, one per sum warp).  Saved statistics: it forms
//    sum(dyhat) (LayerNorm) and sum(dyhat * (x - mean)).  None saved: the
//    row's mean first (LayerNorm), then sum((x - mean)^2) or sum(x^2),
//    sum(dyhat) and sum(dyhat * (x - mean)), as the forward forms them.  Per
//    lane one partial sum per element position over the lane's vectors in
//    order, a pairwise tree over the positions, then a warp butterfly: a
//    fixed order.  Lane 0 stores the row's {rstd, mean, c1 = mean(dyhat),
//    c2 = mean(dyhat * xhat)} beside the stage and arrives on its `ready`
//    mbarrier.
//  * kOutWarps output warps: warp o owns columns [o * VO * 32 * V, (o + 1) *
//    VO * 32 * V) of every row.  For each row in order it waits for `ready`,
//    writes its slice of dx = dyhat*rstd + xhat*a + b with 16-byte streaming
//    stores, adds dy*xhat (and dy) into its register accumulators, and
//    arrives on `consumed`.
// The output warps' columns are disjoint, so each stores its part of the
// CTA's partial row directly.  `ready` completing implies the stage landed;
// `consumed` completing implies every warp is done reading the stage.
// Both the sum and the output warps do their float32 arithmetic in packed
// pairs of elements (fma / mul / add .f32x2): the same operations in the
// same order as the scalar form, so the same bits, in half the issues -- the
// sum warps share the SM's issue slots with the output warps and set the
// row rate, so fewer issues per row is a shorter kernel.
// Every wait is bounded (p.wait_ns, two seconds by default) and taken by all
// lanes of a warp with one outcome: a warp that gives up records the error
// and stops as a whole; the producer then waits (with its own bound) for its
// copies still in flight, so none lands after the CTA has exited.
#pragma once

#include "bwd_ws_layout.h"
#include "gbn_device.cuh"
#include "gbn_launch.h"

namespace gbn {

template <typename T, bool LN, int VO, bool RECOMP>
__global__ void __launch_bounds__(kWsThreads, 1) bwd_ws_kernel(const BwdParams p) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int E = VO * V;
    constexpr int NS = kSumWarps;
    extern __shared__ __align__(128) unsigned char smem[];

    const int N = p.N;
    const int nvec = N / V;
    const int S = p.stages;
    const uint32_t rowb = static_cast<uint32_t>(N) * sizeof(T);
    const WsLayout L = ws_layout(LN, rowb, S, p.stat_rows);
    unsigned char *ring = smem;
    unsigned char *gam_s = smem + L.gam;
    float *st_rstd = reinterpret_cast<float *>(smem + L.stat);
    float *st_mean = st_rstd + p.stat_rows;
    float4 *cval = reinterpret_cast<float4 *>(smem + L.cval);  // [S]: rstd, mean, c1, c2
    int *issued_count = reinterpret_cast<int *>(cval + S);     // rows the producer has issued
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *ready = full + S;
    uint64_t *consumed = ready + S;
    uint64_t *gbar = consumed + S;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t row0;
    int nrows;
    block_rows(p.M, p.G, blockIdx.x, row0, nrows);

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&ready[i], 1);
            mbar_init(&consumed[i], kOutWarps);
        }
        mbar_init(gbar, 1);
        *issued_count = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const float inv_n = 1.0f / static_cast<float>(N);
    const uint64_t wait_ns = p.wait_ns;

    if (warp == 0) {
        // ---- producer
        if (lane == 0) {
            mbar_arrive_expect_tx(gbar, rowb);
            bulk_load_nohint(gam_s, p.gamma, rowb, gbar);
            int issued = 0;
            bool triggered = false;
            RingPos pos;
            for (; issued < nrows; ++issued) {
                if (issued == S) {  // the ring is in flight: let the column reduce launch
                    griddep_launch_dependents();
                    triggered = true;
                }
                if (issued >= S &&
                    !mbar_wait_bounded(&consumed[pos.stage], pos.parity ^ 1u, wait_ns)) {  // row issued - S released
                    record_error(p.err, kErrWaitFull);
                    break;
                }
                const int64_t row = row0 + issued;
                unsigned char *dst = ring + (size_t)pos.stage * 2 * rowb;
                // the consumers' shared loads of the stage (seen through
                // `consumed`) come before the copy that overwrites it
                if (issued >= S) fence_proxy_async();
                mbar_arrive_expect_tx(&full[pos.stage], 2 * rowb);
                bulk_load_nohint(dst, static_cast<const T *>(p.x) + row * p.ld_x, rowb, &full[pos.stage]);
                bulk_load_nohint(dst + rowb, static_cast<const T *>(p.dy) + row * p.ld_dy, rowb, &full[pos.stage]);
                st_release_shared(issued_count, issued + 1);
                pos.next(S);
            }
            if (!triggered) griddep_launch_dependents();
            // gamma and the copies of the last S issued rows have landed
            // before the CTA may exit (earlier rows' stages were released, so
            // they landed): normally these waits return at once; after an
            // abort they bound the wait for copies in flight
            bool drained = mbar_wait_bounded(gbar, 0, kDrainNs);
            for (int kk = issued - S > 0 ? issued - S : 0; drained && kk < issued; ++kk)
                drained = mbar_wait_bounded(&full[kk % S], static_cast<uint32_t>((kk / S) & 1), kDrainNs);
            if (!drained) record_error(p.err, kErrDrain);
        } else {
            griddep_launch_dependents();
        }
        return;
    }

    // ---- the consumer warps: this CTA's saved statistics, staged while the
    // producer's first copies are in flight
    if constexpr (!RECOMP) {
        for (int i = tid - 32; i < nrows; i += static_cast<int>(blockDim.x) - 32) {
            st_rstd[i] = p.rstd[row0 + i];
            if (LN) st_mean[i] = p.mean[row0 + i];
        }
    }
    named_barrier(1, static_cast<int>(blockDim.x) - 32);
    griddep_launch_dependents();
    bool ok = warp_wait_bounded(gbar, 0, wait_ns);  // gamma landed

    if (warp <= NS) {
        // ---- sum warp j takes rows j, j + NS, ...
        const int j = warp - 1;
        for (int k = j; ok && k < nrows; k += NS) {
            const int st = k % S;
            // Sum warps do not take rows in order, so this one may reach row k
            // while the stage still holds row k - S, whose phase of `full`
            // has the other parity: a wait on row k's parity would then pass
            // at once.  Row k is issued only after row k - S was consumed,
            // hence landed; once it is issued the parity is unambiguous.
            ok = ok && __all_sync(0xffffffffu, wait_counter_above(issued_count, k, wait_ns)) &&
                 warp_wait_bounded(&full[st], static_cast<uint32_t>((k / S) & 1), wait_ns);
            if (!ok) break;
            const unsigned char *sx = ring + (size_t)st * 2 * rowb;
            float rs, mu = 0.f, c1, c2;
            if constexpr (RECOMP) {
                // no saved statistics: the mean first (LayerNorm), then the
                // centred squares and the two sums of the backward
                if constexpr (LN) {
                    float2 axp[V / 2];
#pragma unroll
                    for (int i = 0; i < V / 2; ++i) axp[i] = make_float2(0.f, 0.f);
#pragma unroll 2
                    for (int v = lane; v < nvec; v += 32) {
                        float xf[V];
                        Tr::unpack(ld_shared_v4(sx + (size_t)v * 16), xf);
#pragma unroll
                        for (int i = 0; i < V / 2; ++i) axp[i] = pair_add(axp[i], pair_at(xf, i));
                    }
                    float ax[V];
#pragma unroll
                    for (int i = 0; i < V / 2; ++i) ax[2 * i] = axp[i].x, ax[2 * i + 1] = axp[i].y;
#pragma unroll
                    for (int w = 1; w < V; w *= 2)
#pragma unroll
                        for (int e = 0; e < V; e += 2 * w) ax[e] += ax[e + w];
                    mu = warp_sum(ax[0]) * inv_n;
                }
                // sum((x - mean)^2), sum(dyhat), sum(dyhat * (x - mean)), in
                // pairs of element positions
                float2 qp[V / 2], d1p[V / 2], d2p[V / 2];
#pragma unroll
                for (int i = 0; i < V / 2; ++i) qp[i] = d1p[i] = d2p[i] = make_float2(0.f, 0.f);
                const float2 nmu = make_float2(-mu, -mu);
#pragma unroll 2
                for (int v = lane; v < nvec; v += 32) {
                    float xf[V], df[V], gf[V];
                    Tr::unpack(ld_shared_v4(sx + (size_t)v * 16), xf);
                    Tr::unpack(ld_shared_v4(sx + rowb + (size_t)v * 16), df);
                    Tr::unpack(ld_shared_v4(gam_s + (size_t)v * 16), gf);
#pragma unroll
                    for (int i = 0; i < V / 2; ++i) {
                        const float2 d = LN ? pair_add(pair_at(xf, i), nmu) : pair_at(xf, i);
                        const float2 dyhat = pair_mul(pair_at(df, i), pair_at(gf, i));
                        qp[i] = pair_fma(d, d, qp[i]);
                        if constexpr (LN) d1p[i] = pair_add(d1p[i], dyhat);
                        d2p[i] = pair_fma(dyhat, d, d2p[i]);
                    }
                }
                float q[V], d1[V], d2[V];
#pragma unroll
                for (int i = 0; i < V / 2; ++i) {
                    q[2 * i] = qp[i].x, q[2 * i + 1] = qp[i].y;
                    d1[2 * i] = d1p[i].x, d1[2 * i + 1] = d1p[i].y;
                    d2[2 * i] = d2p[i].x, d2[2 * i + 1] = d2p[i].y;
                }
#pragma unroll
                for (int w = 1; w < V; w *= 2) {
#pragma unroll
                    for (int e = 0; e < V; e += 2 * w) {
                        q[e] += q[e + w];
                        if constexpr (LN) d1[e] += d1[e + w];
                        d2[e] += d2[e + w];
                    }
                }
                float sq = q[0], s1 = d2[0], s0 = LN ? d1[0] : 0.f;
                warp_sum2(sq, s1);
                if constexpr (LN) s0 = warp_sum(s0);
                rs = 1.0f / sqrtf(sq * inv_n + p.eps);
                c1 = s0 * inv_n;
                c2 = s1 * rs * inv_n;
            } else {
                rs = st_rstd[k];
                mu = LN ? st_mean[k] : 0.f;
                // one partial sum per element position of a vector (V chains
                // of dependent adds instead of one), added in a fixed order,
                // in pairs of positions
                float2 a0p[V / 2], a1p[V / 2];  // sum(dyhat), sum(dyhat * (x - mean))
#pragma unroll
                for (int i = 0; i < V / 2; ++i) a0p[i] = a1p[i] = make_float2(0.f, 0.f);
                const float2 nmu = make_float2(-mu, -mu);
#pragma unroll 2
                for (int v = lane; v < nvec; v += 32) {
                    float xf[V], df[V], gf[V];
                    Tr::unpack(ld_shared_v4(sx + (size_t)v * 16), xf);
                    Tr::unpack(ld_shared_v4(sx + rowb + (size_t)v * 16), df);
                    Tr::unpack(ld_shared_v4(gam_s + (size_t)v * 16), gf);
#pragma unroll
                    for (int i = 0; i < V / 2; ++i) {
                        const float2 dyhat = pair_mul(pair_at(df, i), pair_at(gf, i));
                        if constexpr (LN) a0p[i] = pair_add(a0p[i], dyhat);
                        a1p[i] = pair_fma(dyhat, LN ? pair_add(pair_at(xf, i), nmu) : pair_at(xf, i), a1p[i]);
                    }
                }
                float a0[LN ? V : 1], a1[V];
#pragma unroll
                for (int i = 0; i < V / 2; ++i) {
                    a1[2 * i] = a1p[i].x, a1[2 * i + 1] = a1p[i].y;
                    if constexpr (LN) a0[2 * i] = a0p[i].x, a0[2 * i + 1] = a0p[i].y;
                }
#pragma unroll
                for (int w = 1; w < V; w *= 2) {
#pragma unroll
                    for (int e = 0; e < V; e += 2 * w) {
                        a1[e] += a1[e + w];
                        if constexpr (LN) a0[e] += a0[e + w];
                    }
                }
                float s0 = 0.f, s1 = a1[0];
                if constexpr (LN) {
                    s0 = a0[0];
                    warp_sum2(s0, s1);
                } else {
                    s1 = warp_sum(s1);
                }
                c1 = s0 * inv_n;
                c2 = s1 * rs * inv_n;
            }
            if (lane == 0) {
                cval[st] = make_float4(rs, mu, c1, c2);
                mbar_arrive(&ready[st]);
            }
        }
        if (!ok) record_error(p.err, kErrWaitFull);
        return;
    }

    // ---- output warp o: columns [o * VO * 32, (o + 1) * VO * 32) in vectors
    const int o = warp - 1 - NS;
    float gam[E], acc_g[E], acc_b[LN ? E : 1];
#pragma unroll
    for (int jv = 0; jv < VO; ++jv) {
        if (ok)
            Tr::unpack(ld_shared_v4(gam_s + (size_t)((o * VO + jv) * 32 + lane) * 16), gam + jv * V);
        else
#pragma unroll
            for (int e = 0; e < V; ++e) gam[jv * V + e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
        acc_g[e] = 0.f;
        if constexpr (LN) acc_b[e] = 0.f;
    }
    RingPos pos;
    for (int k = 0; ok && k < nrows; ++k) {
        ok = warp_wait_bounded(&ready[pos.stage], pos.parity, wait_ns);
        if (!ok) break;
        const unsigned char *sx = ring + (size_t)pos.stage * 2 * rowb;
        const float4 cv = cval[pos.stage];
        const float rs = cv.x, mu = cv.y;
        const float a = -rs * cv.w;             // -rstd * c2
        const float b = LN ? -rs * cv.z : 0.f;  // -rstd * c1
        const float2 rs2 = make_float2(rs, rs), a2 = make_float2(a, a), b2 = make_float2(b, b);
        const float2 nmu2 = make_float2(-mu, -mu);
        T *dxrow = static_cast<T *>(p.dx) + (row0 + k) * p.ld_dx;
#pragma unroll
        for (int jv = 0; jv < VO; ++jv) {
            const int v = (o * VO + jv) * 32 + lane;
            float xf[V], df[V], out[V];
            Tr::unpack(ld_shared_v4(sx + (size_t)v * 16), xf);
            Tr::unpack(ld_shared_v4(sx + rowb + (size_t)v * 16), df);
            // in pairs of elements: xhat, the dgamma (dbeta) accumulators and
            // dx = (dy*gamma)*rstd + (xhat*a + b)
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                const int e = jv * V + 2 * i;
                const float2 d2 = pair_at(df, i);
                const float2 xh = LN ? pair_mul(pair_add(pair_at(xf, i), nmu2), rs2) : pair_mul(pair_at(xf, i), rs2);
                const float2 ag = pair_fma(d2, xh, make_float2(acc_g[e], acc_g[e + 1]));
                acc_g[e] = ag.x, acc_g[e + 1] = ag.y;
                if constexpr (LN) {
                    const float2 ab = pair_add(make_float2(acc_b[e], acc_b[e + 1]), d2);
                    acc_b[e] = ab.x, acc_b[e + 1] = ab.y;
                }
                const float2 dg = pair_mul(d2, make_float2(gam[e], gam[e + 1]));
                const float2 o2 = pair_fma(dg, rs2, LN ? pair_fma(xh, a2, b2) : pair_mul(xh, a2));
                out[2 * i] = o2.x, out[2 * i + 1] = o2.y;
            }
            st_global_cs_v4(dxrow + (size_t)v * V, Tr::pack(out));
        }
        // the warp's shared loads of the stage come before lane 0's release
        __syncwarp();
        if (lane == 0) mbar_arrive(&consumed[pos.stage]);
        pos.next(S);
    }
    if (!ok) record_error(p.err, kErrWaitFull);
    // this CTA's partial row: the warp's own columns (with p.atom_g set, the
    // atomics ablation, added into dgamma / dbeta instead)
    const bool atomic = p.atom_g != nullptr;
    float *pg = atomic ? p.atom_g : p.part + (size_t)blockIdx.x * p.ldp;
    float *pb = atomic ? p.atom_b
                       : (p.part_b ? p.part_b : p.part + (size_t)p.G * p.ldp) + (size_t)blockIdx.x * p.ldp;
    auto put = [atomic](float *dst, const float *v) {
        if (atomic) {
#pragma unroll
            for (int q = 0; q < 4; ++q) atomicAdd(dst + q, v[q]);
        } else {
            *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        }
    };
#pragma unroll
    for (int jv = 0; jv < VO; ++jv) {
        const int v = (o * VO + jv) * 32 + lane;
#pragma unroll
        for (int e = 0; e < V; e += 4) {
            put(pg + (size_t)v * V + e, acc_g + jv * V + e);
            if constexpr (LN) put(pb + (size_t)v * V + e, acc_b + jv * V + e);
        }
    }
}

template <typename T, bool LN, int VO, bool RECOMP>
cudaError_t bwd_ws_launch_vo(const BwdParams &p, size_t smem, cudaStream_t s) {
    static std::atomic<uint64_t> done{0};
    cudaError_t e = ensure_smem_optin(bwd_ws_kernel<T, LN, VO, RECOMP>, done);
    if (e != cudaSuccess) return e;
    bwd_ws_kernel<T, LN, VO, RECOMP><<<p.G, kWsThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// recompute: no saved statistics (p.rstd == nullptr), formed from x with p.eps
template <typename T, bool LN, int VO>
cudaError_t bwd_ws_launch_r(const BwdParams &p, size_t smem, cudaStream_t s) {
    return p.rstd ? bwd_ws_launch_vo<T, LN, VO, false>(p, smem, s) : bwd_ws_launch_vo<T, LN, VO, true>(p, smem, s);
}

template <typename T>
cudaError_t bwd_ws_dispatch(bool ln, int vo, const BwdParams &p, size_t smem, cudaStream_t s) {
    switch (vo) {
        case 1: return ln ? bwd_ws_launch_r<T, true, 1>(p, smem, s) : bwd_ws_launch_r<T, false, 1>(p, smem, s);
        case 2: return ln ? bwd_ws_launch_r<T, true, 2>(p, smem, s) : bwd_ws_launch_r<T, false, 2>(p, smem, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbn
