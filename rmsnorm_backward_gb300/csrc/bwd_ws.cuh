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
//  * warp 0, lane 0 (producer): first copies gamma (mbarrier `gbar`), then
//    issues row k into stage k mod S once every output warp has released row
//    k - S (mbarrier `consumed`, one arrival per output warp); the two
//    copies of a row complete the stage's `full` mbarrier.  Nothing is
//    loaded before the first copy is issued, so HBM is busy from the start.
//  * kSumWarps sum warps: every sum warp takes every row, in row order, and
//    sums its share of the row: 32-vector groups j, j + kSumWarps, ... (per
//    lane one partial sum per element position, a pairwise tree over the
//    positions, then a warp butterfly: a fixed order).  Saved statistics:
//    sum(dyhat) (LayerNorm) and sum(dyhat * (x - mean)).  None saved:
//    RMSNorm sum(x^2) and sum(dyhat * x); LayerNorm first sum(x) (the mean,
//    exchanged among the sum warps through a named barrier), then
//    sum((x - mean)^2), sum(dyhat), sum(dyhat * (x - mean)).  Lane 0 stores
//    the partials beside the stage (sum warp 0 also the row's saved rstd and
//    mean, loaded one row ahead, or the recomputed mean) and arrives on the
//    stage's `ready` mbarrier (one arrival per sum warp).
//  * kOutWarps output warps: warp o owns columns [o * VO * 32 * V, (o + 1) *
//    VO * 32 * V) of every row.  For each row in order it waits for `ready`,
//    adds the sum warps' partials in sum-warp order (the same bits in every
//    output warp), forms rstd (none saved) and c1 = mean(dyhat), c2 =
//    mean(dyhat * xhat), writes its slice of dx = dyhat*rstd + xhat*a + b with
//    16-byte streaming stores, adds dy*xhat (and dy) into its register
//    accumulators, and arrives on `consumed`.
// The output warps' columns are disjoint, so each stores its part of the
// CTA's partial row directly.  `ready` completing implies the stage landed;
// `consumed` completing implies every warp is done reading the stage.  All
// roles take rows in order, so each wait's parity is unambiguous.
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
    // partial sums a sum warp passes on per row
    constexpr int NQ = RECOMP && LN ? 3 : 2;
    extern __shared__ __align__(128) unsigned char smem[];

    const int N = p.N;
    const int groups = N / (32 * V);  // 32-vector groups of a row
    const int S = p.stages;
    const uint32_t rowb = static_cast<uint32_t>(N) * sizeof(T);
    const WsLayout L = ws_layout(rowb, S);
    unsigned char *ring = smem;
    const unsigned char *gam_s = smem + L.gam;
    float4 *cval = reinterpret_cast<float4 *>(smem + L.cval);  // [S][NS + 1]
    float *xch = reinterpret_cast<float *>(smem + L.xch);      // [2][NS], by row parity
    // [2], by row parity: a sum warp reads row k's flag after row k's
    // exchange while a faster one may already set row k + 1's
    volatile int *sum_abort = reinterpret_cast<volatile int *>(xch + 2 * NS);
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
            mbar_init(&ready[i], NS);
            mbar_init(&consumed[i], kOutWarps);
        }
        mbar_init(gbar, 1);
        sum_abort[0] = sum_abort[1] = 0;
        fence_barrier_init();
    }
    __syncthreads();
    griddep_launch_dependents();
    const float inv_n = 1.0f / static_cast<float>(N);
    const uint64_t wait_ns = p.wait_ns;

    if (warp == 0) {
        // ---- producer
        if (lane == 0) {
            mbar_arrive_expect_tx(gbar, rowb);
            bulk_load_nohint(const_cast<unsigned char *>(gam_s), p.gamma, rowb, gbar);
            int issued = 0;
            RingPos pos;
            for (; issued < nrows; ++issued) {
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
                pos.next(S);
            }
            // gamma and the copies of the last S issued rows have landed
            // before the CTA may exit (earlier rows' stages were released, so
            // they landed): normally these waits return at once; after an
            // abort they bound the wait for copies in flight
            bool drained = mbar_wait_bounded(gbar, 0, kDrainNs);
            for (int kk = issued - S > 0 ? issued - S : 0; drained && kk < issued; ++kk)
                drained = mbar_wait_bounded(&full[kk % S], static_cast<uint32_t>((kk / S) & 1), kDrainNs);
            if (!drained) record_error(p.err, kErrDrain);
        }
        return;
    }

    if (warp <= NS) {
        // ---- sum warp j: groups j, j + NS, ... of every row
        const int j = warp - 1;
        bool ok = warp_wait_bounded(gbar, 0, wait_ns);
        // the saved statistics, loaded one row ahead (sum warp 0 passes
        // rstd and mean on to the output warps)
        float mu_next = 0.f, rs_next = 0.f;
        if constexpr (!RECOMP) {
            if (nrows > 0) {
                if (LN) mu_next = p.mean[row0];
                if (j == 0) rs_next = p.rstd[row0];
            }
        }
        RingPos pos;
        for (int k = 0; k < nrows; ++k) {
            ok = ok && warp_wait_bounded(&full[pos.stage], pos.parity, wait_ns);
            if constexpr (!(RECOMP && LN)) {
                if (!ok) {
                    record_error(p.err, kErrWaitFull);
                    break;
                }
            }
            const unsigned char *sx = ring + (size_t)pos.stage * 2 * rowb;
            float mu = 0.f, rs = 0.f;
            if constexpr (!RECOMP) {
                mu = mu_next;
                rs = rs_next;
                if (k + 1 < nrows) {
                    if (LN) mu_next = p.mean[row0 + k + 1];
                    if (j == 0) rs_next = p.rstd[row0 + k + 1];
                }
            }
            if constexpr (RECOMP && LN) {
                // the mean first: this warp's share of sum(x), exchanged
                // with the other sum warps (a warp whose wait ran out still
                // joins the exchange, so none is left waiting; then all stop)
                float ax[V];
#pragma unroll
                for (int e = 0; e < V; ++e) ax[e] = 0.f;
                if (ok) {
                    for (int g = j; g < groups; g += NS) {
                        float xf[V];
                        Tr::unpack(ld_shared_v4(sx + (size_t)(g * 32 + lane) * 16), xf);
#pragma unroll
                        for (int e = 0; e < V; ++e) ax[e] += xf[e];
                    }
                }
#pragma unroll
                for (int w = 1; w < V; w *= 2)
#pragma unroll
                    for (int e = 0; e < V; e += 2 * w) ax[e] += ax[e + w];
                const float sx_part = warp_sum(ax[0]);
                if (lane == 0) {
                    xch[(k & 1) * NS + j] = sx_part;
                    if (!ok) sum_abort[k & 1] = 1;
                }
                named_barrier(1, 32 * NS);
                if (sum_abort[k & 1]) {
                    if (!ok) record_error(p.err, kErrWaitFull);
                    break;
                }
                float t = xch[(k & 1) * NS];
#pragma unroll
                for (int q = 1; q < NS; ++q) t += xch[(k & 1) * NS + q];
                mu = t * inv_n;
            }
            // one partial sum per element position (V chains of dependent
            // adds instead of one), added in a fixed order below
            float a0[V], a1[V], a2[NQ == 3 ? V : 1];
#pragma unroll
            for (int e = 0; e < V; ++e) {
                a0[e] = a1[e] = 0.f;
                if constexpr (NQ == 3) a2[e] = 0.f;
            }
            for (int g = j; g < groups; g += NS) {
                const int v = g * 32 + lane;
                float xf[V], df[V], gf[V];
                Tr::unpack(ld_shared_v4(sx + (size_t)v * 16), xf);
                Tr::unpack(ld_shared_v4(sx + rowb + (size_t)v * 16), df);
                Tr::unpack(ld_shared_v4(gam_s + (size_t)v * 16), gf);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float dyhat = df[e] * gf[e];
                    if constexpr (RECOMP && LN) {
                        const float d = xf[e] - mu;
                        a0[e] = fmaf(d, d, a0[e]);   // sum((x - mean)^2)
                        a1[e] += dyhat;              // sum(dyhat)
                        a2[e] = fmaf(dyhat, d, a2[e]);  // sum(dyhat * (x - mean))
                    } else if constexpr (RECOMP) {
                        a0[e] = fmaf(xf[e], xf[e], a0[e]);  // sum(x^2)
                        a1[e] = fmaf(dyhat, xf[e], a1[e]);  // sum(dyhat * x)
                    } else {
                        if constexpr (LN) a0[e] += dyhat;                    // sum(dyhat)
                        a1[e] = fmaf(dyhat, LN ? xf[e] - mu : xf[e], a1[e]);  // sum(dyhat * (x - mean))
                    }
                }
            }
#pragma unroll
            for (int w = 1; w < V; w *= 2) {
#pragma unroll
                for (int e = 0; e < V; e += 2 * w) {
                    a0[e] += a0[e + w];
                    a1[e] += a1[e + w];
                    if constexpr (NQ == 3) a2[e] += a2[e + w];
                }
            }
            float s0 = a0[0], s1 = a1[0], s2 = 0.f;
            if constexpr (!RECOMP && !LN) {
                s1 = warp_sum(s1);  // RMSNorm with saved rstd: no sum(dyhat)
            } else {
                warp_sum2(s0, s1);
                if constexpr (NQ == 3) s2 = warp_sum(a2[0]);
            }
            if (lane == 0) {
                cval[pos.stage * (NS + 1) + j] = make_float4(s0, s1, s2, 0.f);
                if (j == 0) cval[pos.stage * (NS + 1) + NS] = make_float4(rs, mu, 0.f, 0.f);
                mbar_arrive(&ready[pos.stage]);
            }
            pos.next(S);
        }
        return;
    }

    // ---- output warp o: columns [o * VO * 32, (o + 1) * VO * 32) in vectors
    const int o = warp - 1 - NS;
    bool ok = warp_wait_bounded(gbar, 0, wait_ns);
    if (!ok) record_error(p.err, kErrWaitFull);
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
        if (!warp_wait_bounded(&ready[pos.stage], pos.parity, wait_ns)) {
            record_error(p.err, kErrWaitFull);
            break;
        }
        const unsigned char *sx = ring + (size_t)pos.stage * 2 * rowb;
        // the sum warps' partials, added in sum-warp order
        const float4 *cv = cval + pos.stage * (NS + 1);
        float4 q = cv[0];
#pragma unroll
        for (int jj = 1; jj < NS; ++jj) {
            const float4 t = cv[jj];
            q.x += t.x;
            q.y += t.y;
            q.z += t.z;
        }
        const float4 stat = cv[NS];
        float rs, mu = stat.y, c1 = 0.f, c2;
        if constexpr (RECOMP && LN) {
            rs = 1.0f / sqrtf(q.x * inv_n + p.eps);
            c1 = q.y * inv_n;
            c2 = q.z * rs * inv_n;
        } else if constexpr (RECOMP) {
            rs = 1.0f / sqrtf(q.x * inv_n + p.eps);
            c2 = q.y * rs * inv_n;
        } else {
            rs = stat.x;
            if constexpr (LN) c1 = q.x * inv_n;
            c2 = q.y * rs * inv_n;
        }
        // c1 = mean(dyhat), c2 = mean(dyhat * xhat)
        const float a = -rs * c2;
        const float b = LN ? -rs * c1 : 0.f;
        T *dxrow = static_cast<T *>(p.dx) + (row0 + k) * p.ld_dx;
#pragma unroll
        for (int jv = 0; jv < VO; ++jv) {
            const int v = (o * VO + jv) * 32 + lane;
            float xf[V], df[V], out[V];
            Tr::unpack(ld_shared_v4(sx + (size_t)v * 16), xf);
            Tr::unpack(ld_shared_v4(sx + rowb + (size_t)v * 16), df);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                const float xhat = LN ? (xf[e] - mu) * rs : xf[e] * rs;
                acc_g[jv * V + e] = fmaf(df[e], xhat, acc_g[jv * V + e]);
                if constexpr (LN) acc_b[jv * V + e] += df[e];
                out[e] = fmaf(df[e] * gam[jv * V + e], rs, LN ? fmaf(xhat, a, b) : xhat * a);
            }
            st_global_cs_v4(dxrow + (size_t)v * V, Tr::pack(out));
        }
        // the warp's shared loads of the stage come before lane 0's release
        __syncwarp();
        if (lane == 0) mbar_arrive(&consumed[pos.stage]);
        pos.next(S);
    }
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
