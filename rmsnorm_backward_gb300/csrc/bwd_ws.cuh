// bwd_ws.cuh -- warp-specialised LayerNorm / RMSNorm backward for sm_103a,
// for saved statistics and rows that split into whole warps of 16-byte
// vectors.  Same definition as bwd_kernels.cuh ("Norm backward in Triton --
// the dγ/dβ reduction", section "The gradients"; xhat recomputed from the
// saved mean / rstd, "Norm & activation backward", section "Half one"; the
// per-CTA partial rows of "The hard half").
//
// One persistent CTA per SM owns a contiguous block of rows, streamed
// through a ring of S shared-memory stages (x row, dy row) by 1-D bulk
// copies.  The row's two reductions and its elementwise output run in
// different warps, so no warp waits for a peer's share of a row:
//  * warp 0, lane 0 (producer): issues row k into stage k mod S once every
//    output warp has released row k - S (mbarrier `consumed`, one arrival
//    per output warp); the copies complete the stage's `full` mbarrier.
//  * kSumWarps sum warps: warp j takes rows j, j + kSumWarps, ...; it waits
//    for `full`, forms sum(dyhat) and sum(dyhat*xhat) over the whole row
//    (per lane one partial sum per element position over the lane's vectors
//    in order, a pairwise tree over the positions, then a warp butterfly: a
//    fixed order), stores them beside the stage and arrives on the stage's
//    `ready` mbarrier.
//  * NO output warps: warp o owns columns [o * VO * 32 * V, (o + 1) * VO *
//    32 * V) for every row.  For each row in order it waits for `ready`,
//    writes its slice of dx = dyhat*rstd + xhat*a + b with 16-byte streaming
//    stores, adds dy*xhat (and dy) into its register accumulators, and
//    arrives on `consumed`.
// The output warps' columns are disjoint, so each stores its part of the
// CTA's partial row directly.  `ready` completing implies the stage landed;
// `consumed` completing implies every warp is done reading the stage.
// Every wait is bounded (2 s): a warp that gives up records the error and
// stops; the producer then waits (bounded) for its copies still in flight.
#pragma once

#include "bwd_ws_layout.h"
#include "gbn_device.cuh"
#include "gbn_launch.h"

namespace gbn {

template <typename T, bool LN, int VO>
__global__ void __launch_bounds__(32 * (1 + kSumWarps + 16), 1) bwd_ws_kernel(const BwdParams p) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int E = VO * V;
    extern __shared__ __align__(128) unsigned char smem[];

    const int N = p.N;
    const int nvec = N / V;
    const int S = p.stages;
    const size_t rowb = (size_t)N * sizeof(T);
    const int NO = static_cast<int>(blockDim.x / 32) - 1 - kSumWarps;
    const WsLayout L = ws_layout(LN, rowb, S, p.stat_rows);
    unsigned char *ring = smem;
    const unsigned char *gam_s = smem + L.gam;
    float *st_rstd = reinterpret_cast<float *>(smem + L.stat);
    float *st_mean = st_rstd + p.stat_rows;
    float *cval = reinterpret_cast<float *>(smem + L.cval);
    int *issued_count = reinterpret_cast<int *>(cval + 2 * S);  // rows the producer has issued
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *ready = full + S;
    uint64_t *consumed = ready + S;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t row0;
    int nrows;
    block_rows(p.M, p.G, blockIdx.x, row0, nrows);

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&ready[i], 1);
            mbar_init(&consumed[i], static_cast<uint32_t>(NO));
        }
        fence_barrier_init();
        *issued_count = 0;
    }
    // gamma (raw) and this CTA's statistics, staged once
    for (int v = tid; v < nvec; v += blockDim.x)
        *reinterpret_cast<uint4 *>(const_cast<unsigned char *>(gam_s) + (size_t)v * 16) =
            ld_global_nc_v4(static_cast<const T *>(p.gamma) + (size_t)v * V);
    for (int i = tid; i < nrows; i += blockDim.x) {
        st_rstd[i] = p.rstd[row0 + i];
        if (LN) st_mean[i] = p.mean[row0 + i];
    }
    __syncthreads();
    griddep_launch_dependents();
    const float inv_n = 1.0f / static_cast<float>(N);

    if (warp == 0) {
        // ---- producer
        if (lane == 0) {
            int issued = 0;
            RingPos pos;
            bool dead = false;
            for (; issued < nrows; ++issued) {
                if (issued >= S &&
                    !mbar_wait_bounded(&consumed[pos.stage], pos.parity ^ 1u)) {  // row issued - S released
                    record_error(p.err, kErrWaitFull);
                    dead = true;
                    break;
                }
                const int64_t row = row0 + issued;
                unsigned char *dst = ring + (size_t)pos.stage * 2 * rowb;
                // the consumers' shared loads of the stage (seen through
                // `consumed`) come before the copy that overwrites it
                if (issued >= S) fence_proxy_async();
                mbar_arrive_expect_tx(&full[pos.stage], static_cast<uint32_t>(2 * rowb));
                bulk_load_nohint(dst, static_cast<const T *>(p.x) + row * p.ld_x, static_cast<uint32_t>(rowb),
                                 &full[pos.stage]);
                bulk_load_nohint(dst + rowb, static_cast<const T *>(p.dy) + row * p.ld_dy,
                                 static_cast<uint32_t>(rowb), &full[pos.stage]);
                st_release_shared(issued_count, issued + 1);
                pos.next(S);
            }
            // the copies of the last S issued rows have landed before the CTA
            // may exit (earlier rows' stages were released, so they landed):
            // normally the sum warps saw them all and these waits return at
            // once; after an abort they bound the wait for copies in flight
            (void)dead;
            for (int kk = issued - S > 0 ? issued - S : 0; kk < issued; ++kk) {
                if (!mbar_wait_bounded(&full[kk % S], static_cast<uint32_t>((kk / S) & 1), 100000000ull)) {
                    record_error(p.err, kErrDrain);
                    break;
                }
            }
        }
        return;
    }

    if (warp <= kSumWarps) {
        // ---- sum warp j takes rows j, j + kSumWarps, ...
        const int j = warp - 1;
        for (int k = j; k < nrows; k += kSumWarps) {
            const int st = k % S;
            // Sum warps do not take rows in order, so this one may reach row k
            // while the stage still holds row k - S, whose phase of `full`
            // has the other parity: a wait on row k's parity would then pass
            // at once.  Row k is issued only after row k - S was consumed,
            // hence landed; once it is issued the parity is unambiguous.
            if (!wait_counter_above(issued_count, k) ||
                !mbar_wait_bounded(&full[st], static_cast<uint32_t>((k / S) & 1))) {
                record_error(p.err, kErrWaitFull);
                break;
            }
            const unsigned char *sx = ring + (size_t)st * 2 * rowb;
            const float rs = st_rstd[k];
            const float mu = LN ? st_mean[k] : 0.f;
            // one partial sum per element position of a vector (V chains of
            // dependent adds instead of one), added in a fixed order below
            float a0[LN ? V : 1], a1[V];  // sum(dyhat), sum(dyhat * (x - mean))
#pragma unroll
            for (int e = 0; e < V; ++e) {
                a1[e] = 0.f;
                if constexpr (LN) a0[e] = 0.f;
            }
#pragma unroll 2
            for (int v = lane; v < nvec; v += 32) {
                float xf[V], df[V], gf[V];
                Tr::unpack(ld_shared_v4(sx + (size_t)v * 16), xf);
                Tr::unpack(ld_shared_v4(sx + rowb + (size_t)v * 16), df);
                Tr::unpack(ld_shared_v4(gam_s + (size_t)v * 16), gf);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float dyhat = df[e] * gf[e];
                    if constexpr (LN) a0[e] += dyhat;
                    a1[e] = fmaf(dyhat, LN ? xf[e] - mu : xf[e], a1[e]);
                }
            }
#pragma unroll
            for (int w = 1; w < V; w *= 2) {
#pragma unroll
                for (int e = 0; e < V; e += 2 * w) {
                    a1[e] += a1[e + w];
                    if constexpr (LN) a0[e] += a0[e + w];
                }
            }
            float s0 = LN ? a0[0] : 0.f, s1 = a1[0];
            if constexpr (LN)
                warp_sum2(s0, s1);
            else
                s1 = warp_sum(s1);
            if (lane == 0) {
                // c1 = mean(dyhat), c2 = mean(dyhat * xhat)
                cval[2 * st] = s0 * inv_n;
                cval[2 * st + 1] = s1 * rs * inv_n;
                mbar_arrive(&ready[st]);
            }
        }
        return;
    }

    // ---- output warp o: columns [o * VO * 32, (o + 1) * VO * 32) in vectors
    const int o = warp - 1 - kSumWarps;
    // gamma in registers, except at 4 vectors a lane, where the accumulators
    // need the registers and gamma is read from shared memory every row
    constexpr bool GREG = VO <= 2;
    float gam[GREG ? E : 1], acc_g[E], acc_b[LN ? E : 1];
    if constexpr (GREG) {
#pragma unroll
        for (int jv = 0; jv < VO; ++jv)
            Tr::unpack(ld_shared_v4(gam_s + (size_t)((o * VO + jv) * 32 + lane) * 16), gam + jv * V);
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
        acc_g[e] = 0.f;
        if constexpr (LN) acc_b[e] = 0.f;
    }
    RingPos pos;
    for (int k = 0; k < nrows; ++k) {
        if (!mbar_wait_bounded(&ready[pos.stage], pos.parity)) {
            record_error(p.err, kErrWaitFull);
            break;
        }
        const unsigned char *sx = ring + (size_t)pos.stage * 2 * rowb;
        const float c1 = cval[2 * pos.stage], c2 = cval[2 * pos.stage + 1];
        const float rs = st_rstd[k];
        const float mu = LN ? st_mean[k] : 0.f;
        const float a = -rs * c2;
        const float b = LN ? -rs * c1 : 0.f;
        T *dxrow = static_cast<T *>(p.dx) + (row0 + k) * p.ld_dx;
#pragma unroll
        for (int jv = 0; jv < VO; ++jv) {
            const int v = (o * VO + jv) * 32 + lane;
            float xf[V], df[V], gf[V], out[V];
            Tr::unpack(ld_shared_v4(sx + (size_t)v * 16), xf);
            Tr::unpack(ld_shared_v4(sx + rowb + (size_t)v * 16), df);
            if constexpr (!GREG) Tr::unpack(ld_shared_v4(gam_s + (size_t)v * 16), gf);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                const float g = GREG ? gam[jv * V + e] : gf[e];
                const float xhat = LN ? (xf[e] - mu) * rs : xf[e] * rs;
                acc_g[jv * V + e] = fmaf(df[e], xhat, acc_g[jv * V + e]);
                if constexpr (LN) acc_b[jv * V + e] += df[e];
                out[e] = fmaf(df[e] * g, rs, LN ? fmaf(xhat, a, b) : xhat * a);
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

template <typename T, bool LN, int VO>
cudaError_t bwd_ws_launch_vo(const BwdParams &p, int threads, size_t smem, cudaStream_t s) {
    static std::atomic<uint64_t> done{0};
    cudaError_t e = ensure_smem_optin(bwd_ws_kernel<T, LN, VO>, done);
    if (e != cudaSuccess) return e;
    bwd_ws_kernel<T, LN, VO><<<p.G, threads, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_ws_dispatch(bool ln, int vo, const BwdParams &p, int threads, size_t smem, cudaStream_t s) {
    switch (vo) {
        case 1: return ln ? bwd_ws_launch_vo<T, true, 1>(p, threads, smem, s) : bwd_ws_launch_vo<T, false, 1>(p, threads, smem, s);
        case 2: return ln ? bwd_ws_launch_vo<T, true, 2>(p, threads, smem, s) : bwd_ws_launch_vo<T, false, 2>(p, threads, smem, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbn
