// norm_bwd.cu -- LayerNorm / RMSNorm backward kernels for sm_103a.
//
// Definition followed: "Norm backward in Triton -- the dγ/dβ reduction",
// section "The gradients": with dyhat = dy*gamma,
//   dx = rstd*(dyhat - mean(dyhat) - xhat*mean(dyhat*xhat))   (RMSNorm: no
//   mean(dyhat) term), dgamma = sum over rows of dy*xhat, dbeta = sum of dy.
// xhat is recomputed from the saved per-row mean / rstd, never stored
// ("Norm & activation backward", section "Half one").  dgamma / dbeta use the
// disjoint-row-block scheme of "Norm backward in Triton", section "The hard
// half": each CTA owns a contiguous block of rows, accumulates its partial
// sums in registers and stores one partial row (no atomics); a second kernel
// sums the partial rows per column in a fixed order.
//
// Kernels:
//  * staged (bwd_staged_kernel): one persistent CTA per SM; its rows are
//    spread over slots of tpr threads.  Each slot streams x and dy rows
//    through a ring of shared-memory stages filled by 1-D bulk (TMA) copies.
//    A thread owns fixed 16-byte column vectors: it reads its vectors of x
//    and dy from the stage, forms the two in-row sums (warp shuffles plus one
//    named barrier), reads them again to write dx with 16-byte stores (the
//    stage is refilled once the slot's next barrier shows that every thread
//    is done with it), and keeps fp32
//    accumulators of dy*xhat and dy for its columns over all the slot's
//    rows.  At the end the slots' accumulators are added in slot order in
//    shared memory and the CTA stores its partial row.
//  * plain (bwd_plain_kernel): any N and alignment, scalar loads, the CTA's
//    own partial row in global memory as the accumulator.
//  * colsum_kernel: dgamma[j] = sum over g of part[g][j] in a fixed order.
#include "gbn_device.cuh"
#include "gbn_launch.h"

namespace gbn {

static __device__ int g_error_flag = 0;

template <typename T, bool LN, int NV, bool HOLD>
__global__ void __launch_bounds__(kRingThreads, 1) bwd_staged_kernel(const BwdParams p) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int E = NV * V;  // elements a thread owns per row
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

    const RingLayout L = ring_layout(true, LN, sizeof(T), N, tpr, S, p.stat_rows, blockDim.x);
    unsigned char *ring = smem + L.ring_off + (size_t)slot * S * stage_bytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bar_off) + slot * S;
    float *st_rstd = reinterpret_cast<float *>(smem + L.stat_off);
    float *st_mean = st_rstd + p.stat_rows;
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
    const T *dyg = static_cast<const T *>(p.dy);
    auto issue = [&](int k) {
        const int st = k % S;
        const int64_t row = row0 + slot + (int64_t)k * slots;
        unsigned char *dst = ring + (size_t)st * stage_bytes;
        mbar_arrive_expect_tx(&bar[st], stage_bytes);
        bulk_load(dst, xg + row * N, rowb, &bar[st], pol);
        bulk_load(dst + rowb, dyg + row * N, rowb, &bar[st], pol);
    };
    int issued = 0;
    if (ts == 0) {
        for (; issued < S && issued < ns; ++issued) issue(issued);
    }

    // this CTA's saved statistics, staged once
    for (int i = tid; i < nrows; i += blockDim.x) {
        st_rstd[i] = p.rstd[row0 + i];
        if (LN) st_mean[i] = p.mean[row0 + i];
    }
    // gamma: unpacked once (HOLD) or kept as raw vectors
    float gam[HOLD ? E : 1];
    uint4 graw[HOLD ? 1 : NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int v = ts + j * tpr;
        const uint4 g = v < nvec ? ld_global_nc_v4(static_cast<const T *>(p.gamma) + (size_t)v * V)
                                 : make_uint4(0, 0, 0, 0);
        if constexpr (HOLD)
            Tr::unpack(g, gam + j * V);
        else
            graw[j] = g;
    }
    float acc_g[E], acc_b[LN ? E : 1];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        acc_g[e] = 0.f;
        if constexpr (LN) acc_b[e] = 0.f;
    }
    __syncthreads();
    griddep_launch_dependents();

    const float fn = static_cast<float>(N);
    int k = 0;
    for (; k < ns; ++k) {
        const int st = k % S;
        const bool timed_out = !mbar_wait_bounded(&bar[st], (k / S) & 1);
        if (timed_out) record_error(p.err, kErrWaitFull);
        const int i = slot + k * slots;
        const float rs = st_rstd[i];
        const float mu = LN ? st_mean[i] : 0.f;
        const unsigned char *sx = ring + (size_t)st * stage_bytes;
        // pass 1 over the staged row: the two in-row sums, the per-column
        // accumulators of dy*xhat and dy, and (HOLD) xhat, dyhat kept in
        // registers for pass 2
        float xh[HOLD ? E : 1], dh[HOLD ? E : 1];
        float s[2] = {0.f, 0.f};  // sum(dyhat), sum(dyhat*xhat)
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int v = ts + j * tpr;
            float xf[V], df[V], gl[V];
            if (v < nvec) {
                Tr::unpack(*reinterpret_cast<const uint4 *>(sx + (size_t)v * 16), xf);
                Tr::unpack(*reinterpret_cast<const uint4 *>(sx + rowb + (size_t)v * 16), df);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) xf[e] = df[e] = 0.f;
            }
            if constexpr (!HOLD) Tr::unpack(graw[j], gl);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                const float g = HOLD ? gam[j * V + e] : gl[e];
                const float xhat = LN ? (xf[e] - mu) * rs : xf[e] * rs;
                const float dyhat = df[e] * g;
                if constexpr (LN) s[0] += dyhat;
                s[1] = fmaf(dyhat, xhat, s[1]);
                acc_g[j * V + e] = fmaf(df[e], xhat, acc_g[j * V + e]);
                if constexpr (LN) acc_b[j * V + e] += df[e];
                if constexpr (HOLD) {
                    xh[j * V + e] = xhat;
                    dh[j * V + e] = dyhat;
                }
            }
        }
        const bool abort = slot_reduce<2>(s, red + (k & 1) * W * 2, flag, timed_out, W, warp, lane, 1 + slot, tpr);
        if (abort) break;
        // HOLD: the slot is done with this stage; otherwise it re-reads this
        // stage in pass 2 and the previous stage is the one now free
        if (ts == 0 && issued < ns && (HOLD || k > 0)) {
            fence_proxy_async();
            issue(issued++);
        }
        // pass 2: dx = rstd*(dyhat - c1 - xhat*c2) = dyhat*rstd + xhat*a + b
        const float a = -rs * (s[1] / fn);
        const float b = LN ? -rs * (s[0] / fn) : 0.f;
        T *dxrow = static_cast<T *>(p.dx) + (row0 + i) * N;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int v = ts + j * tpr;
            if (v < nvec) {
                float o[V];
                if constexpr (HOLD) {
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        o[e] = fmaf(dh[j * V + e], rs, LN ? fmaf(xh[j * V + e], a, b) : xh[j * V + e] * a);
                } else {
                    float xf[V], df[V], gl[V];
                    Tr::unpack(*reinterpret_cast<const uint4 *>(sx + (size_t)v * 16), xf);
                    Tr::unpack(*reinterpret_cast<const uint4 *>(sx + rowb + (size_t)v * 16), df);
                    Tr::unpack(graw[j], gl);
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float xhat = LN ? (xf[e] - mu) * rs : xf[e] * rs;
                        o[e] = fmaf(df[e] * gl[e], rs, LN ? fmaf(xhat, a, b) : xhat * a);
                    }
                }
                st_global_cs_v4(dxrow + (size_t)v * V, Tr::pack(o));
            }
        }
    }
    if (ts == 0) {
        for (int kk = k; kk < issued; ++kk) {
            if (!mbar_wait_bounded(&bar[kk % S], (kk / S) & 1, 100000000ull)) {
                record_error(p.err, kErrDrain);
                break;
            }
        }
    }

    // ---- this CTA's partial row(s) --------------------------------------
    const int ldp = p.ldp;
    float *pg = p.part + (size_t)blockIdx.x * ldp;
    float *pb = p.part + ((size_t)p.G + blockIdx.x) * ldp;
    if (slots == 1) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int v = ts + j * tpr;
            if (v < nvec) {
#pragma unroll
                for (int e = 0; e < V; e += 4) {
                    *reinterpret_cast<float4 *>(pg + (size_t)v * V + e) =
                        make_float4(acc_g[j * V + e], acc_g[j * V + e + 1], acc_g[j * V + e + 2], acc_g[j * V + e + 3]);
                    if constexpr (LN)
                        *reinterpret_cast<float4 *>(pb + (size_t)v * V + e) = make_float4(
                            acc_b[j * V + e], acc_b[j * V + e + 1], acc_b[j * V + e + 2], acc_b[j * V + e + 3]);
                }
            }
        }
        return;
    }
    // several slots: add their accumulators in slot order, in shared memory
    __syncthreads();  // every slot is done with its ring stages
    float *comb = reinterpret_cast<float *>(smem + L.ring_off);
    float *comb_g = comb + (size_t)slot * ldp;
    float *comb_b = comb + ((size_t)slots + slot) * ldp;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int v = ts + j * tpr;
        if (v < nvec) {
#pragma unroll
            for (int e = 0; e < V; e += 4) {
                *reinterpret_cast<float4 *>(comb_g + (size_t)v * V + e) =
                    make_float4(acc_g[j * V + e], acc_g[j * V + e + 1], acc_g[j * V + e + 2], acc_g[j * V + e + 3]);
                if constexpr (LN)
                    *reinterpret_cast<float4 *>(comb_b + (size_t)v * V + e) =
                        make_float4(acc_b[j * V + e], acc_b[j * V + e + 1], acc_b[j * V + e + 2], acc_b[j * V + e + 3]);
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
        *reinterpret_cast<float4 *>(pg + c) = a;
        if (LN) {
            const float *cb = comb + (size_t)slots * ldp;
            float4 d = *reinterpret_cast<const float4 *>(cb + c);
            for (int s2 = 1; s2 < slots; ++s2) {
                const float4 b = *reinterpret_cast<const float4 *>(cb + (size_t)s2 * ldp + c);
                d.x += b.x; d.y += b.y; d.z += b.z; d.w += b.w;
            }
            *reinterpret_cast<float4 *>(pb + c) = d;
        }
    }
}

template <typename T, bool LN>
__global__ void __launch_bounds__(kGenericThreads) bwd_plain_kernel(const BwdParams p) {
    using Tr = Traits<T>;
    __shared__ float sm[kGenericThreads / 32];
    const int N = p.N;
    const float fn = static_cast<float>(N);
    int64_t row0;
    int nrows;
    block_rows(p.M, p.G, blockIdx.x, row0, nrows);
    float *pg = p.part + (size_t)blockIdx.x * p.ldp;
    float *pb = p.part + ((size_t)p.G + blockIdx.x) * p.ldp;
    griddep_launch_dependents();
    // column j is always handled by thread j % blockDim.x: a fixed order per column
    for (int j = threadIdx.x; j < N; j += blockDim.x) {
        pg[j] = 0.f;
        if (LN) pb[j] = 0.f;
    }
    const T *g = static_cast<const T *>(p.gamma);
    for (int i = 0; i < nrows; ++i) {
        const int64_t row = row0 + i;
        const T *xr = static_cast<const T *>(p.x) + row * N;
        const T *dyr = static_cast<const T *>(p.dy) + row * N;
        const float rs = p.rstd[row];
        const float mu = LN ? p.mean[row] : 0.f;
        float s1 = 0.f, s2 = 0.f;
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            const float xhat = (Tr::load1(xr + j) - mu) * rs;
            const float dyhat = Tr::load1(dyr + j) * Tr::load1(g + j);
            s1 += dyhat;
            s2 = fmaf(dyhat, xhat, s2);
        }
        const float c1 = LN ? block_sum(s1, sm) / fn : 0.f;
        const float c2 = block_sum(s2, sm) / fn;
        T *dxr = static_cast<T *>(p.dx) + row * N;
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            const float xhat = (Tr::load1(xr + j) - mu) * rs;
            const float dy = Tr::load1(dyr + j);
            const float dyhat = dy * Tr::load1(g + j);
            Tr::store1(dxr + j, (dyhat - fmaf(xhat, c2, c1)) * rs);
            pg[j] = fmaf(dy, xhat, pg[j]);
            if (LN) pb[j] += dy;
        }
    }
}

// dgamma[j] (blockIdx.y = 0) or dbeta[j] (blockIdx.y = 1) = sum over g of
// part[g][j].  Thread (slice, q) sums rows g = slice, slice + 16, ... of
// column 32*blockIdx.x + q in that order (its loads issued together), then
// the 16 slice sums are added in slice order: a fixed order per column.
constexpr int kColsumSlices = 16;
__global__ void __launch_bounds__(32 * kColsumSlices) colsum_kernel(const float *__restrict__ part, int G, int ldp,
                                                                     int N, float *__restrict__ dgamma,
                                                                     float *__restrict__ dbeta) {
    __shared__ float sm[kColsumSlices][33];
    griddep_wait();  // the partial rows of the kernel before this one
    const float *P = part + (size_t)blockIdx.y * G * ldp;
    float *out = blockIdx.y ? dbeta : dgamma;
    const int q = threadIdx.x & 31, slice = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + q;
    float a = 0.f;
    if (c < N) {
        for (int g0 = slice; g0 < G; g0 += kColsumSlices * 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int g = g0 + u * kColsumSlices;
                v[u] = g < G ? __ldcg(P + (size_t)g * ldp + c) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) a += v[u];
        }
    }
    sm[slice][q] = a;
    __syncthreads();
    if (slice == 0 && c < N) {
        float t = sm[0][q];
        for (int s2 = 1; s2 < kColsumSlices; ++s2) t += sm[s2][q];
        out[c] = t;
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
namespace {

template <typename T, bool LN, int NV, bool HOLD>
cudaError_t bwd_staged_t(const BwdParams &p, size_t smem, cudaStream_t s) {
    static thread_local int set_for_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (set_for_dev != dev) {
        int optin = 0;
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(bwd_staged_kernel<T, LN, NV, HOLD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin);
        if (e != cudaSuccess) return e;
        set_for_dev = dev;
    }
    bwd_staged_kernel<T, LN, NV, HOLD><<<p.G, kRingThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// held-register variants cover up to 16 elements per thread; the re-read
// variants the wider rows
template <typename T, bool LN>
cudaError_t bwd_staged_nv(int nv, const BwdParams &p, size_t smem, cudaStream_t s) {
    constexpr int V = Traits<T>::kVec;
    if (nv * V <= 16) {
        switch (nv) {
            case 1: return bwd_staged_t<T, LN, 1, true>(p, smem, s);
            case 2: return bwd_staged_t<T, LN, 2, true>(p, smem, s);
            case 3: if constexpr (3 * V <= 16) return bwd_staged_t<T, LN, 3, true>(p, smem, s); break;
            case 4: if constexpr (4 * V <= 16) return bwd_staged_t<T, LN, 4, true>(p, smem, s); break;
        }
        return cudaErrorInvalidValue;
    }
    if constexpr (V == 8) {
        switch (nv) {
            case 3: return bwd_staged_t<T, LN, 3, false>(p, smem, s);
            case 4: return bwd_staged_t<T, LN, 4, false>(p, smem, s);
        }
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t bwd_staged_ln(bool ln, int nv, const BwdParams &p, size_t smem, cudaStream_t s) {
    return ln ? bwd_staged_nv<T, true>(nv, p, smem, s) : bwd_staged_nv<T, false>(nv, p, smem, s);
}

template <typename T>
cudaError_t bwd_plain_ln(bool ln, const BwdParams &p, cudaStream_t s) {
    if (ln)
        bwd_plain_kernel<T, true><<<p.G, kGenericThreads, 0, s>>>(p);
    else
        bwd_plain_kernel<T, false><<<p.G, kGenericThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_staged(int dtype, bool ln, int nv, const BwdParams &p, size_t smem, cudaStream_t s) {
    switch (dtype) {
        case 0: return bwd_staged_ln<float>(ln, nv, p, smem, s);
        case 1: return bwd_staged_ln<__half>(ln, nv, p, smem, s);
        case 2: return bwd_staged_ln<__nv_bfloat16>(ln, nv, p, smem, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_plain(int dtype, bool ln, const BwdParams &p, cudaStream_t s) {
    switch (dtype) {
        case 0: return bwd_plain_ln<float>(ln, p, s);
        case 1: return bwd_plain_ln<__half>(ln, p, s);
        case 2: return bwd_plain_ln<__nv_bfloat16>(ln, p, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_colsum(const float *part, int G, int ldp, int N, float *dgamma, float *dbeta, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + 31) / 32, dbeta ? 2 : 1);
    cfg.blockDim = dim3(32 * kColsumSlices);
    cfg.stream = s;
    // launched as a programmatic dependent of the rows kernel before it
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, colsum_kernel, part, G, ldp, N, dgamma, dbeta);
}

cudaError_t error_flag_address(int **addr) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(addr), g_error_flag);
}

cudaError_t read_error_flag(int *value, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_error_flag, sizeof(int));
    if (e != cudaSuccess) return e;
    if (clear) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_error_flag, &zero, sizeof(int));
    }
    return e;
}

}  // namespace gbn
