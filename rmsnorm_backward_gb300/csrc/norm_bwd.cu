// norm_bwd.cu -- the column reduce of the backward's partial rows, the
// per-device error flag, and the dtype dispatch to the kernels instantiated
// in fwd_{f32,f16,bf16}.cu and bwd_{f32,f16,bf16}.cu.
//
// The reduce finishes dgamma[j] = sum over rows of dy*xhat and dbeta[j] =
// sum over rows of dy ("Norm backward in Triton -- the dγ/dβ reduction",
// section "The gradients"), summing the per-CTA partial rows in a fixed
// order ("The hard half": a second, small kernel over the [GROUPS, d]
// workspace), so the result does not depend on timing.
#include <type_traits>

#include "gbn_device.cuh"
#include "gbn_launch.h"

namespace gbn {

static __device__ int g_error_flag = 0;

// dgamma (blockIdx.y = 0) or dbeta (blockIdx.y = 1): CTA x sums columns
// [32*VEC*x, 32*VEC*(x + 1)) of the partial rows with colsum_range (one
// fixed order per SLICES, whatever VEC).
template <typename OutT, bool ACC, int SLICES, int VEC>
__global__ void __launch_bounds__(32 * SLICES) colsum_kernel(const float *__restrict__ part, int G, int ldp,
                                                                     int N, OutT *__restrict__ dgamma,
                                                                     OutT *__restrict__ dbeta) {
    __shared__ float sm[SLICES * (32 * VEC + 1)];
    griddep_wait();  // the partial rows of the kernel before this one
    const float *P = part + (size_t)blockIdx.y * G * ldp;
    OutT *out = blockIdx.y ? dbeta : dgamma;
    const int c0 = blockIdx.x * 32 * VEC;
    // accumulate: the buffer's previous value is added after the fixed-order
    // sum; 16-bit outputs are rounded to nearest even
    colsum_range<SLICES, VEC>(
        P, G, ldp, c0, min(N, c0 + 32 * VEC),
        [&](int c, float t) {
            if constexpr (std::is_same<OutT, float>::value) {
                out[c] = ACC ? out[c] + t : t;
            } else {
                Traits<OutT>::store1(out + c, ACC ? Traits<OutT>::load1(out + c) + t : t);
            }
        },
        sm);
}

// ---------------------------------------------------------------------------
// launchers: dtype dispatch to the per-dtype instantiations
// ---------------------------------------------------------------------------
cudaError_t launch_fwd_staged_f32(bool, int, bool, const FwdParams &, size_t, cudaStream_t);
cudaError_t launch_fwd_staged_f16(bool, int, bool, const FwdParams &, size_t, cudaStream_t);
cudaError_t launch_fwd_staged_bf16(bool, int, bool, const FwdParams &, size_t, cudaStream_t);
cudaError_t launch_fwd_plain_f32(bool, const FwdParams &, cudaStream_t);
cudaError_t launch_fwd_plain_f16(bool, const FwdParams &, cudaStream_t);
cudaError_t launch_fwd_plain_bf16(bool, const FwdParams &, cudaStream_t);
cudaError_t launch_bwd_staged_f32(bool, int, bool, const BwdParams &, size_t, cudaStream_t);
cudaError_t launch_bwd_staged_f16(bool, int, bool, const BwdParams &, size_t, cudaStream_t);
cudaError_t launch_bwd_staged_bf16(bool, int, bool, const BwdParams &, size_t, cudaStream_t);
cudaError_t launch_bwd_plain_f32(bool, const BwdParams &, cudaStream_t);
cudaError_t launch_bwd_plain_f16(bool, const BwdParams &, cudaStream_t);
cudaError_t launch_bwd_plain_bf16(bool, const BwdParams &, cudaStream_t);

cudaError_t launch_bwd_ws_f32(bool, int, const BwdParams &, size_t, cudaStream_t);
cudaError_t launch_bwd_ws_f16(bool, int, const BwdParams &, size_t, cudaStream_t);
cudaError_t launch_bwd_ws_bf16(bool, int, const BwdParams &, size_t, cudaStream_t);

cudaError_t launch_bwd_ws(int dtype, bool ln, int vo, const BwdParams &p, size_t smem, cudaStream_t s) {
    switch (dtype) {
        case 0: return launch_bwd_ws_f32(ln, vo, p, smem, s);
        case 1: return launch_bwd_ws_f16(ln, vo, p, smem, s);
        case 2: return launch_bwd_ws_bf16(ln, vo, p, smem, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_colwalk_f32(bool, const BwdParams &, float *, float *, bool, cudaStream_t);
cudaError_t launch_colwalk_f16(bool, const BwdParams &, float *, float *, bool, cudaStream_t);
cudaError_t launch_colwalk_bf16(bool, const BwdParams &, float *, float *, bool, cudaStream_t);

cudaError_t launch_colwalk(int dtype, bool ln, const BwdParams &p, float *dgamma, float *dbeta, bool accumulate,
                           cudaStream_t s) {
    switch (dtype) {
        case 0: return launch_colwalk_f32(ln, p, dgamma, dbeta, accumulate, s);
        case 1: return launch_colwalk_f16(ln, p, dgamma, dbeta, accumulate, s);
        case 2: return launch_colwalk_bf16(ln, p, dgamma, dbeta, accumulate, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_staged(int dtype, bool ln, int nv, bool full, const FwdParams &p, size_t smem,
                              cudaStream_t s) {
    switch (dtype) {
        case 0: return launch_fwd_staged_f32(ln, nv, full, p, smem, s);
        case 1: return launch_fwd_staged_f16(ln, nv, full, p, smem, s);
        case 2: return launch_fwd_staged_bf16(ln, nv, full, p, smem, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_plain(int dtype, bool ln, const FwdParams &p, cudaStream_t s) {
    switch (dtype) {
        case 0: return launch_fwd_plain_f32(ln, p, s);
        case 1: return launch_fwd_plain_f16(ln, p, s);
        case 2: return launch_fwd_plain_bf16(ln, p, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_staged(int dtype, bool ln, int nv, bool full, const BwdParams &p, size_t smem,
                              cudaStream_t s) {
    switch (dtype) {
        case 0: return launch_bwd_staged_f32(ln, nv, full, p, smem, s);
        case 1: return launch_bwd_staged_f16(ln, nv, full, p, smem, s);
        case 2: return launch_bwd_staged_bf16(ln, nv, full, p, smem, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_plain(int dtype, bool ln, const BwdParams &p, cudaStream_t s) {
    switch (dtype) {
        case 0: return launch_bwd_plain_f32(ln, p, s);
        case 1: return launch_bwd_plain_f16(ln, p, s);
        case 2: return launch_bwd_plain_bf16(ln, p, s);
    }
    return cudaErrorInvalidValue;
}

template <typename OutT, bool ACC, int SLICES, int VEC>
cudaError_t launch_colsum_t(const float *part, int G, int ldp, int N, void *dgamma, void *dbeta, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + 32 * VEC - 1) / (32 * VEC), dbeta ? 2 : 1);
    cfg.blockDim = dim3(32 * SLICES);
    cfg.stream = s;
    // launched as a programmatic dependent of the rows kernel before it
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, colsum_kernel<OutT, ACC, SLICES, VEC>, part, G, ldp, N,
                              static_cast<OutT *>(dgamma), static_cast<OutT *>(dbeta));
}

template <typename OutT, bool ACC, int SLICES>
cudaError_t launch_colsum_v(const float *part, int G, int ldp, int N, void *dg, void *db, int vec, cudaStream_t s) {
    if constexpr (SLICES == 8) {
        if (vec == 4) return launch_colsum_t<OutT, ACC, SLICES, 4>(part, G, ldp, N, dg, db, s);
    }
    return launch_colsum_t<OutT, ACC, SLICES, 1>(part, G, ldp, N, dg, db, s);
}

template <typename OutT>
cudaError_t launch_colsum_acc(const float *part, int G, int ldp, int N, void *dg, void *db, bool acc, bool small,
                              int vec, cudaStream_t s) {
    if (small)
        return acc ? launch_colsum_v<OutT, true, 8>(part, G, ldp, N, dg, db, vec, s)
                   : launch_colsum_v<OutT, false, 8>(part, G, ldp, N, dg, db, vec, s);
    return acc ? launch_colsum_v<OutT, true, 16>(part, G, ldp, N, dg, db, vec, s)
               : launch_colsum_v<OutT, false, 16>(part, G, ldp, N, dg, db, vec, s);
}

// vec: columns a lane sums (1 or 4).  8 slices: four when one would need
// more CTAs than SMs, so a wide partial block is read in one wave of loads
// (1151x8192 f16 LayerNorm: 1.2 us less than one column a lane).  16 slices
// stay at one column a lane: with four the compiler kept fewer loads in
// flight (8192x16384 RMSNorm: 1.1 us more).
cudaError_t launch_colsum(const float *part, int G, int ldp, int N, void *dgamma, void *dbeta, int out_dtype,
                          bool accumulate, bool small, int sms, cudaStream_t s) {
    const int arrays = dbeta ? 2 : 1;
    int vec = 1;
    if (small && (int64_t)((N + 31) / 32) * arrays > sms) vec = 4;
    if (ldp % vec != 0 || (reinterpret_cast<uintptr_t>(part) & (4 * vec - 1)) != 0) vec = 1;
    switch (out_dtype) {
        case 0: return launch_colsum_acc<float>(part, G, ldp, N, dgamma, dbeta, accumulate, small, vec, s);
        case 1: return launch_colsum_acc<__half>(part, G, ldp, N, dgamma, dbeta, accumulate, small, vec, s);
        case 2: return launch_colsum_acc<__nv_bfloat16>(part, G, ldp, N, dgamma, dbeta, accumulate, small, vec, s);
    }
    return cudaErrorInvalidValue;
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
