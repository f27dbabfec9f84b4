// fwd_bf16.cu -- the forward kernels for __nv_bfloat16 storage (templates in fwd_kernels.cuh).
#include "fwd_kernels.cuh"

namespace gbn {

cudaError_t launch_fwd_staged_bf16(bool ln, int nv, bool full, const FwdParams &p, size_t smem, cudaStream_t s) {
    return fwd_staged_dispatch<__nv_bfloat16>(ln, nv, full, p, smem, s);
}

cudaError_t launch_fwd_plain_bf16(bool ln, const FwdParams &p, cudaStream_t s) { return fwd_plain_dispatch<__nv_bfloat16>(ln, p, s); }

}  // namespace gbn
