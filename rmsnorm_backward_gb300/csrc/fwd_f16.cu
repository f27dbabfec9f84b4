// fwd_f16.cu -- the forward kernels for __half storage (templates in fwd_kernels.cuh).
#include "fwd_kernels.cuh"

namespace gbn {

cudaError_t launch_fwd_staged_f16(bool ln, int nv, bool full, const FwdParams &p, size_t smem, cudaStream_t s) {
    return fwd_staged_dispatch<__half>(ln, nv, full, p, smem, s);
}

cudaError_t launch_fwd_plain_f16(bool ln, const FwdParams &p, cudaStream_t s) { return fwd_plain_dispatch<__half>(ln, p, s); }

}  // namespace gbn
