// fwd_f32.cu -- the forward kernels for float storage (templates in fwd_kernels.cuh).
#include "fwd_kernels.cuh"

namespace gbn {

cudaError_t launch_fwd_staged_f32(bool ln, int nv, bool full, const FwdParams &p, size_t smem, cudaStream_t s) {
    return fwd_staged_dispatch<float>(ln, nv, full, p, smem, s);
}

cudaError_t launch_fwd_plain_f32(bool ln, const FwdParams &p, cudaStream_t s) { return fwd_plain_dispatch<float>(ln, p, s); }

}  // namespace gbn
