// bwd_f32.cu -- the backward kernels for float storage (templates in bwd_kernels.cuh).
#include "bwd_kernels.cuh"
#include "bwd_ws.cuh"

namespace gbn {

cudaError_t launch_bwd_staged_f32(bool ln, int nv, bool full, const BwdParams &p, size_t smem, cudaStream_t s) {
    return bwd_staged_dispatch<float>(ln, nv, full, p, smem, s);
}

cudaError_t launch_bwd_ws_f32(bool ln, int vo, const BwdParams &p, size_t smem, cudaStream_t s) {
    return bwd_ws_dispatch<float>(ln, vo, p, smem, s);
}

cudaError_t launch_bwd_plain_f32(bool ln, const BwdParams &p, cudaStream_t s) { return bwd_plain_dispatch<float>(ln, p, s); }

cudaError_t launch_colwalk_f32(bool ln, const BwdParams &p, float *dg, float *db, bool acc, cudaStream_t s) {
    return colwalk_dispatch<float>(ln, p, dg, db, acc, s);
}

}  // namespace gbn
