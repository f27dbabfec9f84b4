// bwd_bf16.cu -- the backward kernels for __nv_bfloat16 storage (templates in bwd_kernels.cuh).
#include "bwd_kernels.cuh"
#include "bwd_ws.cuh"

namespace gbn {

cudaError_t launch_bwd_staged_bf16(bool ln, int nv, bool full, const BwdParams &p, size_t smem, cudaStream_t s) {
    return bwd_staged_dispatch<__nv_bfloat16>(ln, nv, full, p, smem, s);
}

cudaError_t launch_bwd_ws_bf16(bool ln, int vo, const BwdParams &p, size_t smem, cudaStream_t s) {
    return bwd_ws_dispatch<__nv_bfloat16>(ln, vo, p, smem, s);
}

cudaError_t launch_bwd_plain_bf16(bool ln, const BwdParams &p, cudaStream_t s) { return bwd_plain_dispatch<__nv_bfloat16>(ln, p, s); }

cudaError_t launch_colwalk_bf16(bool ln, const BwdParams &p, float *dg, float *db, bool acc, cudaStream_t s) {
    return colwalk_dispatch<__nv_bfloat16>(ln, p, dg, db, acc, s);
}

}  // namespace gbn
