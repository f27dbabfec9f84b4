/*
 * gbnorm.h -- C ABI of the GB300 (sm_103a) LayerNorm / RMSNorm forward and
 * backward library (libgbnorm.so).
 *
 * The operations are the ones defined on the page "Norm backward in Triton --
 * the dγ/dβ reduction", section "The gradients" (and, with the same formulas,
 * "Norm & activation backward", section "LayerNorm backward, derived"):
 *
 *   LayerNorm, per row x of length N:
 *     mean = sum(x)/N,  var = sum((x-mean)^2)/N  (biased, after the mean),
 *     rstd = 1/sqrt(var + eps),  xhat = (x-mean)*rstd,  y = gamma*xhat + beta
 *   RMSNorm, per row:
 *     rstd = 1/sqrt(sum(x^2)/N + eps),  xhat = x*rstd,  y = gamma*xhat
 *   Backward, with dyhat = dy*gamma:
 *     dx = rstd*(dyhat - mean(dyhat) - xhat*mean(dyhat*xhat))
 *          (RMSNorm: without the mean(dyhat) term)
 *     dgamma[j] = sum over rows of dy*xhat,  dbeta[j] = sum over rows of dy
 *
 * The backward recomputes xhat from the saved per-row mean / rstd instead of
 * reading a stored xhat ("Norm & activation backward", section "Half one").
 * dgamma / dbeta are reduced deterministically: each CTA owns a contiguous
 * block of rows and writes one fp32 partial row into a caller-provided
 * [G, N] workspace; a second kernel sums the G partial rows per column in a
 * fixed order ("Norm backward in Triton", section "The hard half", the
 * disjoint-row-block variant).  No floating-point atomics are used, so
 * dgamma / dbeta are bit-identical from run to run for the same inputs,
 * shapes, dtype, device and buffer alignment.
 *
 * Conventions shared by every call:
 *   - Tensors are row-major and contiguous: element (r, j) of an [M, N] tensor
 *     is at index r*N + j.  gamma, beta, dgamma, dbeta are length N; mean and
 *     rstd are length M.
 *   - x, y, dy, dx, gamma, beta are of type `dtype` (gbn_dtype).  mean, rstd,
 *     dgamma, dbeta are always float32.
 *   - Every pointer is DEVICE memory owned by the caller, on the current CUDA
 *     device.  The library allocates nothing, frees nothing and never
 *     synchronises: each call only enqueues kernels on `stream` (0 = the
 *     legacy default stream) and returns.
 *   - Outputs are overwritten, never accumulated into.
 *   - Arithmetic is float32 with float32 reductions; results stored in
 *     fp16 / bf16 are rounded to nearest even.
 *   - 16-byte aligned pointers with N*sizeof(dtype) a multiple of 16 take the
 *     bulk-copy (TMA) staged kernels; anything else takes a plain-load kernel
 *     with the same results up to float32 rounding order.
 *   - Return value: GBN_OK (0) or a gbn_status code.  Argument errors are
 *     detected on the host before anything is enqueued.  GBN_ECUDA means a
 *     launch or a CUDA query failed (the CUDA error is cleared).  Faults of
 *     kernels already enqueued surface at the caller's next synchronisation,
 *     as with any CUDA call.
 */
#ifndef GBNORM_H
#define GBNORM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GBN_F32 = 0,  /* float32 storage                     */
    GBN_F16 = 1,  /* IEEE binary16 storage               */
    GBN_BF16 = 2  /* bfloat16 storage                    */
} gbn_dtype;

typedef enum {
    GBN_OK = 0,
    GBN_EINVAL = 1,     /* null pointer, M < 0, N < 1 or too large, bad eps   */
    GBN_EDTYPE = 2,     /* dtype not one of gbn_dtype                         */
    GBN_EWORKSPACE = 4, /* workspace_bytes below gbn_bwd_workspace_bytes()    */
    GBN_ECUDA = 5,      /* a CUDA launch or query failed                      */
    GBN_EDEVICE = 6,    /* a kernel gave up on a bounded wait (see below)     */
    GBN_ESCRATCH = 7    /* rms_bwd_noalloc: problem exceeds its static scratch */
} gbn_status;

/* Largest N accepted by every call. */
#define GBN_MAX_N (1 << 24)

/*
 * Bytes of device workspace the backward (ln_bwd / rms_bwd and their two
 * phases) needs for an [M, N] problem of `dtype` on the CURRENT device;
 * has_beta = 1 for LayerNorm (dgamma and dbeta partials), 0 for RMSNorm.
 * The size depends on the device's SM count.  The workspace may have any
 * alignment.  Returns 0 if M <= 0 (no workspace is needed) or the arguments
 * are invalid.
 */
size_t gbn_bwd_workspace_bytes(int64_t M, int64_t N, int dtype, int has_beta);

/*
 * LayerNorm forward ("Norm backward in Triton", "The gradients", forward
 * line; "05: Layer norm", kernel ln_fwd: mean first, then the biased
 * variance of the centred row, eps under the root).
 *   x [M,N] dtype (in), gamma [N], beta [N] dtype (in),
 *   y [M,N] dtype (out), mean [M] f32 (out), rstd [M] f32 (out).
 *   eps >= 0 and finite.  M = 0 is a no-op.
 */
int ln_fwd(const void *x, const void *gamma, const void *beta, void *y,
           float *mean, float *rstd, float eps, int64_t M, int64_t N,
           int dtype, cudaStream_t stream);

/*
 * RMSNorm forward ("Norm backward in Triton", "The gradients", RMSNorm
 * paragraph): rstd = 1/sqrt(mean(x^2) + eps), y = gamma * x * rstd.
 *   x [M,N] (in), gamma [N] (in), y [M,N] (out), rstd [M] f32 (out).
 */
int rms_fwd(const void *x, const void *gamma, void *y, float *rstd, float eps,
            int64_t M, int64_t N, int dtype, cudaStream_t stream);

/*
 * LayerNorm backward ("Norm backward in Triton", "The gradients": dx, dgamma,
 * dbeta lines; the dx kernel recomputes xhat from the saved statistics).
 *   dy, x [M,N] dtype (in); gamma [N] dtype (in); mean, rstd [M] f32 (in,
 *   as written by ln_fwd); dx [M,N] dtype (out); dgamma, dbeta [N] f32 (out).
 *   eps is used only when mean and rstd are both NULL: then nothing was
 *   saved and the backward forms each row's mean and rstd from x itself,
 *   as ln_fwd does ("Norm & activation backward", "Half one": the
 *   save-nothing option of the save-vs-recompute table); x is read once
 *   either way.  Passing only one of mean / rstd is GBN_EINVAL.
 *   workspace: device scratch of at least gbn_bwd_workspace_bytes(M, N,
 *   dtype, 1) bytes, owned by the caller; its contents on entry do not
 *   matter and on return are the per-CTA partials.  It must not be used by
 *   another call that runs concurrently.
 *   M = 0: dgamma and dbeta are set to zero, nothing else is touched.
 */
int ln_bwd(const void *dy, const void *x, const void *gamma, const float *mean,
           const float *rstd, void *dx, float *dgamma, float *dbeta, float eps,
           int64_t M, int64_t N, int dtype, void *workspace,
           size_t workspace_bytes, cudaStream_t stream);

/*
 * RMSNorm backward: LayerNorm's without the mean and without the mean(dyhat)
 * term, and without dbeta.  Arguments as for ln_bwd (rstd NULL: recomputed
 * from x with eps); the workspace size is gbn_bwd_workspace_bytes(M, N,
 * dtype, 0).
 */
int rms_bwd(const void *dy, const void *x, const void *gamma, const float *rstd,
            void *dx, float *dgamma, float eps, int64_t M, int64_t N, int dtype,
            void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Options of the extended calls below.  A NULL options pointer, or a
 * zero-initialised struct, means: contiguous rows, outputs overwritten,
 * dgamma / dbeta in float32 -- exactly the plain calls above.
 *   ld_x, ld_dy, ld_out: row strides in elements of x, dy and the row output
 *     (y in the forward, dx in the backward); 0 means N, else >= N.  Rows
 *     stay contiguous within themselves ("Norm backward in Triton",
 *     "The dx kernel": the stride_row argument).  The bulk-copy staged
 *     kernels need every stride times the element size to be a multiple of
 *     16 bytes; other strides take the plain-load kernels.
 *   accumulate (backward): 1 adds this call's sums to what dgamma / dbeta
 *     hold ("Matmul backward in Triton", the grad buffer is accumulated
 *     into, never overwritten); the previous value is added after the
 *     fixed-order sum, so the result stays deterministic.  With M = 0 the
 *     buffers are left as they are.
 *   grad_dtype (backward): storage type of dgamma / dbeta: GBN_F32 (the
 *     default) or the dtype of the call (the parameters' own type, the cast
 *     the pages' reduce kernels apply at the end), rounded to nearest even.
 *   reduce_mode (backward): how dgamma / dbeta are reduced across rows.
 *     GBN_REDUCE_PARTIALS (0, the default): per-CTA partial rows in the
 *       workspace, summed per column in a fixed order; deterministic.
 *     GBN_REDUCE_ATOMIC (1): each CTA adds its partial row into dgamma /
 *       dbeta with float32 atomics ("Norm backward in Triton", "atomic_add
 *       straight to a [d] buffer", at CTA granularity); NOT deterministic
 *       (the order of the additions varies from run to run).  Needs
 *       grad_dtype GBN_F32.
 *     GBN_REDUCE_COLWALK (2): a second kernel in which each CTA owns 32
 *       columns and walks every row of x and dy again ("05: Layer norm",
 *       kernel ln_bwd_dwdb); deterministic, one more read of x and dy.
 *       Needs grad_dtype GBN_F32 and the saved statistics.
 *     The last two exist to measure what the default costs or saves.
 *   kernel: which kernel takes the rows (forward and backward).
 *     GBN_KERNEL_AUTO (0, the default): the fastest one that applies.
 *     GBN_KERNEL_SLOT (1): the slot-staged bulk-copy kernel, never the
 *       warp-specialised backward; the plain kernel where rows are not
 *       16-byte aligned.
 *     GBN_KERNEL_PLAIN (2): the plain-load kernel.
 *     Every kernel gives the same results up to float32 rounding order, and
 *     dgamma / dbeta keep one summation order per (M, N, dtype, device)
 *     for a given kernel.
 *   host_chunk (host-buffer calls only): rows (norm) or elements
 *     (activation) per pipeline chunk; 0 means about 16 MiB of each input.
 *   wait_limit_ns (backward): how long a kernel's warp waits for data from
 *     another warp or a bulk copy before it gives up and reports error 1
 *     through gbn_device_error(); 0 means two seconds.  The wait for the
 *     kernel's own copies in flight before it exits keeps its own limit.
 *     A diagnostic: a tiny value makes the waits run out on purpose, so the
 *     error path can be tested without a fault.
 * Fields that a call does not use must be zero.
 */
enum { GBN_REDUCE_PARTIALS = 0, GBN_REDUCE_ATOMIC = 1, GBN_REDUCE_COLWALK = 2 };
enum { GBN_KERNEL_AUTO = 0, GBN_KERNEL_SLOT = 1, GBN_KERNEL_PLAIN = 2 };

typedef struct {
    int64_t ld_x;
    int64_t ld_dy;
    int64_t ld_out;
    int accumulate;
    int grad_dtype;
    int reduce_mode;
    int kernel;
    int64_t host_chunk;
    int64_t wait_limit_ns;
} gbn_options;

/* The four operations with gbn_options; dgamma / dbeta are `void *` of type
 * opt->grad_dtype.  Everything else as in the plain calls. */
int ln_fwd_ex(const void *x, const void *gamma, const void *beta, void *y,
              float *mean, float *rstd, float eps, int64_t M, int64_t N,
              int dtype, const gbn_options *opt, cudaStream_t stream);
int rms_fwd_ex(const void *x, const void *gamma, void *y, float *rstd,
               float eps, int64_t M, int64_t N, int dtype,
               const gbn_options *opt, cudaStream_t stream);
int ln_bwd_ex(const void *dy, const void *x, const void *gamma,
              const float *mean, const float *rstd, void *dx, void *dgamma,
              void *dbeta, float eps, int64_t M, int64_t N, int dtype,
              void *workspace, size_t workspace_bytes, const gbn_options *opt,
              cudaStream_t stream);
int rms_bwd_ex(const void *dy, const void *x, const void *gamma,
               const float *rstd, void *dx, void *dgamma, float eps,
               int64_t M, int64_t N, int dtype, void *workspace,
               size_t workspace_bytes, const gbn_options *opt,
               cudaStream_t stream);

/*
 * rms_bwd_noalloc: rms_bwd for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it is a packaging of rms_bwd.
 *
 * Some callers cannot call cudaMalloc (or any allocating routine) where they
 * run the backward: code inside an allocator's own callback, where
 * allocating would re-enter the allocator; engines and plugins that run
 * under a device-memory budget fixed up front and are handed no workspace;
 * latency-critical loops that cannot afford the implicit device
 * synchronisation a cudaMalloc / cudaFree may cause.  This call takes
 * the same inputs and outputs as rms_bwd but no workspace: the per-CTA
 * partial rows go to a static device array of GBN_NOALLOC_SCRATCH_BYTES
 * that the library holds on every GPU that loads it, until the process
 * exits.  It allocates nothing and frees nothing.
 *   - Problems needing more than GBN_NOALLOC_SCRATCH_BYTES of workspace
 *     (gbn_bwd_workspace_bytes(M, N, dtype, 0)) return GBN_ESCRATCH before
 *     anything is enqueued.
 *   - The first call on a device looks up the array's device address with
 *     that device current (cudaGetSymbolAddress) and caches it; make that
 *     first call before any stream capture.
 *   - All calls on a device share the one array, which keeps the last
 *     call's partial rows; nothing in it needs clearing between calls.
 *     Calls that overlap on the GPU (other streams, other threads) race on
 *     it and give wrong dgamma: order them on one stream or with events.
 */
#define GBN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int rms_bwd_noalloc(const void *dy, const void *x, const void *gamma,
                    const float *rstd, void *dx, float *dgamma, float eps,
                    int64_t M, int64_t N, int dtype, cudaStream_t stream);

/*
 * The two phases of the backward, for callers that time or overlap them
 * separately.  *_bwd_rows runs only the fused per-row kernel: dx, plus the
 * per-CTA partial rows written into `workspace` ("Norm backward in Triton",
 * "The hard half": one partial row per block of rows).  gbn_bwd_reduce then
 * sums those partial rows per column in a fixed order into dgamma (and
 * dbeta when has_beta = 1).  Running ln_bwd_rows then gbn_bwd_reduce on one
 * stream, with the same (M, N, dtype) and workspace, is exactly ln_bwd.
 */
int ln_bwd_rows(const void *dy, const void *x, const void *gamma,
                const float *mean, const float *rstd, void *dx, int64_t M,
                int64_t N, int dtype, void *workspace, size_t workspace_bytes,
                cudaStream_t stream);
int rms_bwd_rows(const void *dy, const void *x, const void *gamma,
                 const float *rstd, void *dx, int64_t M, int64_t N, int dtype,
                 void *workspace, size_t workspace_bytes, cudaStream_t stream);
int gbn_bwd_reduce(const void *workspace, size_t workspace_bytes, int64_t M,
                   int64_t N, int dtype, int has_beta, float *dgamma,
                   float *dbeta, cudaStream_t stream);

/*
 * Describes the launch the backward takes for an [M, N] problem on the
 * current device: *G = number of row blocks (CTAs, rows of the partial
 * workspace), and for 16-byte aligned buffers and saved statistics
 * *staged = 2 (the warp-specialised bulk-copy kernel), 1 (the slot-staged
 * bulk-copy kernel) or 0 (the plain-load kernel, which every alignment can
 * take).  Either output pointer may be NULL.  Returns a gbn_status.
 */
int gbn_bwd_plan(int64_t M, int64_t N, int dtype, int has_beta, int *G,
                 int *staged);

/*
 * Backward from HOST buffers ("Norm backward in Triton -- the dγ/dβ
 * reduction", section "The gradients"; the same results as ln_bwd / rms_bwd
 * up to the grouping of the dgamma / dbeta partial sums).
 *   dy, x, dx: [M, N] row-major host memory of `dtype`; gamma [N] host;
 *   mean (LayerNorm), rstd: [M] float32 host (the forward's statistics);
 *   dgamma, dbeta (LayerNorm): [N] float32 host outputs.  Page-locked
 *   (pinned) host memory lets the copies overlap; pageable memory works but
 *   its copies serialise.  dx may alias dy.
 *   workspace: DEVICE memory of at least gbn_bwd_host_workspace_bytes(M, N,
 *   dtype, has_beta) bytes, any alignment: gamma, the statistics, three
 *   chunk buffers per tensor, the partial rows and the device dgamma / dbeta.
 * The rows are cut into chunks of about 16 MiB of each input, after a ramp
 * of 1/8, 1/4 and 1/2 of that which starts the pipeline sooner.  gamma and the
 * statistics are copied in first; then chunk i's x and dy are copied in on
 * one internal stream while chunk i-1's backward runs on `stream` and chunk
 * i-2's dx is copied out on another internal stream;
 * the internal streams (two per device, created on first use) are ordered
 * after the work already on `stream`, and `stream` waits for them at the end,
 * so the results are complete once `stream` is.  dgamma / dbeta: every chunk
 * writes its partial rows into one block of the workspace and a single
 * fixed-order column reduce sums them (deterministic).
 * Errors: argument errors before anything is enqueued; M = 0 writes zeros
 * into dgamma / dbeta at once; GBN_ECUDA if a CUDA call fails part-way (the
 * work enqueued until then still runs, and `stream` is made to wait for it
 * where CUDA still allows, so the buffers may be reused in stream order).
 */
size_t gbn_bwd_host_workspace_bytes(int64_t M, int64_t N, int dtype, int has_beta);
int ln_bwd_host(const void *dy, const void *x, const void *gamma, const float *mean, const float *rstd, void *dx,
                float *dgamma, float *dbeta, int64_t M, int64_t N, int dtype, void *workspace,
                size_t workspace_bytes, cudaStream_t stream);
int rms_bwd_host(const void *dy, const void *x, const void *gamma, const float *rstd, void *dx, float *dgamma,
                 int64_t M, int64_t N, int dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The host-buffer backward with gbn_options.  Of the options, only
 * host_chunk (rows per chunk after the ramp; 0 = about 16 MiB of each
 * input), kernel and wait_limit_ns apply; the others must be zero.  The
 * workspace size depends on host_chunk.
 */
size_t gbn_bwd_host_workspace_bytes_ex(int64_t M, int64_t N, int dtype, int has_beta, const gbn_options *opt);
int ln_bwd_host_ex(const void *dy, const void *x, const void *gamma, const float *mean, const float *rstd,
                   void *dx, float *dgamma, float *dbeta, int64_t M, int64_t N, int dtype, void *workspace,
                   size_t workspace_bytes, const gbn_options *opt, cudaStream_t stream);
int rms_bwd_host_ex(const void *dy, const void *x, const void *gamma, const float *rstd, void *dx, float *dgamma,
                    int64_t M, int64_t N, int dtype, void *workspace, size_t workspace_bytes,
                    const gbn_options *opt, cudaStream_t stream);

/*
 * Activation backward ("Norm backward in Triton", section "Activation
 * backward -- fuse it into the epilogue"): dx = dy * f'(preact), the
 * derivative recomputed from the saved pre-activation, for
 *   silu_bwd: f'(x) = sigma(x) * (1 + x * (1 - sigma(x))),
 *   gelu_bwd: the exact (erf) GELU, f'(x) = Phi(x) + x * phi(x).
 *   dy, preact (in), dx (out): n contiguous elements of `dtype`, device
 *   memory; dx may alias dy.  Float32 arithmetic, dx rounded to nearest
 *   even.  n = 0 is a no-op.
 */
int silu_bwd(const void *dy, const void *preact, void *dx, int64_t n, int dtype, cudaStream_t stream);
int gelu_bwd(const void *dy, const void *preact, void *dx, int64_t n, int dtype, cudaStream_t stream);

/*
 * The activation backward from HOST buffers: dy, preact (in), dx (out) are n
 * elements of `dtype` in host memory (pinned for overlap; dx may alias dy).
 * workspace: DEVICE memory of at least gbn_act_host_workspace_bytes(n,
 * dtype) bytes, any alignment.  The elements are cut into chunks of about
 * 16 MiB of each tensor (after a ramp of 1/8, 1/4, 1/2 of that); chunk i is
 * copied in on an internal stream while chunk i-1's kernel runs on `stream`
 * and chunk i-2's dx is copied out on another internal stream, through
 * three device buffers per tensor; `stream` waits for the internal streams
 * at the end, so dx is complete once `stream` is.  Errors as for silu_bwd,
 * plus GBN_EWORKSPACE; GBN_ECUDA if a CUDA call fails part-way (the work
 * enqueued until then still runs, and `stream` waits for it as above).
 */
size_t gbn_act_host_workspace_bytes(int64_t n, int dtype);
int silu_bwd_host(const void *dy, const void *preact, void *dx, int64_t n, int dtype, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream);
int gelu_bwd_host(const void *dy, const void *preact, void *dx, int64_t n, int dtype, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream);

/* The host-buffer activation backward with gbn_options: only host_chunk
 * (elements per chunk after the ramp; 0 = about 16 MiB of each tensor)
 * applies; the other fields must be zero. */
size_t gbn_act_host_workspace_bytes_ex(int64_t n, int dtype, const gbn_options *opt);
int silu_bwd_host_ex(const void *dy, const void *preact, void *dx, int64_t n, int dtype, void *workspace,
                     size_t workspace_bytes, const gbn_options *opt, cudaStream_t stream);
int gelu_bwd_host_ex(const void *dy, const void *preact, void *dx, int64_t n, int dtype, void *workspace,
                     size_t workspace_bytes, const gbn_options *opt, cudaStream_t stream);

/*
 * Every wait inside the library's kernels (on a shared-memory barrier that
 * a bulk copy completes) gives up after about two seconds; the kernel then
 * records an error code in a per-device flag, drains its own copies with
 * another bounded wait and returns instead of hanging.  This call
 * synchronises the current device, returns the flag (0 = no error) and, if
 * clear != 0, resets it.  GBN_ECUDA (as a negative number) if the
 * synchronisation or the read fails.  Codes: 1 a bulk copy did not
 * complete; 2 copies still in flight when the kernel gave up draining them.
 */
int gbn_device_error(int clear);

/* A static, human-readable name of a gbn_status code. */
const char *gbn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GBNORM_H */
