// act_bwd.cu -- activation backward for sm_103a: dx = dy * f'(preact), the
// derivative recomputed from the saved pre-activation instead of stored
// ("Norm backward in Triton -- the dγ/dβ reduction", section "Activation
// backward -- fuse it into the epilogue").
//   SiLU: f'(x) = sigma(x) * (1 + x * (1 - sigma(x))).
//   GELU, exact (erf) form: f'(x) = Phi(x) + x * phi(x).
// Elementwise and HBM-bound (read dy and preact, write dx) once the
// derivative costs few enough instructions: exponentials are exp2 of a
// pre-scaled argument, 16-bit outputs take packed float32-pair arithmetic,
// and GELU's distribution function takes a published fit that shares phi's
// exponential.  Copies into per-warp shared-memory rings keep HBM busy while
// the warps compute (the kernel's own comment has the layout).
#include <type_traits>

#include "gbn_device.cuh"
#include "gbn_launch.h"

namespace gbn {

// log2(e) as a float32 head and the double remainder, and ln(2)
constexpr float kLog2e = 1.44269504088896341f;
constexpr float kLog2eLo = (float)(1.44269504088896340736 - (double)1.44269504088896341f);
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kInvSqrt2Pi = 0.39894228040143268f;  // 1 / sqrt(2 pi)
constexpr float kLog2InvSqrt2Pi = -1.32574806473616f;  // log2(1 / sqrt(2 pi))

// rcp.approx (1 ulp) and ex2.approx (2^-22 relative), used where the argument
// range is known: reciprocals of [1, 7], powers of two of [-2, 1]
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// exp(-(v_hi + v_lo)) for v_hi >= 0 in float32, subnormal results kept, with
// u log2 e carried as a head and a tail so the product's rounding (|v| 2^-24
// relative in the result) does not reach a float32 output
__device__ __forceinline__ float exp_neg_exact(float v_hi, float v_lo) {
    v_hi = fminf(v_hi, 128.0f);  // e^-128 is below float32's least subnormal
    const float y = -v_hi * kLog2e;
    const float r = exp2f(y);
    const float y_lo = fmaf(-v_hi, kLog2e, -y) - v_hi * kLog2eLo - v_lo * kLog2e;
    return fmaf(r, y_lo * kLn2, r);
}

// erfc(z) = t exp(-z^2 + P(t)), t = 1 / (1 + z / 2), z >= 0, fractional error
// below 1.2e-7 (Numerical Recipes, Press et al., section 6.2, "erfcc", a
// Chebyshev fit).  Carried here in base 2 and shifted for the tail mass
// Phi(-a) = erfc(a / sqrt 2) / 2 = t * phi(a) * 2^Q(t), with
// Q = P log2(e) + log2(sqrt(2 pi) / 2): Q lies in [-1.6, 0.33].
constexpr double kL2e = 1.44269504088896340736;
constexpr double kQShift = 0.32574806473616;  // log2(sqrt(2 pi) / 2)
constexpr float kQ0 = (float)(-1.26551223 * kL2e + kQShift);
constexpr float kQ1 = (float)(1.00002368 * kL2e);
constexpr float kQ2 = (float)(0.37409196 * kL2e);
constexpr float kQ3 = (float)(0.09678418 * kL2e);
constexpr float kQ4 = (float)(-0.18628806 * kL2e);
constexpr float kQ5 = (float)(0.27886807 * kL2e);
constexpr float kQ6 = (float)(-1.13520398 * kL2e);
constexpr float kQ7 = (float)(1.48851587 * kL2e);
constexpr float kQ8 = (float)(-0.82215223 * kL2e);
constexpr float kQ9 = (float)(0.17087277 * kL2e);
__device__ __forceinline__ float tail_exponent(float t) {
    float q = kQ9;
    q = fmaf(q, t, kQ8);
    q = fmaf(q, t, kQ7);
    q = fmaf(q, t, kQ6);
    q = fmaf(q, t, kQ5);
    q = fmaf(q, t, kQ4);
    q = fmaf(q, t, kQ3);
    q = fmaf(q, t, kQ2);
    q = fmaf(q, t, kQ1);
    return fmaf(q, t, kQ0);
}

// f'(x).  EXACT (float32 outputs) keeps every exponential to a few float32
// ulp; otherwise (16-bit outputs) errors of order 1e-5 relative are allowed,
// far below half an fp16 / bf16 ulp.
template <int ACT, bool EXACT>
__device__ __forceinline__ float act_grad(float x) {
    const float ax = fabsf(x);
    if constexpr (ACT == kActSilu) {
        // with e = exp(-|x|) <= 1 and r = 1 / (1 + e): sigma(x) = r and
        // 1 - sigma(x) = e r for x >= 0, the two swapped for x < 0; nothing
        // overflows and neither factor is formed by cancellation
        const float e = EXACT ? exp_neg_exact(ax, 0.0f) : exp2f(-ax * kLog2e);
        const float r = rcp_approx(1.0f + e);
        const float er = e * r;
        const float s = x >= 0.0f ? r : er;
        const float oms = x >= 0.0f ? er : r;
        return s * fmaf(x, oms, 1.0f);
    } else {
        // GELU'(x) = Phi(x) + x phi(x).  a = min(|x|, 16) (both terms
        // underflow beyond 14.5); phi(a) = exp(-a^2 / 2) / sqrt(2 pi) with
        // a^2 = hi + lo exactly; the tail mass Phi(-a) = t phi(a) 2^Q(t);
        // Phi(x) is the tail for x < 0 and 1 - tail otherwise.
        const float a = fminf(ax, 16.0f);
        const float hi = a * a;
        float pdf;
        if constexpr (EXACT) {
            pdf = kInvSqrt2Pi * exp_neg_exact(0.5f * hi, 0.5f * fmaf(a, a, -hi));
        } else {
            pdf = exp2f(fmaf(hi, -0.5f * kLog2e, kLog2InvSqrt2Pi));
        }
        const float t = rcp_approx(fmaf(a, 0.35355339059327376f, 1.0f));  // 1 / (1 + z / 2), z = a / sqrt 2
        const float tail = t * pdf * ex2_approx(tail_exponent(t));
        const float cdf = x < 0.0f ? tail : 1.0f - tail;
        return fmaf(x, pdf, cdf);
    }
}

// ---------------------------------------------------------------------------
// packed float32 pairs (sm_100 and later: add / mul / fma on .f32x2)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 splat(float v) { return make_float2(v, v); }

// a where the sign bit of x is set, b otherwise (-0 counts as negative)
__device__ __forceinline__ float sel_neg(float x, float a, float b) {
    return static_cast<int>(__float_as_uint(x)) < 0 ? a : b;
}

// f'(x) on a pair, for 16-bit outputs (errors of order 1e-5 relative, far
// below half an fp16 / bf16 ulp).  Exponentials that can fall below
// float32's normal range are taken as 2^64 times their value and scaled back
// once, so subnormal results keep their value.
template <int ACT>
__device__ __forceinline__ float2 act_grad2(float2 x) {
    constexpr float k2m64 = 5.42101086242752217e-20f;  // 2^-64
    if constexpr (ACT == kActSilu) {
        // e = exp(-a), a = min(|x|, 128); r = 1 / (1 + e); s = sigma(x) is r
        // for x >= 0 and e r for x < 0, and in both cases
        // SiLU'(x) = s (1 + x (1 - s)) = s + x (r e r)
        const float2 a = make_float2(fminf(fabsf(x.x), 128.0f), fminf(fabsf(x.y), 128.0f));
        const float2 y = fma2(a, splat(-kLog2e), splat(64.0f));
        const float2 e = mul2(make_float2(ex2_approx(y.x), ex2_approx(y.y)), splat(k2m64));
        const float2 d = fma2(e, splat(1.0f), splat(1.0f));
        const float2 r = make_float2(rcp_approx(d.x), rcp_approx(d.y));
        const float2 er = mul2(e, r);
        const float2 s = make_float2(sel_neg(x.x, er.x, r.x), sel_neg(x.y, er.y, r.y));
        return fma2(x, mul2(r, er), s);
    } else {
        // a = min(|x|, 16); p = 2^64 phi(a); t = 1 / (1 + a / (2 sqrt 2));
        // tail = Phi(-a) = t phi(a) 2^Q(t).  With g = tail - a phi(a):
        // GELU'(x) = g for x < 0 and 1 - g for x >= 0
        const float2 a = make_float2(fminf(fabsf(x.x), 16.0f), fminf(fabsf(x.y), 16.0f));
        const float2 y = fma2(mul2(a, a), splat(-0.5f * kLog2e), splat(kLog2InvSqrt2Pi + 64.0f));
        const float2 p = make_float2(ex2_approx(y.x), ex2_approx(y.y));
        const float2 dt = fma2(a, splat(0.35355339059327376f), splat(1.0f));
        const float2 t = make_float2(rcp_approx(dt.x), rcp_approx(dt.y));
        float2 q = splat(kQ9);
        q = fma2(q, t, splat(kQ8));
        q = fma2(q, t, splat(kQ7));
        q = fma2(q, t, splat(kQ6));
        q = fma2(q, t, splat(kQ5));
        q = fma2(q, t, splat(kQ4));
        q = fma2(q, t, splat(kQ3));
        q = fma2(q, t, splat(kQ2));
        q = fma2(q, t, splat(kQ1));
        q = fma2(q, t, splat(kQ0));
        const float2 tg = mul2(t, make_float2(ex2_approx(q.x), ex2_approx(q.y)));
        const float2 g = mul2(fma2(a, splat(-1.0f), tg), p);  // 2^64 g
        // -g where x >= 0, g where x < 0; base 1 where x >= 0
        const uint32_t sx = __float_as_uint(x.x) & 0x80000000u, sy = __float_as_uint(x.y) & 0x80000000u;
        const float2 h = make_float2(__uint_as_float(__float_as_uint(g.x) ^ sx ^ 0x80000000u),
                                     __uint_as_float(__float_as_uint(g.y) ^ sy ^ 0x80000000u));
        const float2 base = make_float2(sx ? 0.0f : 1.0f, sy ? 0.0f : 1.0f);
        return fma2(h, splat(k2m64), base);
    }
}

// dx for one 16-byte vector of dy and preact (16-bit outputs: packed pairs)
template <typename T, int ACT>
__device__ __forceinline__ uint4 act_vec(const uint4 &dy, const uint4 &pre) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    float d[V], x[V], o[V];
    Tr::unpack(dy, d);
    Tr::unpack(pre, x);
    if constexpr (std::is_same_v<T, float>) {
#pragma unroll
        for (int e = 0; e < V; ++e) o[e] = d[e] * act_grad<ACT, true>(x[e]);
    } else {
#pragma unroll
        for (int e = 0; e < V; e += 2) {
            const float2 r = mul2(make_float2(d[e], d[e + 1]), act_grad2<ACT>(make_float2(x[e], x[e + 1])));
            o[e] = r.x;
            o[e + 1] = r.y;
        }
    }
    return Tr::pack(o);
}

template <typename T, int ACT>
__device__ __forceinline__ float act_one(float dy, float x) {
    return dy * act_grad<ACT, std::is_same_v<T, float>>(x);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// Launch shape per activation (threads per CTA, 16-byte vectors per lane per
// chunk, ring stages per warp), the fastest of a sweep at 16384 x 4096 bf16:
// SiLU 512 / 2 / 3 (1 KB chunks, 96 KB of rings), GELU 768 / 4 / 2 (2 KB
// chunks, 192 KB).  GELU computes longer per byte and gains from more warps
// and larger copies.
template <int ACT>
struct ActShape;
template <>
struct ActShape<kActSilu> {
    static constexpr int kThreads = 512, kVecPerLane = 2, kStages = 3;
};
template <>
struct ActShape<kActGelu> {
    static constexpr int kThreads = 768, kVecPerLane = 4, kStages = 2;
};

// One CTA per SM.  The aligned part of the tensors is cut into chunks of
// 32 lanes x VL 16-byte vectors per input; each CTA takes a contiguous run of
// chunks and deals them to its warps in turn.  Every warp runs its own ring
// of S chunks in shared memory: lane 0 keeps the warp's next chunks of dy
// and preact in flight with 1-D bulk copies, the lanes work through the
// current chunk in place, and a warp-level sync frees the stage for the next
// copy.  Warps never wait on one another, so copies stay in flight while any
// warp computes.  dx leaves with 16-byte streaming stores.  Elements after
// the last full chunk, and all of them when a pointer is not 16-byte aligned,
// take a grid-stride loop of plain loads.  dx may alias dy: a chunk's dx is
// written only after its copy of dy has landed, and the tail loop reads each
// element before the same thread writes it.
template <typename T, int ACT>
__global__ void __launch_bounds__(ActShape<ACT>::kThreads, 1) act_bwd_kernel(const ActParams p) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int VL = ActShape<ACT>::kVecPerLane;
    constexpr int S = ActShape<ACT>::kStages;
    constexpr uint32_t kChunkBytes = 32 * VL * 16;  // per input
    constexpr int64_t kChunkElems = kChunkBytes / sizeof(T);
    constexpr int kWarps = ActShape<ACT>::kThreads / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    const T *dy = static_cast<const T *>(p.dy);
    const T *pre = static_cast<const T *>(p.pre);
    T *dx = static_cast<T *>(p.dx);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char *ring = smem + (size_t)warp * S * 2 * kChunkBytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + (size_t)kWarps * S * 2 * kChunkBytes) + warp * S;

    // this CTA's run of chunks, and this warp's share of it (every kWarps-th)
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t base = p.nchunks / G, rem = p.nchunks % G;
    const int64_t c0 = b * base + (b < rem ? b : rem);
    const int64_t ncta = base + (b < rem ? 1 : 0);
    const int64_t nw = ncta > warp ? (ncta - warp + kWarps - 1) / kWarps : 0;

    if (nw > 0) {
        if (lane == 0) {
            for (int i = 0; i < S; ++i) mbar_init(&bar[i], 1);
            fence_barrier_init();
        }
        __syncwarp();
        int64_t issued = 0;
        auto issue = [&]() {
            const int st = static_cast<int>(issued % S);
            unsigned char *dst = ring + (size_t)st * 2 * kChunkBytes;
            const int64_t e0 = (c0 + warp + issued * kWarps) * kChunkElems;
            mbar_arrive_expect_tx(&bar[st], 2 * kChunkBytes);
            bulk_load_nohint(dst, dy + e0, kChunkBytes, &bar[st]);
            bulk_load_nohint(dst + kChunkBytes, pre + e0, kChunkBytes, &bar[st]);
            ++issued;
        };
        if (lane == 0)
            while (issued < nw && issued < S) issue();
        int64_t k = 0;
        for (; k < nw; ++k) {
            const int st = static_cast<int>(k % S);
            const bool ok = mbar_wait_bounded(&bar[st], static_cast<uint32_t>((k / S) & 1));
            if (!ok) record_error(p.err, kErrWaitFull);
            if (__any_sync(0xffffffffu, !ok)) break;
            // the lanes work through the chunk in place, one vector of each
            // input at a time, so registers do not grow with the chunk
            const unsigned char *src = ring + (size_t)st * 2 * kChunkBytes + (size_t)lane * 16;
            T *out = dx + (c0 + warp + k * kWarps) * kChunkElems + (int64_t)lane * V;
#pragma unroll
            for (int j = 0; j < VL; ++j)
                st_global_cs_v4(out + j * 32 * V, act_vec<T, ACT>(ld_shared_v4(src + j * 512),
                                                                   ld_shared_v4(src + kChunkBytes + j * 512)));
            // the warp sync orders every lane's shared loads before lane 0's
            // proxy fence and the copy that refills the stage
            __syncwarp();
            if (lane == 0 && issued < nw) {
                fence_proxy_async();
                issue();
            }
        }
        // after an abort, wait (bounded) for this warp's copies still in
        // flight before the CTA's shared memory is released
        if (lane == 0) {
            for (int64_t kk = k; kk < issued; ++kk) {
                if (!mbar_wait_bounded(&bar[kk % S], static_cast<uint32_t>((kk / S) & 1), kDrainNs)) {
                    record_error(p.err, kErrDrain);
                    break;
                }
            }
        }
    }

    // the rest: [nchunks * kChunkElems, n)
    const int64_t start = p.nchunks * kChunkElems;
    const int64_t tg = (int64_t)blockIdx.x * blockDim.x + tid;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t nvec = p.vec_ok ? (p.n - start) / V : 0;
    for (int64_t i = tg; i < nvec; i += stride) {
        const int64_t e = start + i * V;
        st_global_cs_v4(dx + e, act_vec<T, ACT>(ld_global_nc_v4(dy + e), ld_global_nc_v4(pre + e)));
    }
    for (int64_t j = start + nvec * V + tg; j < p.n; j += stride)
        Tr::store1(dx + j, act_one<T, ACT>(Tr::load1(dy + j), Tr::load1(pre + j)));
}

template <typename T, int ACT>
cudaError_t act_launch(const void *dy, const void *pre, void *dx, int64_t n, int sms, int *err, cudaStream_t s) {
    using Sh = ActShape<ACT>;
    constexpr int V = Traits<T>::kVec;
    constexpr int kWarps = Sh::kThreads / 32;
    constexpr int64_t kChunkElems = 32 * Sh::kVecPerLane * 16 / sizeof(T);
    static std::atomic<uint64_t> done{0};
    cudaError_t e = ensure_smem_optin(act_bwd_kernel<T, ACT>, done);
    if (e != cudaSuccess) return e;
    ActParams p;
    p.dy = dy;
    p.pre = pre;
    p.dx = dx;
    p.n = n;
    p.err = err;
    p.vec_ok = ((reinterpret_cast<uintptr_t>(dy) | reinterpret_cast<uintptr_t>(pre) |
                 reinterpret_cast<uintptr_t>(dx)) & 15u) == 0;
    p.nchunks = p.vec_ok ? n / kChunkElems : 0;
    const size_t smem = (size_t)kWarps * Sh::kStages * (2 * 32 * Sh::kVecPerLane * 16 + sizeof(uint64_t));
    // one CTA per SM; fewer when there is less work
    const int64_t per_cta = (int64_t)Sh::kThreads * Sh::kVecPerLane * V;  // elements of one round of chunks
    const int64_t want = p.nchunks > 0 ? (p.nchunks + kWarps - 1) / kWarps : (n + per_cta - 1) / per_cta;
    int64_t blocks = want < sms ? want : sms;
    if (blocks < 1) blocks = 1;
    act_bwd_kernel<T, ACT><<<static_cast<unsigned>(blocks), Sh::kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int ACT>
cudaError_t act_dtype(int dtype, const void *dy, const void *pre, void *dx, int64_t n, int sms, int *err,
                      cudaStream_t s) {
    switch (dtype) {
        case 0: return act_launch<float, ACT>(dy, pre, dx, n, sms, err, s);
        case 1: return act_launch<__half, ACT>(dy, pre, dx, n, sms, err, s);
        case 2: return act_launch<__nv_bfloat16, ACT>(dy, pre, dx, n, sms, err, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_act_bwd(int act, int dtype, const void *dy, const void *pre, void *dx, int64_t n, int sms,
                           int *err, cudaStream_t s) {
    return act == kActSilu ? act_dtype<kActSilu>(dtype, dy, pre, dx, n, sms, err, s)
                           : act_dtype<kActGelu>(dtype, dy, pre, dx, n, sms, err, s);
}

}  // namespace gbn
