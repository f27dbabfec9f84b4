// gbn_device.cuh -- device-side building blocks shared by the forward and
// backward kernels: 16-byte vector load/store traits for the three storage
// dtypes, inline-PTX wrappers for shared-memory mbarriers and 1-D bulk
// (TMA) copies, named barriers, and bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gbn_launch.h"

namespace gbn {

// ---------------------------------------------------------------------------
// storage dtypes: a 16-byte vector holds kVec elements
// ---------------------------------------------------------------------------
template <typename T>
struct Traits;

template <>
struct Traits<float> {
    static constexpr int kVec = 4;
    __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float *f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static float load1(const float *p) { return *p; }
    __device__ __forceinline__ static void store1(float *p, float v) { *p = v; }
};

template <>
struct Traits<__half> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 p = __half22float2(h);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
    __device__ __forceinline__ static uint4 pack(const float *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ __forceinline__ static float load1(const __half *p) { return __half2float(*p); }
    __device__ __forceinline__ static void store1(__half *p, float v) { *p = __float2half_rn(v); }
};

template <>
struct Traits<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // a bf16 is the upper half of the float with the same bits
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ __forceinline__ static float load1(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    __device__ __forceinline__ static void store1(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
};

// ---------------------------------------------------------------------------
// error flag: one per device, read and cleared by gbn_device_error()
// ---------------------------------------------------------------------------
enum : int {
    kErrWaitFull = 1,   // a bulk copy did not complete within the wait limit
    kErrDrain = 2,      // copies still in flight at exit after the wait limit
};

// the flag lives in norm_bwd.cu; kernels receive its address in their
// parameter block (no relocatable device code needed)
__device__ __forceinline__ void record_error(int *flag, int code) { atomicCAS(flag, 0, code); }

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// makes barrier initialisation visible to the async (bulk copy) proxy
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// one arrival (release semantics: this thread's earlier writes are visible
// to a thread that then observes the phase complete)
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// non-blocking look at whether the phase with the given parity completed
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete, giving up
// after ~limit_ns (checked on the global timer before the first suspending
// poll and every 64 polls after it) or 2^28 polls, whichever comes first.
// Returns false on giving up.  The first look does not suspend, so a limit
// far below a copy's latency gives up at once on a phase still open.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitNs) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        if ((it & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
        if (mbar_try_wait(bar, parity)) return true;
    }
    return false;
}

// a counter in shared memory written by one thread and polled by others
__device__ __forceinline__ void st_release_shared(int *p, int v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_shared(const int *p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}

// Waits until *counter > k, giving up after ~limit_ns (checked on the global
// timer before the first poll that follows a failed look, then every 64
// polls).  Returns false on giving up.
__device__ __forceinline__ bool wait_counter_above(const int *counter, int k, uint64_t limit_ns) {
    if (ld_acquire_shared(counter) > k) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        if ((it & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
        if (ld_acquire_shared(counter) > k) return true;
    }
    return false;
}

// mbar_wait_bounded by every lane of a warp, with one outcome for the warp:
// false if any lane gave up, so that the warp stops as a whole and no lane
// is left behind in a later warp-wide shuffle or __syncwarp
__device__ __forceinline__ bool warp_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const bool ok = mbar_wait_bounded(bar, parity, limit_ns);
    return __all_sync(0xffffffffu, ok) != 0;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` of
// transaction count on `bar`.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_load_nohint(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// programmatic dependent launch: let the next kernel on the stream launch
// now (it waits in griddep_wait until this grid has finished and its
// memory is visible)
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// barrier over `count` threads (a multiple of 32) of this CTA, id in 1..15.
// bar.sync is the aligned form: each participating warp must execute it
// converged.  Callers often reach it right after a branch taken by one lane
// (lane 0 storing a warp's sum), and a warp need not reconverge after a
// branch on its own, so the warp is reconverged first.
__device__ __forceinline__ void named_barrier(int id, int count) {
    __syncwarp();
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// 16-byte global load through the read-only path, no L1 allocation
__device__ __forceinline__ uint4 ld_global_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte streaming global store
__device__ __forceinline__ void st_global_cs_v4(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------
// butterfly sum over the 32 lanes; every lane ends with the same bits (each
// step adds the same two operands on both partner lanes)
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Row partition of M rows over G blocks: block b owns [row_begin, row_begin + rows).
__host__ __device__ __forceinline__ void block_rows(int64_t M, int G, int b, int64_t &row_begin, int &rows) {
    const int64_t base = M / G;
    const int64_t rem = M % G;
    row_begin = b * base + (b < rem ? b : rem);
    rows = static_cast<int>(base + (b < rem ? 1 : 0));
}

}  // namespace gbn

namespace gbn {

// Floats of reduction scratch per slot: 128, as [buffer][NQ][16 warps].
constexpr int kRedStride = 16;

// Sums the NQ values of every thread of one row slot (W warps, tpr = 32*W
// threads, named barrier bar_id) and leaves the totals in v on every thread
// of the slot: a butterfly within each warp, then the W warp sums added in
// warp order (read as 16-byte vectors).  `buf` is this slot's scratch of
// NQ*kRedStride floats; consecutive calls must alternate buffers.  Also
// returns, uniformly over the slot, whether any of its threads passed
// give_up = true (a wait that ran out); `flag` is the slot's abort flag.
// Butterfly sum of two values over the 32 lanes with six shuffles: after the
// first exchange, lanes 0-15 carry partial sums of v0 and lanes 16-31 of v1;
// four more butterfly steps finish both (each half's lanes end with the same
// bits), and a last exchange gives every lane both totals.
__device__ __forceinline__ void warp_sum2(float &v0, float &v1) {
    const bool hi = (threadIdx.x & 16) != 0;
    const float send = hi ? v0 : v1;
    const float keep = hi ? v1 : v0;
    float t = keep + __shfl_xor_sync(0xffffffffu, send, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    const float other = __shfl_xor_sync(0xffffffffu, t, 16);
    v0 = hi ? other : t;
    v1 = hi ? t : other;
}

template <int NQ>
__device__ __forceinline__ bool slot_reduce(float (&v)[NQ], float *buf, volatile int *flag, bool give_up,
                                            int W, int warp, int lane, int bar_id, int tpr) {
    if constexpr (NQ == 2) {
        warp_sum2(v[0], v[1]);
    } else {
#pragma unroll
        for (int q = 0; q < NQ; ++q) v[q] = warp_sum(v[q]);
    }
    if (W == 1) return __any_sync(0xffffffffu, give_up) != 0;
    if (give_up) *flag = 1;
    if (lane == 0) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) buf[q * kRedStride + warp] = v[q];
    }
    named_barrier(bar_id, tpr);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        const float *b = buf + q * kRedStride;
        if (W == 2) {
            const float2 t = *reinterpret_cast<const float2 *>(b);
            v[q] = t.x + t.y;
        } else {
            float s = 0.f;
            for (int w = 0; w < W; w += 4) {
                const float4 t = *reinterpret_cast<const float4 *>(b + w);
                s = w == 0 ? t.x : s + t.x;
                s += t.y;
                s += t.z;
                s += t.w;
            }
            v[q] = s;
        }
    }
    return *flag != 0;
}

// Stage ring position of one slot: stage index and the parity of the use of
// that stage, advanced without division.
struct RingPos {
    int stage = 0;
    uint32_t parity = 0;
    __device__ __forceinline__ void next(int S) {
        if (++stage == S) {
            stage = 0;
            parity ^= 1u;
        }
    }
};

// Block-wide sum for the plain-load kernels (blockDim.x = 32 * warps); every
// thread gets the same bits.  `sm` holds one float per warp.
__device__ __forceinline__ float block_sum(float v, float *sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    v = warp_sum(v);
    if (lane == 0) sm[warp] = v;
    __syncthreads();
    float s = sm[0];
    for (int w = 1; w < nw; ++w) s += sm[w];
    __syncthreads();
    return s;
}

}  // namespace gbn

namespace gbn {

// ---------------------------------------------------------------------------
// dgamma / dbeta column sums of the [G][ldp] partial rows, in one fixed order
// ---------------------------------------------------------------------------
// Two shapes: 8 slices (256-thread CTAs) beside the warp-specialised rows
// kernel, where they fit beside it on an SM and so start, as its
// programmatic dependent, as soon as that grid completes (16 slices measured
// 1.2-1.6 us slower there, 4 slices slower too); 16 slices (512 threads)
// beside the other rows kernels, which leave no room for them (8 slices
// measured up to 2 us slower there).
template <int SLICES>
struct ColsumShape {
    static constexpr int kBatch = 192 / SLICES;  // loads a thread issues together: one batch up to G = 192
};

// Packed float32 pairs (sm_100 and later: fma / mul / add on .f32x2): each
// half rounds as the scalar instruction would, so a pair computes exactly
// what two scalar operations compute, in one issue.
__device__ __forceinline__ float2 pair_fma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 pair_mul(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 pair_add(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// elements 2i, 2i+1 of an unpacked vector as a pair
__device__ __forceinline__ float2 pair_at(const float *f, int i) { return make_float2(f[2 * i], f[2 * i + 1]); }

// VEC consecutive fp32 values from L2, VEC = 1, 2 or 4 (address aligned to
// 4 * VEC bytes)
template <int VEC>
__device__ __forceinline__ void ldcg_vec(const float *p, float (&v)[VEC]) {
    if constexpr (VEC == 4) {
        const float4 t = __ldcg(reinterpret_cast<const float4 *>(p));
        v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
    } else if constexpr (VEC == 2) {
        const float2 t = __ldcg(reinterpret_cast<const float2 *>(p));
        v[0] = t.x, v[1] = t.y;
    } else {
        v[0] = __ldcg(p);
    }
}

// sum over g < G of P[g*ldp + c], for c in [c0, c1), 32 * VEC columns a
// pass: lane q of slice s (threads 32*s + q, s < SLICES) holds columns
// cb + VEC*q .. cb + VEC*q + VEC-1 and adds rows s, s + SLICES, ... of each
// in increasing order (ColsumShape::kBatch loads of VEC values issued
// together), then slice 0 adds the slice sums in slice order.  Each
// column's order depends on SLICES only, so every VEC and CTA shape with
// the same SLICES gives the same bits per column.  Needs at least
// 32 * SLICES threads (the others only join the barriers),
// sm[SLICES * (32 * VEC + 1)], P aligned to 4 * VEC bytes and ldp a
// multiple of VEC (a lane's VEC values then never cross the end of a
// partial row: columns from N up to ldp are padding that is read, never
// stored).  P is read through L2 (written by an earlier grid).  store(c,
// sum) writes the result of column c.
template <int SLICES, int VEC, typename Store>
__device__ __forceinline__ void colsum_range(const float *P, int G, int ldp, int c0, int c1, Store store,
                                             float *sm) {
    constexpr int kColsumSlices = SLICES;
    constexpr int kColsumBatch = ColsumShape<SLICES>::kBatch;
    constexpr int W = 32 * VEC + 1;  // row pitch of sm
    const int q = threadIdx.x & 31, slice = threadIdx.x >> 5;
    for (int cb = c0; cb < c1; cb += 32 * VEC) {
        const int c = cb + q * VEC;
        float a[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) a[j] = 0.f;
        if (slice < kColsumSlices && c < c1) {
            for (int g0 = slice; g0 < G; g0 += kColsumSlices * kColsumBatch) {
                float v[kColsumBatch][VEC];
#pragma unroll
                for (int u = 0; u < kColsumBatch; ++u) {
                    const int g = g0 + u * kColsumSlices;
                    if constexpr (VEC == 1) {
                        // every load is issued (rows past the end read the
                        // last row again and count as 0), so the compiler
                        // keeps the whole batch in flight: 65536x1024
                        // LayerNorm 1.4 us faster than a branch per load
                        float t[1];
                        ldcg_vec<1>(P + (size_t)(g < G ? g : G - 1) * ldp + c, t);
                        v[u][0] = g < G ? t[0] : 0.f;
                    } else if (g < G) {
                        // wider lanes keep the branch: with the unconditional
                        // form the compiler interleaved loads and adds and
                        // 1151x8192 LayerNorm lost 4.4 us
                        ldcg_vec<VEC>(P + (size_t)g * ldp + c, v[u]);
                    } else {
#pragma unroll
                        for (int j = 0; j < VEC; ++j) v[u][j] = 0.f;
                    }
                }
#pragma unroll
                for (int u = 0; u < kColsumBatch; ++u)
#pragma unroll
                    for (int j = 0; j < VEC; ++j) a[j] += v[u][j];
            }
        }
        if (slice < kColsumSlices)
#pragma unroll
            for (int j = 0; j < VEC; ++j) sm[slice * W + q * VEC + j] = a[j];
        __syncthreads();
        if (slice == 0) {
#pragma unroll
            for (int i = q; i < 32 * VEC; i += 32) {
                if (cb + i < c1) {
                    float t = sm[i];
                    for (int s2 = 1; s2 < kColsumSlices; ++s2) t += sm[s2 * W + i];
                    store(cb + i, t);
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace gbn
