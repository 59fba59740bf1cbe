// Kernels of the fused data-parallel step for sm_103a (GB300).
//
// The path is a pure HBM stream: per element it reads R bf16 gradients and
// the fp32 master/m/v, and writes master/m/v and R bf16 parameters, about
// 0.3 flop per byte, so there is no contraction for the tensor cores.  What
// matters is that every byte moves once, in full 32-byte sectors, with
// enough loads in flight per SM to cover HBM latency:
//   * one thread owns 8 consecutive elements, so each replica's gradient and
//     parameter is one 16-byte access and each fp32 array two; a warp
//     touches 512 contiguous bytes per bf16 stream and 1 KiB per fp32
//     stream.  The reducing step with fp32 accumulators takes 4 elements
//     per thread instead (its loads are three times larger), and so does
//     the first accumulation micro-step (a store-heavy widening copy);
//   * all of a thread's loads (R + 6 vectors, R = 8 gives 224 bytes) are
//     issued before any arithmetic, so each thread has them all in flight;
//   * streaming cache hints (ld/st .cs, evict-first) keep the single-use
//     stream from displacing other kernels' working sets in L2;
//   * one vector per thread and as many blocks as the range needs: blocks
//     retire and are replaced independently, so loads keep streaming while
//     other warps compute (measured on GB300: 2.66 ms for the 336M-parameter
//     R=8 step, against 2.93 ms for a grid-stride grid capped at the
//     resident block count, whose warps move through load/compute/store in
//     lock step).  The loop is still grid-stride so a CTA budget can cap it;
//   * consecutive buckets of one call are chained with programmatic
//     dependent launch: each block lets the next bucket's grid launch as
//     soon as it starts, and waits for the previous bucket's grid to finish
//     only when its own work is done.  Buckets touch disjoint elements, so
//     the next bucket's blocks fill SMs as this bucket's tail drains, and
//     the final wait keeps completion transitive (the last bucket of a call
//     completes only after every earlier one).  A step's first bucket (and
//     a rank step) is a programmatic dependent too, but waits before it
//     touches memory, since it may read what the previous kernel wrote;
//   * under a CTA budget the same per-vector code runs in wide CTAs (768
//     threads, one per SM, grid = the budget, each thread striding over the
//     range), with the fp32 state in 32-byte accesses where it is 32-byte
//     aligned: one SM then streams about 98 GB/s, so a budget of about 70
//     SMs reaches HBM bandwidth.
//
// Arithmetic is IEEE binary32 with each operation rounded on its own
// (__fadd_rn/__fmul_rn/__fdiv_rn/__fsqrt_rn never contract to FMA), in the
// order given in include/cc_dp.h, so the results are bit-identical to any
// other correctly rounded evaluation of that order.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "cc_dp_device.cuh"
#include "cc_dp_internal.h"

// Launch shape (compile-time tuning parameters).
#ifndef CC_DP_THREADS
#define CC_DP_THREADS 256      // threads per block
#endif
#ifndef CC_DP_MIN_BLOCKS
#define CC_DP_MIN_BLOCKS 1     // __launch_bounds__ minimum resident blocks per SM
#endif
#ifndef CC_DP_BLOCKS_PER_SM
#define CC_DP_BLOCKS_PER_SM 0  // grid = SMs x this; 0 = SMs x occupancy
#endif
#ifndef CC_DP_PERSISTENT
#define CC_DP_PERSISTENT 0     // 1: cap the grid at SMs x resident blocks
#endif
#ifndef CC_DP_PDL
#define CC_DP_PDL 1            // chain consecutive buckets with programmatic launch
#endif
#ifndef CC_DP_PDL_FIRST
#define CC_DP_PDL_FIRST 1      // a step's first bucket too, waiting for the previous step
#endif
#ifndef CC_DP_ACC_HALF
#define CC_DP_ACC_HALF 1       // accumulator variant: 4 elements per thread
#endif
#ifndef CC_DP_PLAIN_HALF
#define CC_DP_PLAIN_HALF 0     // plain variant: 4 elements per thread (measured: no gain)
#endif
#ifndef CC_DP_ACCUM_FIRST_HALF
#define CC_DP_ACCUM_FIRST_HALF 1  // first micro-step: 4 elements per thread
#endif

namespace ccdp {
namespace {

using namespace dev;

constexpr int kThreads = CC_DP_THREADS;
#ifndef CC_DP_WIDE_THREADS
#define CC_DP_WIDE_THREADS 768  // threads of one CTA of the CTA-budget form
#endif
constexpr int kWideThreads = CC_DP_WIDE_THREADS;
#ifndef CC_DP_WIDE_V8
#define CC_DP_WIDE_V8 1         // the wide form's fp32 state in 256-bit accesses where aligned
#endif
constexpr bool kWideV8 = CC_DP_WIDE_V8 != 0;
#ifndef CC_DP_FULL_V8
#define CC_DP_FULL_V8 0         // the whole-GPU form too (measured slower: off)
#endif
constexpr bool kFullV8 = CC_DP_FULL_V8 != 0;

struct FusedParams {
    const uint4 *g[CC_MAX_R];      // 8 bf16 per vector
    const float4 *acc[CC_MAX_R];   // 2 float4 per vector
    uint4 *out[CC_MAX_R];
    float4 *master, *m, *v;        // 2 float4 per vector
    AdamScalars c;
    size_t vec_begin;              // first 8-element vector of the range
    size_t num_vec;                // full vectors in the range
    size_t tail_begin;             // first element of the partial vector
    int tail_len;                  // 0..7 elements after the full vectors
    int wait_first;                // wait for the preceding grid before any access
    int v8;                        // master/m/v 32-byte aligned: 256-bit accesses (wide form)
};

// 256-bit streaming accesses of 8 consecutive floats (sm_100 and later; the
// address must be 32-byte aligned).
__device__ __forceinline__ void ldcs8(const float *p, float (&r)[8]) {
    asm volatile("ld.global.cs.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]),
                   "=f"(r[6]), "=f"(r[7])
                 : "l"(p));
}
__device__ __forceinline__ void stcs8(float *p, const float (&r)[8]) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 ::"l"(p), "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]),
                   "f"(r[6]), "f"(r[7])
                 : "memory");
}

// ONE_OUT: the parameters go to out[0] only (one rank's own slab in the
// multi-GPU form, from where the AllGather distributes them); otherwise to
// all R replica slabs.
// V8: the fp32 state moves as one 32-byte access per array instead of two
// 16-byte ones (fewer memory instructions; the wide CTA-budget form).
template <int R, bool ACC, bool ONE_OUT, bool FAST, bool V8 = false>
__device__ __forceinline__ void fused_vector(const FusedParams &p, size_t vi) {
    // Issue every load of this vector before any arithmetic.
    uint4 gq[R];
#pragma unroll
    for (int r = 0; r < R; ++r) gq[r] = __ldcs(p.g[r] + vi);
    float4 aq[ACC ? R : 1][2];
    if constexpr (ACC) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            aq[r][0] = __ldcs(p.acc[r] + 2 * vi);
            aq[r][1] = __ldcs(p.acc[r] + 2 * vi + 1);
        }
    }
    float pw[8], mm[8], vv[8];
    if constexpr (V8) {
        ldcs8(reinterpret_cast<const float *>(p.master) + 8 * vi, pw);
        ldcs8(reinterpret_cast<const float *>(p.m) + 8 * vi, mm);
        ldcs8(reinterpret_cast<const float *>(p.v) + 8 * vi, vv);
    } else {
        const float4 w0 = __ldcs(p.master + 2 * vi), w1 = __ldcs(p.master + 2 * vi + 1);
        const float4 m0 = __ldcs(p.m + 2 * vi), m1 = __ldcs(p.m + 2 * vi + 1);
        const float4 v0 = __ldcs(p.v + 2 * vi), v1 = __ldcs(p.v + 2 * vi + 1);
        const float w8[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const float m8[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        const float v8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            pw[k] = w8[k];
            mm[k] = m8[k];
            vv[k] = v8[k];
        }
    }

    // Reduce in replica order.
    float s[8];
    if constexpr (ACC) {
        float a0[8] = {aq[0][0].x, aq[0][0].y, aq[0][0].z, aq[0][0].w,
                       aq[0][1].x, aq[0][1].y, aq[0][1].z, aq[0][1].w};
        add8_bf16(a0, gq[0]);                      // acc[0] + g[0]
#pragma unroll
        for (int k = 0; k < 8; ++k) s[k] = a0[k];
    } else {
        widen8(gq[0], s);
    }
#pragma unroll
    for (int r = 1; r < R; ++r) {
        if constexpr (ACC) {
            float ar[8] = {aq[r][0].x, aq[r][0].y, aq[r][0].z, aq[r][0].w,
                           aq[r][1].x, aq[r][1].y, aq[r][1].z, aq[r][1].w};
            add8_bf16(ar, gq[r]);                  // acc[r] + g[r]
#pragma unroll
            for (int k = 0; k < 8; ++k) s[k] = __fadd_rn(s[k], ar[k]);
        } else {
            add8_bf16(s, gq[r]);
        }
    }

#pragma unroll
    for (int k = 0; k < 8; ++k) adamw_step<FAST>(s[k], pw[k], mm[k], vv[k], p.c);

    if constexpr (V8) {
        stcs8(reinterpret_cast<float *>(p.master) + 8 * vi, pw);
        stcs8(reinterpret_cast<float *>(p.m) + 8 * vi, mm);
        stcs8(reinterpret_cast<float *>(p.v) + 8 * vi, vv);
    } else {
        __stcs(p.master + 2 * vi, make_float4(pw[0], pw[1], pw[2], pw[3]));
        __stcs(p.master + 2 * vi + 1, make_float4(pw[4], pw[5], pw[6], pw[7]));
        __stcs(p.m + 2 * vi, make_float4(mm[0], mm[1], mm[2], mm[3]));
        __stcs(p.m + 2 * vi + 1, make_float4(mm[4], mm[5], mm[6], mm[7]));
        __stcs(p.v + 2 * vi, make_float4(vv[0], vv[1], vv[2], vv[3]));
        __stcs(p.v + 2 * vi + 1, make_float4(vv[4], vv[5], vv[6], vv[7]));
    }
    uint4 o;
    o.x = pack_bf16x2(pw[0], pw[1]);
    o.y = pack_bf16x2(pw[2], pw[3]);
    o.z = pack_bf16x2(pw[4], pw[5]);
    o.w = pack_bf16x2(pw[6], pw[7]);
#pragma unroll
    for (int r = 0; r < (ONE_OUT ? 1 : R); ++r) __stcs(p.out[r] + vi, o);
}

// Half vectors: one thread owns 4 consecutive elements.  A warp's fp32
// accesses are then one 16-byte access per thread, 512 contiguous bytes per
// instruction, every 32-byte sector written whole by one store; with 8
// elements per thread each fp32 store instruction half-fills 32 sectors
// and the next one fills the other halves.  The bf16 accesses become 8
// bytes per thread (256 contiguous bytes per warp instruction).  For the
// reducing step with accumulators it also halves the registers that the
// loads in flight take (R = 8: 480 bytes for a full vector, 142 registers
// and one 256-thread block per SM).
template <int R, bool ACC, bool ONE_OUT, bool FAST>
__device__ __forceinline__ void fused_half(const FusedParams &p, size_t hv) {
    uint2 gq[R];
    float4 aq[ACC ? R : 1];
#pragma unroll
    for (int r = 0; r < R; ++r) gq[r] = __ldcs(reinterpret_cast<const uint2 *>(p.g[r]) + hv);
    if constexpr (ACC) {
#pragma unroll
        for (int r = 0; r < R; ++r) aq[r] = __ldcs(p.acc[r] + hv);
    }
    const float4 w = __ldcs(p.master + hv);
    const float4 m = __ldcs(p.m + hv);
    const float4 v = __ldcs(p.v + hv);

    // Plain: g[0], then s + g[r].  Accumulated: acc[0] + g[0], then
    // s + (acc[r] + g[r]).  Replica order either way.
    float s[4];
    if constexpr (ACC) {
        s[0] = add_bf16_lo(aq[0].x, gq[0].x);
        s[1] = add_bf16_hi(aq[0].y, gq[0].x);
        s[2] = add_bf16_lo(aq[0].z, gq[0].y);
        s[3] = add_bf16_hi(aq[0].w, gq[0].y);
    } else {
        s[0] = bf16_lo(gq[0].x);
        s[1] = bf16_hi(gq[0].x);
        s[2] = bf16_lo(gq[0].y);
        s[3] = bf16_hi(gq[0].y);
    }
#pragma unroll
    for (int r = 1; r < R; ++r) {
        if constexpr (ACC) {
            s[0] = __fadd_rn(s[0], add_bf16_lo(aq[r].x, gq[r].x));
            s[1] = __fadd_rn(s[1], add_bf16_hi(aq[r].y, gq[r].x));
            s[2] = __fadd_rn(s[2], add_bf16_lo(aq[r].z, gq[r].y));
            s[3] = __fadd_rn(s[3], add_bf16_hi(aq[r].w, gq[r].y));
        } else {
            s[0] = add_bf16_lo(s[0], gq[r].x);
            s[1] = add_bf16_hi(s[1], gq[r].x);
            s[2] = add_bf16_lo(s[2], gq[r].y);
            s[3] = add_bf16_hi(s[3], gq[r].y);
        }
    }

    float pw[4] = {w.x, w.y, w.z, w.w};
    float mm[4] = {m.x, m.y, m.z, m.w};
    float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) adamw_step<FAST>(s[k], pw[k], mm[k], vv[k], p.c);

    __stcs(p.master + hv, make_float4(pw[0], pw[1], pw[2], pw[3]));
    __stcs(p.m + hv, make_float4(mm[0], mm[1], mm[2], mm[3]));
    __stcs(p.v + hv, make_float4(vv[0], vv[1], vv[2], vv[3]));
    const uint2 o = make_uint2(pack_bf16x2(pw[0], pw[1]), pack_bf16x2(pw[2], pw[3]));
#pragma unroll
    for (int r = 0; r < (ONE_OUT ? 1 : R); ++r)
        __stcs(reinterpret_cast<uint2 *>(p.out[r]) + hv, o);
}

// Threads per 8-element vector of the fused kernel.
template <bool ACC>
__host__ __device__ constexpr int threads_per_vector() {
    return (ACC ? CC_DP_ACC_HALF : CC_DP_PLAIN_HALF) ? 2 : 1;
}

// One element of the partial last vector (scalar accesses).
template <int R, bool ACC, bool ONE_OUT, bool FAST>
__device__ __forceinline__ void fused_scalar(const FusedParams &p, size_t i) {
    float s = bf16_at(p.g[0], i);
    if constexpr (ACC) s = __fadd_rn(reinterpret_cast<const float *>(p.acc[0])[i], s);
#pragma unroll
    for (int r = 1; r < R; ++r) {
        const float t = bf16_at(p.g[r], i);
        if constexpr (ACC)
            s = __fadd_rn(s, __fadd_rn(reinterpret_cast<const float *>(p.acc[r])[i], t));
        else
            s = __fadd_rn(s, t);
    }
    float *pm = reinterpret_cast<float *>(p.master);
    float *mm = reinterpret_cast<float *>(p.m);
    float *vv = reinterpret_cast<float *>(p.v);
    float pw = pm[i], m = mm[i], v = vv[i];
    adamw_step<FAST>(s, pw, m, v, p.c);
    pm[i] = pw;
    mm[i] = m;
    vv[i] = v;
    const __nv_bfloat16 b = __float2bfloat16_rn(pw);
#pragma unroll
    for (int r = 0; r < (ONE_OUT ? 1 : R); ++r) reinterpret_cast<__nv_bfloat16 *>(p.out[r])[i] = b;
}

// Programmatic dependent launch (sm_90+).  Without a programmatic
// predecessor both are no-ops.
__device__ __forceinline__ void allow_dependents_to_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_predecessor_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// THREADS = kThreads: the whole-GPU form, several CTAs per SM.  THREADS =
// kWideThreads: the CTA-budget form, one wide CTA per SM and a grid of at
// most the budget, each thread striding over the range.
template <int R, bool ACC, bool ONE_OUT, bool FAST, int THREADS>
__global__ void __launch_bounds__(THREADS, THREADS == kThreads ? CC_DP_MIN_BLOCKS : 1)
fused_step_kernel(const __grid_constant__ FusedParams p) {
    allow_dependents_to_launch();
    if (p.wait_first) wait_for_predecessor_grid();
    const size_t stride = static_cast<size_t>(gridDim.x) * THREADS;
    const size_t first = static_cast<size_t>(blockIdx.x) * THREADS + threadIdx.x;
    if constexpr (threads_per_vector<ACC>() == 2) {
        for (size_t i = first; i < 2 * p.num_vec; i += stride)
            fused_half<R, ACC, ONE_OUT, FAST>(p, 2 * p.vec_begin + i);
    } else if (((kWideV8 && THREADS == kWideThreads) || (kFullV8 && THREADS == kThreads)) &&
               p.v8) {
        for (size_t i = first; i < p.num_vec; i += stride)
            fused_vector<R, ACC, ONE_OUT, FAST, true>(p, p.vec_begin + i);
    } else {
        for (size_t i = first; i < p.num_vec; i += stride)
            fused_vector<R, ACC, ONE_OUT, FAST>(p, p.vec_begin + i);
    }
    if (blockIdx.x == gridDim.x - 1 && static_cast<int>(threadIdx.x) < p.tail_len)
        fused_scalar<R, ACC, ONE_OUT, FAST>(p, p.tail_begin + threadIdx.x);
    wait_for_predecessor_grid();
}

// ---------------------------------------------------------------------------
// Local accumulation micro-step: acc[r] = g[r] on the first micro-step (a
// copy: no "0 +", so -0 stays -0), acc[r] + g[r] on later ones.  One thread
// owns one vector across all R replicas and issues every load of it before
// any add, like the fused kernel; one vector per thread.  Later micro-steps
// take 8-element vectors (R x 48 bytes in flight).  The first micro-step is
// a widening copy that writes twice what it reads; it takes 4-element half
// vectors so that each fp32 store instruction writes whole sectors (with 8
// elements per thread each store half-fills 32 sectors and stalls on the
// store queue: 2.54 against 2.30 ms for the 336M-parameter R=8 slab).
// ---------------------------------------------------------------------------
struct AccumParams {
    const uint4 *g[CC_MAX_R];
    float4 *acc[CC_MAX_R];
    size_t num_vec;
    size_t tail_begin;
    int tail_len;
};

template <int R>
__device__ __forceinline__ void accumulate_first(const AccumParams &p, size_t vi) {
    uint4 gq[R];
#pragma unroll
    for (int r = 0; r < R; ++r) gq[r] = __ldcs(p.g[r] + vi);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float t[8];
        widen8(gq[r], t);
        __stcs(p.acc[r] + 2 * vi, make_float4(t[0], t[1], t[2], t[3]));
        __stcs(p.acc[r] + 2 * vi + 1, make_float4(t[4], t[5], t[6], t[7]));
    }
}

// Half vector hv (elements 4*hv .. 4*hv+3): one 8-byte load and one
// 16-byte store per replica, whole sectors per warp instruction.
template <int R>
__device__ __forceinline__ void accumulate_first_half(const AccumParams &p, size_t hv) {
    uint2 gq[R];
#pragma unroll
    for (int r = 0; r < R; ++r) gq[r] = __ldcs(reinterpret_cast<const uint2 *>(p.g[r]) + hv);
#pragma unroll
    for (int r = 0; r < R; ++r)
        __stcs(p.acc[r] + hv, make_float4(bf16_lo(gq[r].x), bf16_hi(gq[r].x),
                                          bf16_lo(gq[r].y), bf16_hi(gq[r].y)));
}

// Threads per 8-element vector of the accumulation kernel.
template <bool FIRST>
__host__ __device__ constexpr int accum_threads_per_vector() {
    return (FIRST && CC_DP_ACCUM_FIRST_HALF) ? 2 : 1;
}

template <int R>
__device__ __forceinline__ void accumulate_later(const AccumParams &p, size_t vi) {
    uint4 gq[R];
    float4 aq[R][2];
#pragma unroll
    for (int r = 0; r < R; ++r) gq[r] = __ldcs(p.g[r] + vi);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        aq[r][0] = __ldcs(p.acc[r] + 2 * vi);
        aq[r][1] = __ldcs(p.acc[r] + 2 * vi + 1);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float a[8] = {aq[r][0].x, aq[r][0].y, aq[r][0].z, aq[r][0].w,
                      aq[r][1].x, aq[r][1].y, aq[r][1].z, aq[r][1].w};
        add8_bf16(a, gq[r]);
        __stcs(p.acc[r] + 2 * vi, make_float4(a[0], a[1], a[2], a[3]));
        __stcs(p.acc[r] + 2 * vi + 1, make_float4(a[4], a[5], a[6], a[7]));
    }
}

template <int R, bool FIRST>
__global__ void __launch_bounds__(kThreads)
accumulate_kernel(const __grid_constant__ AccumParams p) {
    const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
    const size_t first = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
    if constexpr (accum_threads_per_vector<FIRST>() == 2) {
        for (size_t i = first; i < 2 * p.num_vec; i += stride) accumulate_first_half<R>(p, i);
    } else {
        for (size_t i = first; i < p.num_vec; i += stride) {
            if constexpr (FIRST)
                accumulate_first<R>(p, i);
            else
                accumulate_later<R>(p, i);
        }
    }
    if (blockIdx.x == gridDim.x - 1 && static_cast<int>(threadIdx.x) < p.tail_len) {
        const size_t e = p.tail_begin + threadIdx.x;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float *a = reinterpret_cast<float *>(p.acc[r]);
            const float t = bf16_at(p.g[r], e);
            a[e] = FIRST ? t : __fadd_rn(a[e], t);
        }
    }
}

__global__ void __launch_bounds__(kThreads)
l2_flush_kernel(uint4 *buf, size_t num_vec, uint32_t salt) {
    const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
    for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
         i < num_vec; i += stride)
        buf[i] = make_uint4(salt, static_cast<uint32_t>(i), salt, 0u);
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------

using FusedKernel = void (*)(FusedParams);

// The one-output form exists without accumulators and in the exact
// arithmetic only (the multi-GPU rank step); other combinations with it are
// null.
// The wide (CTA-budget) form exists without the one-output switch.
template <int R>
FusedKernel pick_fused(bool acc, bool one_out, bool fast, bool wide) {
    if (wide) {
        if (one_out) return nullptr;
        if (fast)
            return acc ? fused_step_kernel<R, true, false, true, kWideThreads>
                       : fused_step_kernel<R, false, false, true, kWideThreads>;
        return acc ? fused_step_kernel<R, true, false, false, kWideThreads>
                   : fused_step_kernel<R, false, false, false, kWideThreads>;
    }
    if (one_out)
        return (acc || fast) ? nullptr : fused_step_kernel<R, false, true, false, kThreads>;
    if (fast)
        return acc ? fused_step_kernel<R, true, false, true, kThreads>
                   : fused_step_kernel<R, false, false, true, kThreads>;
    return acc ? fused_step_kernel<R, true, false, false, kThreads>
               : fused_step_kernel<R, false, false, false, kThreads>;
}

FusedKernel fused_kernel_for(int R, bool acc, bool one_out = false, bool fast = false,
                             bool wide = false) {
    switch (R) {
        case 1: return pick_fused<1>(acc, one_out, fast, wide);
        case 2: return pick_fused<2>(acc, one_out, fast, wide);
        case 3: return pick_fused<3>(acc, one_out, fast, wide);
        case 4: return pick_fused<4>(acc, one_out, fast, wide);
        case 5: return pick_fused<5>(acc, one_out, fast, wide);
        case 6: return pick_fused<6>(acc, one_out, fast, wide);
        case 7: return pick_fused<7>(acc, one_out, fast, wide);
        case 8: return pick_fused<8>(acc, one_out, fast, wide);
        case 9: return pick_fused<9>(acc, one_out, fast, wide);
        case 10: return pick_fused<10>(acc, one_out, fast, wide);
        case 11: return pick_fused<11>(acc, one_out, fast, wide);
        case 12: return pick_fused<12>(acc, one_out, fast, wide);
        case 13: return pick_fused<13>(acc, one_out, fast, wide);
        case 14: return pick_fused<14>(acc, one_out, fast, wide);
        case 15: return pick_fused<15>(acc, one_out, fast, wide);
        case 16: return pick_fused<16>(acc, one_out, fast, wide);
        default: return nullptr;
    }
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    cudaError_t status = cudaSuccess;
    int sm_count = 0;
    int major = 0, minor = 0;
    int fused_blocks_per_sm[CC_MAX_R + 1][2] = {};
};

DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mutex;

cudaError_t device_info(DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    DeviceInfo &d = g_devices[dev];
    std::lock_guard<std::mutex> lock(g_devices_mutex);
    if (!d.ready) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e == cudaSuccess) {
            d.sm_count = prop.multiProcessorCount;
            d.major = prop.major;
            d.minor = prop.minor;
            for (int r = 1; r <= CC_MAX_R && e == cudaSuccess; ++r)
                for (int a = 0; a < 2 && e == cudaSuccess; ++a)
                    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                        &d.fused_blocks_per_sm[r][a],
                        reinterpret_cast<const void *>(fused_kernel_for(r, a != 0)),
                        kThreads, 0);
        }
        d.status = e;
        d.ready = true;
    }
    *out = &d;
    return d.status;
}

size_t div_up(size_t a, size_t b) { return (a + b - 1) / b; }

}  // namespace

cudaError_t device_sm_count(int *count) {
    DeviceInfo *d = nullptr;
    const cudaError_t e = device_info(&d);
    if (e == cudaSuccess) *count = d->sm_count;
    return e;
}

cudaError_t check_device(int *major, int *minor) {
    DeviceInfo *d = nullptr;
    const cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return e;
    *major = d->major;
    *minor = d->minor;
    return cudaSuccess;
}

cudaError_t launch_fused(const Slabs &s, const AdamScalars &c, size_t begin,
                         size_t end, int max_ctas, bool chain, cudaStream_t stream,
                         bool wait_first) {
    if (end <= begin) return cudaSuccess;
    DeviceInfo *d = nullptr;
    cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return e;
    const bool acc = s.acc[0] != nullptr;
    const bool wide = max_ctas > 0;
    FusedKernel kern = fused_kernel_for(s.R, acc, s.one_out, s.fast, wide);
    if (!kern) return cudaErrorInvalidValue;
    FusedParams p{};
    for (int r = 0; r < s.R; ++r) {
        p.g[r] = static_cast<const uint4 *>(s.grads[r]);
        p.acc[r] = reinterpret_cast<const float4 *>(s.acc[r]);
        p.out[r] = static_cast<uint4 *>(s.out[r]);
    }
    p.master = reinterpret_cast<float4 *>(s.master);
    p.m = reinterpret_cast<float4 *>(s.m);
    p.v = reinterpret_cast<float4 *>(s.v);
    p.c = c;
    p.vec_begin = begin / CC_PAD_ELEMS;
    p.num_vec = (end - begin) / CC_PAD_ELEMS;
    p.tail_begin = begin + p.num_vec * CC_PAD_ELEMS;
    p.tail_len = static_cast<int>(end - p.tail_begin);
    p.v8 = (wide || kFullV8) && ((reinterpret_cast<uintptr_t>(s.master) | reinterpret_cast<uintptr_t>(s.m) |
                     reinterpret_cast<uintptr_t>(s.v)) % 32 == 0);
    wait_first = wait_first && CC_DP_PDL_FIRST;
    p.wait_first = wait_first && CC_DP_PDL;

    const size_t units = p.num_vec * (acc ? threads_per_vector<true>()
                                          : threads_per_vector<false>());
    const int threads = wide ? kWideThreads : kThreads;
    size_t blocks = div_up(units, static_cast<size_t>(threads));
    if (wide) {
        // the budget: at most max_ctas wide CTAs, one per SM
        if (blocks > static_cast<size_t>(max_ctas)) blocks = max_ctas;
    } else {
        const size_t per_sm = CC_DP_BLOCKS_PER_SM > 0
                                  ? static_cast<size_t>(CC_DP_BLOCKS_PER_SM)
                                  : static_cast<size_t>(d->fused_blocks_per_sm[s.R][acc ? 1 : 0]);
        const size_t resident = static_cast<size_t>(d->sm_count) * per_sm;
        if (CC_DP_PERSISTENT && resident > 0 && blocks > resident) blocks = resident;
    }
    if (blocks == 0) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ((chain || wait_first) && CC_DP_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

using AccumKernel = void (*)(AccumParams);

template <int R>
AccumKernel pick_accum(bool first) {
    return first ? accumulate_kernel<R, true> : accumulate_kernel<R, false>;
}

AccumKernel accum_kernel_for(int R, bool first) {
    switch (R) {
        case 1: return pick_accum<1>(first);   case 2: return pick_accum<2>(first);
        case 3: return pick_accum<3>(first);   case 4: return pick_accum<4>(first);
        case 5: return pick_accum<5>(first);   case 6: return pick_accum<6>(first);
        case 7: return pick_accum<7>(first);   case 8: return pick_accum<8>(first);
        case 9: return pick_accum<9>(first);   case 10: return pick_accum<10>(first);
        case 11: return pick_accum<11>(first); case 12: return pick_accum<12>(first);
        case 13: return pick_accum<13>(first); case 14: return pick_accum<14>(first);
        case 15: return pick_accum<15>(first); case 16: return pick_accum<16>(first);
        default: return nullptr;
    }
}

cudaError_t launch_accumulate(const void *const *grads, float *const *acc,
                              int R, size_t n, bool first,
                              cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    AccumParams p{};
    for (int r = 0; r < R; ++r) {
        p.g[r] = static_cast<const uint4 *>(grads[r]);
        p.acc[r] = reinterpret_cast<float4 *>(acc[r]);
    }
    p.num_vec = n / CC_PAD_ELEMS;
    p.tail_begin = p.num_vec * CC_PAD_ELEMS;
    p.tail_len = static_cast<int>(n - p.tail_begin);
    const size_t units = p.num_vec * (first ? accum_threads_per_vector<true>()
                                            : accum_threads_per_vector<false>());
    size_t blocks = div_up(units, kThreads);
    if (blocks > 0x7FFFFFFFu) blocks = 0x7FFFFFFFu;   // grid-stride covers the rest
    if (blocks == 0) blocks = 1;
    accum_kernel_for(R, first)<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_l2_flush(void *buf, size_t bytes, cudaStream_t stream) {
    const size_t nv = bytes / 16;
    if (nv == 0) return cudaSuccess;
    DeviceInfo *d = nullptr;
    cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return e;
    static std::atomic<uint32_t> counter{0};
    const uint32_t salt = 0x9E3779B9u * (counter.fetch_add(1) + 1u);
    size_t blocks = div_up(nv, kThreads);
    const size_t cap = static_cast<size_t>(d->sm_count) * 8;
    if (blocks > cap) blocks = cap;
    l2_flush_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        static_cast<uint4 *>(buf), nv, salt);
    return cudaGetLastError();
}

}  // namespace ccdp
