// Per-element device arithmetic of the fused data-parallel step, shared by
// both kernel engines (cc_dp_kernels.cu, cc_dp_bulk.cu) so that they compute
// bit-identical results.  Every operation is one IEEE binary32 rounding in
// the order given in include/cc_dp.h.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "cc_dp_internal.h"

#ifndef CC_DP_MIXED_ADD
#define CC_DP_MIXED_ADD 1   // fold the bf16 widening into the add (sm_100+)
#endif

namespace ccdp {
namespace dev {

__device__ __forceinline__ float bf16_lo(uint32_t w) {
    return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t w) {
    return __uint_as_float(w & 0xFFFF0000u);
}
__device__ __forceinline__ float bf16_at(const void *base, size_t i) {
    const unsigned short h = static_cast<const unsigned short *>(base)[i];
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ void widen8(const uint4 q, float t[8]) {
    t[0] = bf16_lo(q.x); t[1] = bf16_hi(q.x);
    t[2] = bf16_lo(q.y); t[3] = bf16_hi(q.y);
    t[4] = bf16_lo(q.z); t[5] = bf16_hi(q.z);
    t[6] = bf16_lo(q.w); t[7] = bf16_hi(q.w);
}

// s + (the bf16 in the low / high half of w), one IEEE binary32 rounding.
// Widening bf16 to binary32 is exact, so this equals __fadd_rn(s, widened);
// the mixed-precision add takes the bf16 operand directly.
__device__ __forceinline__ float add_bf16_lo(float s, uint32_t w) {
#if CC_DP_MIXED_ADD
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "add.rn.f32.bf16 %0, lo, %2;\n\t}" : "=f"(r) : "r"(w), "f"(s));
    return r;
#else
    return __fadd_rn(s, bf16_lo(w));
#endif
}
__device__ __forceinline__ float add_bf16_hi(float s, uint32_t w) {
#if CC_DP_MIXED_ADD
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "add.rn.f32.bf16 %0, hi, %2;\n\t}" : "=f"(r) : "r"(w), "f"(s));
    return r;
#else
    return __fadd_rn(s, bf16_hi(w));
#endif
}

// s[0..7] += the 8 bf16 of q, each add one rounding.
__device__ __forceinline__ void add8_bf16(float s[8], const uint4 q) {
    s[0] = add_bf16_lo(s[0], q.x); s[1] = add_bf16_hi(s[1], q.x);
    s[2] = add_bf16_lo(s[2], q.y); s[3] = add_bf16_hi(s[3], q.y);
    s[4] = add_bf16_lo(s[4], q.z); s[5] = add_bf16_hi(s[5], q.z);
    s[6] = add_bf16_lo(s[6], q.w); s[7] = add_bf16_hi(s[7], q.w);
}

// Two fp32 -> bf16x2, round to nearest even; a lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// One AdamW step on one element, given the reduced gradient s.
__device__ __forceinline__ void adamw(float s, float &p, float &m, float &v,
                                      const AdamScalars &c) {
    const float g = __fmul_rn(s, c.inv_scale);
    const float m_new = __fadd_rn(__fmul_rn(c.beta1, m), __fmul_rn(c.one_minus_b1, g));
    const float v_new = __fadd_rn(__fmul_rn(c.beta2, v),
                                  __fmul_rn(c.one_minus_b2, __fmul_rn(g, g)));
    const float m_hat = __fdiv_rn(m_new, c.bias_corr1);
    const float v_hat = __fdiv_rn(v_new, c.bias_corr2);
    const float denom = __fadd_rn(__fsqrt_rn(v_hat), c.eps);
    const float update = __fmul_rn(c.lr, __fdiv_rn(m_hat, denom));
    p = __fsub_rn(__fmul_rn(p, c.decay), update);
    m = m_new;
    v = v_new;
}

// The opt-in fast form of the same step (CC_ARITH_FAST): m and v exactly as
// above; the two bias-correction divisions become multiplications by
// reciprocals rounded once on the host, the square root stays IEEE, and the
// quotient m^/(sqrt(v^) + eps) is CUDA's fast division __fdividef (2 ulp
// for normal denominators; eps > 0 keeps the denominator normal).  The
// parameter then differs from the correctly rounded step by a few ulp of the
// update, the bf16 copy by at most one bf16 ulp.
__device__ __forceinline__ void adamw_fast(float s, float &p, float &m, float &v,
                                           const AdamScalars &c) {
    const float g = __fmul_rn(s, c.inv_scale);
    const float m_new = __fadd_rn(__fmul_rn(c.beta1, m), __fmul_rn(c.one_minus_b1, g));
    const float v_new = __fadd_rn(__fmul_rn(c.beta2, v),
                                  __fmul_rn(c.one_minus_b2, __fmul_rn(g, g)));
    const float m_hat = __fmul_rn(m_new, c.inv_bias_corr1);
    const float v_hat = __fmul_rn(v_new, c.inv_bias_corr2);
    const float denom = __fadd_rn(__fsqrt_rn(v_hat), c.eps);
    const float update = __fmul_rn(c.lr, __fdividef(m_hat, denom));
    p = __fsub_rn(__fmul_rn(p, c.decay), update);
    m = m_new;
    v = v_new;
}

// The step in the arithmetic the kernel was instantiated for.
template <bool FAST>
__device__ __forceinline__ void adamw_step(float s, float &p, float &m, float &v,
                                           const AdamScalars &c) {
    if constexpr (FAST)
        adamw_fast(s, p, m, v, c);
    else
        adamw(s, p, m, v, c);
}

}  // namespace dev
}  // namespace ccdp
