/*
 * Oracle for the fused data-parallel step.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg (and
 * its `--impl reference` arm) may load this library.  The product path never
 * does: it shares no source, header, constant or helper with this file.
 *
 * What it computes, element by element, single-threaded, in IEEE binary32
 * with every operation rounded separately (build with -ffp-contract=off):
 *
 *   The data-parallel result of CoCoNet ("LIT-735: Breaking the Computation
 *   and Communication Abstraction Barrier in Distributed Machine Learning
 *   Workloads", Key takeaways, the data-parallel bullet): the replicas'
 *   gradients are sum-reduced (the ReduceScatter), one Adam step with
 *   decoupled weight decay is applied to the reduced gradient (the fused
 *   optimizer), and the updated parameters are handed back to every replica
 *   (the AllGather).  Fusion and bucketing change only speed, never values,
 *   so the oracle is the plain definition of that result:
 *
 *     s   = sum over replicas r = 0..R-1, in that order, of g[r]
 *           (starting from g[0] itself, not from 0)
 *     g^  = s * (1/grad_scale)                     unscale
 *     m'  = b1*m + (1-b1)*g^                       first moment
 *     v'  = b2*v + (1-b2)*(g^*g^)                  second moment
 *     m^  = m' / (1 - b1^t),  v^ = v' / (1 - b2^t) bias correction
 *     p'  = p*(1 - lr*wd) - lr*(m^ / (sqrt(v^) + eps))
 *     out[r] = bf16_rne(p')  for every replica r
 *
 *   Adam with decoupled weight decay is the textbook optimizer (Kingma & Ba,
 *   Algorithm 1; Loshchilov & Hutter, decoupled weight decay); the pages
 *   name Adam but print no formula.
 *
 *   Gradient accumulation ("Overlapping Communication and Computation",
 *   paragraph on accumulation): k-1 micro-steps only add each replica's
 *   gradient into that replica's own fp32 accumulator; the k-th step forms
 *   each replica's local total acc[r] + g[r] and then reduces across
 *   replicas as above.
 *
 * The tensor-parallel AllReduce ("LIT-735", Key takeaways: the model-
 * parallel MatMul-then-AllReduce, overlapped in chunks): R ranks each hold a
 * partial fp32 product; every rank receives their sum, replica 0 first, in
 * that order, rounded once to bf16 (oracle_tp_allreduce).
 *
 * Parity pins (tests/test_oracle_pins.py): closed form at step 1, R=1 against
 * torch.optim.AdamW on CPU, exact integer sums, replica identity, k-step
 * accumulation against the single step on summed gradients, the bf16 cast
 * against an independent rounding over every bf16 rounding class, and
 * brute force in double on tiny inputs.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_MAX_R 16

static float bits_to_f32(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t f32_to_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* bfloat16 is the top half of a binary32.  Widening is exact. */
float oracle_bf16_widen(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/*
 * binary32 -> bfloat16, round to nearest, ties to even.
 * Adding 0x7FFF plus the kept half's lowest bit to the full pattern carries
 * into the kept half exactly when the dropped half is above one half-ulp, or
 * equal to it with an odd kept half.  A carry out of the mantissa bumps the
 * exponent, which is the correct rounding (up to infinity at the top).
 * NaN is kept a NaN: sign and top payload bits kept, quiet bit set.
 */
uint16_t oracle_bf16_round(float x) {
    uint32_t u = f32_to_bits(x);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* Bulk versions for the Python side (one call per array). */
void oracle_bf16_round_array(const float *x, uint16_t *out, size_t n) {
    for (size_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(x[i]);
}

void oracle_bf16_widen_array(const uint16_t *h, float *out, size_t n) {
    for (size_t i = 0; i < n; ++i) out[i] = oracle_bf16_widen(h[i]);
}

/*
 * Micro-steps 1..k-1 of gradient accumulation: each replica adds its own
 * gradient into its own fp32 accumulator; no value crosses replicas.
 * first != 0 starts the accumulator from this micro-step's gradient.
 */
int oracle_accumulate_local(const uint16_t *const *grads, float *const *acc,
                            size_t n, int R, int first) {
    if (R < 1 || R > ORACLE_MAX_R) return -1;
    for (int r = 0; r < R; ++r) {
        for (size_t i = 0; i < n; ++i) {
            float g = oracle_bf16_widen(grads[r][i]);
            if (first)
                acc[r][i] = g;
            else
                acc[r][i] = acc[r][i] + g;
        }
    }
    return 0;
}

/*
 * One optimizer step on the replica-summed gradient, redistributed to every
 * replica.  acc may be NULL (no accumulation); otherwise acc[r] holds
 * replica r's sum of the earlier micro-steps and is added to g[r] first.
 * master, m, v are updated in place.  Returns 0, or -1 on a bad argument.
 */
int oracle_fused_dp_step(const uint16_t *const *grads, const float *const *acc,
                         float *master, float *m, float *v,
                         uint16_t *const *params_out, size_t n, int R,
                         float lr, float beta1, float beta2, float eps,
                         float weight_decay, int step, float grad_scale) {
    if (R < 1 || R > ORACLE_MAX_R || step < 1) return -1;

    /* Scalars, each rounded to binary32 once. */
    const float one_minus_b1 = 1.0f - beta1;
    const float one_minus_b2 = 1.0f - beta2;
    const float bias_corr1 = (float)(1.0 - pow((double)beta1, (double)step));
    const float bias_corr2 = (float)(1.0 - pow((double)beta2, (double)step));
    const float lr_wd = lr * weight_decay;
    const float decay = 1.0f - lr_wd;
    const float inv_scale = 1.0f / grad_scale;

    for (size_t i = 0; i < n; ++i) {
        /* Reduce: replica 0 first, then 1, 2, ... in order. */
        float s;
        if (acc) {
            s = acc[0][i] + oracle_bf16_widen(grads[0][i]);
            for (int r = 1; r < R; ++r) {
                float local = acc[r][i] + oracle_bf16_widen(grads[r][i]);
                s = s + local;
            }
        } else {
            s = oracle_bf16_widen(grads[0][i]);
            for (int r = 1; r < R; ++r) s = s + oracle_bf16_widen(grads[r][i]);
        }

        const float g = s * inv_scale;

        const float m_decayed = beta1 * m[i];
        const float m_in = one_minus_b1 * g;
        const float m_new = m_decayed + m_in;

        const float g_sq = g * g;
        const float v_decayed = beta2 * v[i];
        const float v_in = one_minus_b2 * g_sq;
        const float v_new = v_decayed + v_in;

        const float m_hat = m_new / bias_corr1;
        const float v_hat = v_new / bias_corr2;
        const float denom = sqrtf(v_hat) + eps;
        const float ratio = m_hat / denom;
        const float update = lr * ratio;

        const float p_decayed = master[i] * decay;
        const float p_new = p_decayed - update;

        m[i] = m_new;
        v[i] = v_new;
        master[i] = p_new;

        const uint16_t b = oracle_bf16_round(p_new);
        for (int r = 0; r < R; ++r) params_out[r][i] = b;
    }
    return 0;
}

/*
 * The sum over R partial products, in rank order r = 0..R-1 starting from
 * partial[0] itself, rounded to bf16 and handed to every rank.
 */
int oracle_tp_allreduce(const float *const *partials, uint16_t *const *out,
                        size_t n, int R) {
    if (R < 1 || R > ORACLE_MAX_R) return -1;
    for (size_t i = 0; i < n; ++i) {
        float s = partials[0][i];
        for (int r = 1; r < R; ++r) s = s + partials[r][i];
        const uint16_t b = oracle_bf16_round(s);
        for (int r = 0; r < R; ++r) out[r][i] = b;
    }
    return 0;
}
