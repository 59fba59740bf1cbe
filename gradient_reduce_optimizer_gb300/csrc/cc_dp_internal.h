// Internal interface between the C-ABI layer and the kernels of the fused
// data-parallel step.  Not installed; the public ABI is include/cc_dp.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "cc_dp.h"

namespace ccdp {

// AdamW scalars, each rounded to binary32 once on the host (see
// make_scalars in cc_dp_api.cu for how each is formed).
struct AdamScalars {
    float beta1, beta2;
    float one_minus_b1, one_minus_b2;
    float bias_corr1, bias_corr2;
    float lr, eps;
    float decay;      // 1 - lr*wd  (decoupled weight decay factor)
    float inv_scale;  // 1 / grad_scale
    float inv_bias_corr1, inv_bias_corr2;   // 1 / bias_corrX (fast arithmetic only)
};

// The slabs of one step.  Pointers are whole-slab bases; kernels index them
// by element.  acc[r] are all null when the step does not accumulate.
struct Slabs {
    int R;
    const void *grads[CC_MAX_R];   // bf16[n]
    const float *acc[CC_MAX_R];    // fp32[n] or null
    void *out[CC_MAX_R];           // bf16[n]
    float *master, *m, *v;         // fp32[n]
    bool one_out = false;          // parameters to out[0] only (the multi-GPU
                                   // rank step; plain kernel, no accumulators)
    bool fast = false;             // the opt-in fast arithmetic (CC_ARITH_FAST)
    bool bulk_copy = false;        // CTA budgets on the TMA bulk-copy engine
                                   // (CC_ENGINE_BULK_COPY), not the wide kernel
};

// Enqueue the fused reduce + AdamW + redistribute kernel over elements
// [begin, end) on `stream`.  Requires begin % CC_PAD_ELEMS == 0 and 16-byte
// aligned slab bases (checked by the caller).  max_ctas > 0 launches the
// CTA-budget form: at most max_ctas wide CTAs (one per SM), each thread
// striding over the range.
// chain = true launches it as a programmatic dependent of the kernel just
// before it on `stream`, which must be a fused-step launch on a disjoint
// element range (the next bucket of the same step).  wait_first = true
// launches it as a programmatic dependent of whatever kernel precedes it,
// on whose results it may depend: its CTAs may become resident while that
// kernel finishes, but touch no memory before it has completed (the first
// bucket of a step, after the previous step's last bucket).
cudaError_t launch_fused(const Slabs &s, const AdamScalars &c, size_t begin,
                         size_t end, int max_ctas, bool chain,
                         cudaStream_t stream, bool wait_first = false);

// Enqueue the bulk-copy engine of the same step over [begin, end) on at most
// num_ctas SMs (one persistent CTA per SM; 0 = every SM).  Same arithmetic
// and requirements as launch_fused.
cudaError_t launch_fused_bulk(const Slabs &s, const AdamScalars &c, size_t begin,
                              size_t end, int num_ctas, cudaStream_t stream);

// The fused step over [begin, end) with the engine a CTA budget calls for:
// max_ctas > 0 runs the wide-CTA form of the fused kernel on that many SMs
// (or, with s.bulk_copy, the TMA bulk-copy engine), 0 the plain kernel over
// the whole GPU.  Either kernel form chains to the previous bucket if
// `chain`.
inline cudaError_t launch_step_range(const Slabs &s, const AdamScalars &c, size_t begin,
                                     size_t end, int max_ctas, bool chain,
                                     cudaStream_t stream) {
    return (max_ctas > 0 && s.bulk_copy)
               ? launch_fused_bulk(s, c, begin, end, max_ctas, stream)
               : launch_fused(s, c, begin, end, max_ctas, chain, stream);
}

// Enqueue the unfused schedule of one bucket: reduce into `workspace`
// (fp32, at least end - begin elements), AdamW from it, then R-1 copies of
// replica 0's parameters.  Same values as launch_fused.
cudaError_t launch_unfused_bucket(const Slabs &s, const AdamScalars &c, float *workspace,
                                  size_t begin, size_t end, cudaStream_t stream);

// Elements per bucket for a bf16 byte size (0 = the whole slab).
size_t bucket_elems(size_t bucket_bytes, size_t n);

// Arm a one-shot failure of the next bulk-engine launch on this thread: its
// producer never issues tile `tile` (counted from the launch's first tile),
// and its pipeline waits give up after timeout_ns.  tile < 0 disarms.
void arm_bulk_stall(long long tile, unsigned long long timeout_ns);

// Read (and optionally clear) the bulk engine's status word: 0, or codes of
// waits that ran out (1 consumer, 2 producer, 4 drain).  Synchronous.
cudaError_t read_bulk_status(unsigned *status, bool clear);

// The fused tensor-parallel MatMul + AllReduce (cc_tp_fused.cu) on shapes
// already validated; max_ctas > 0 caps the persistent grid; ws (ws_bytes,
// at least tp_fused_workspace's figure) lets the last wave be split, NULL
// keeps it whole.  Returns a cc_status (the reason recorded with fail()).
int launch_tp_fused(const void *const *x, const void *const *w, void *const *out,
                    float *const *partials, int m, int n, int k, int R, int max_ctas,
                    void *ws, size_t ws_bytes, cudaStream_t stream);
// Workspace bytes launch_tp_fused uses on the current device for this shape
// and CTA cap (0: it splits nothing).
int tp_fused_workspace(int m, int n, int R, int max_ctas, size_t *bytes);
// Whether the fused kernel tiles m x n with k/R per rank: m % 128 == 0,
// (k/R) % 64 == 0, and n a multiple of 128 or 192.
bool tp_fused_shape_ok(int m, int n, int kr);

// Read (and optionally clear) the fused tensor-parallel kernel's status word:
// 0, or codes of waits that ran out (8 producer, 16 MMA, 32 epilogue, 64
// drain).  Synchronous.
cudaError_t read_tp_status(unsigned *status, bool clear);

// Multiprocessor count of the current device (queried once per device).
cudaError_t device_sm_count(int *count);

// Enqueue one local accumulation micro-step over [0, n).
cudaError_t launch_accumulate(const void *const *grads, float *const *acc,
                              int R, size_t n, bool first,
                              cudaStream_t stream);

// Enqueue a write of `bytes` (rounded down to 16) into `buf`.
cudaError_t launch_l2_flush(void *buf, size_t bytes, cudaStream_t stream);

// Compute capability of the current device (queried once per device).
cudaError_t check_device(int *major, int *minor);

// ---- host-side helpers of the C-ABI layer (cc_dp_api.cu) -----------------

// Record a one-line reason for cc_last_error() and return `status`.
int fail(int status, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail_cuda(cudaError_t e, const char *what);
const char *last_error();

// CC_OK if the current device is an sm_103 GB300, else CC_ERR_UNSUPPORTED.
int ensure_device();

// CC_OK if [ptr, ptr + bytes) lies inside one device allocation.
int check_device_range(const void *ptr, size_t bytes, const char *name);

// As check_device_range; with allow_host, a range inside one page-locked
// host allocation mapped at the same device address is accepted too.
int check_slab_range(const void *ptr, size_t bytes, const char *name, bool allow_host);

// The one-shot launch failure armed by cc_inject_launch_failure: true (and
// disarmed) when the bucket launch about to be made must fail instead.
bool injected_failure();

// Validate and round the AdamW hyper-parameters to the kernel's scalars.
int make_scalars(float lr, float beta1, float beta2, float eps,
                 float weight_decay, int step, float grad_scale,
                 AdamScalars *c);

// Validate a slab set (R, pointers, alignment, aliasing, device ranges of n
// elements; gradient and parameter replica slabs may be page-locked host
// memory) and fill `s`.  need_acc selects whether acc[] is used.
int validate_slabs(const void *const *grads, const float *const *acc,
                   float *master, float *m, float *v, void *const *params_out,
                   size_t n, int R, bool need_acc, Slabs *s);

}  // namespace ccdp
