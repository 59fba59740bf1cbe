// C ABI of the fused data-parallel step (include/cc_dp.h): argument
// validation, the host-side AdamW scalars, the bucket planner and the
// per-bucket launch loop.  Every step of the arithmetic runs in the kernels
// of cc_dp_kernels.cu; this file only checks, plans and launches.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

#include "cc_dp_internal.h"
#include "cc_trace.h"

namespace ccdp {

namespace {
thread_local char g_last_error[512] = "";
}

const char *last_error() { return g_last_error; }

int fail(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

int fail_cuda(cudaError_t e, const char *what) {
    return fail(CC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
                cudaGetErrorString(e));
}

namespace {

bool finite(float x) { return std::isfinite(x); }

using MemGetAddressRangeFn = CUresult (*)(CUdeviceptr *, size_t *, CUdeviceptr);

// Driver entry points, looked up once (thread-safe static initialisation)
// through the runtime so that the library needs no link-time libcuda.
void *driver_entry_point(const char *symbol) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(symbol, &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return p;
    return nullptr;
}

MemGetAddressRangeFn address_range_fn() {
    static const MemGetAddressRangeFn fn =
        reinterpret_cast<MemGetAddressRangeFn>(driver_entry_point("cuMemGetAddressRange"));
    return fn;
}

}  // namespace

namespace {

using PointerGetAttributeFn = CUresult (*)(void *, CUpointer_attribute, CUdeviceptr);

PointerGetAttributeFn pointer_attribute_fn() {
    static const PointerGetAttributeFn fn =
        reinterpret_cast<PointerGetAttributeFn>(driver_entry_point("cuPointerGetAttribute"));
    return fn;
}

int check_within(const void *ptr, size_t bytes, uintptr_t base, size_t size,
                 const char *name, const char *kind) {
    const uintptr_t p = reinterpret_cast<uintptr_t>(ptr);
    if (p < base || p - base > size || bytes > size - (p - base))
        return fail(CC_ERR_INVALID,
                    "%s: %zu bytes at %p run past the end of its %s allocation "
                    "(%zu bytes at %p)", name, bytes, ptr, kind, size,
                    reinterpret_cast<void *>(base));
    return CC_OK;
}

// [ptr, ptr + bytes) inside one page-locked host allocation that the GPU
// reaches at the same address (CUDA pinned memory under unified addressing:
// kernels read and write it over the host link, NVLink-C2C on Grace).
int check_host_range(const void *ptr, size_t bytes, const char *name) {
    PointerGetAttributeFn fn = pointer_attribute_fn();
    if (!fn) return fail(CC_ERR_UNSUPPORTED, "cuPointerGetAttribute unavailable");
    const CUdeviceptr dp = reinterpret_cast<CUdeviceptr>(ptr);
    unsigned int type = 0;
    if (fn(&type, CU_POINTER_ATTRIBUTE_MEMORY_TYPE, dp) != CUDA_SUCCESS ||
        type != CU_MEMORYTYPE_HOST)
        return fail(CC_ERR_INVALID,
                    "%s=%p is neither device memory nor page-locked host memory", name, ptr);
    CUdeviceptr mapped = 0;
    if (fn(&mapped, CU_POINTER_ATTRIBUTE_DEVICE_POINTER, dp) != CUDA_SUCCESS || mapped != dp)
        return fail(CC_ERR_INVALID,
                    "%s=%p: page-locked host memory not mapped at the same device address",
                    name, ptr);
    CUdeviceptr start = 0;
    size_t size = 0;
    if (fn(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, dp) != CUDA_SUCCESS ||
        fn(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, dp) != CUDA_SUCCESS)
        return fail(CC_ERR_UNSUPPORTED, "%s=%p: cannot bound its host allocation", name, ptr);
    return check_within(ptr, bytes, start, size, name, "page-locked host");
}

}  // namespace

int check_device_range(const void *ptr, size_t bytes, const char *name) {
    return check_slab_range(ptr, bytes, name, false);
}

int check_slab_range(const void *ptr, size_t bytes, const char *name, bool allow_host) {
    MemGetAddressRangeFn fn = address_range_fn();
    if (!fn) return fail(CC_ERR_UNSUPPORTED, "cuMemGetAddressRange unavailable");
    CUdeviceptr base = 0;
    size_t size = 0;
    const CUresult r = fn(&base, &size, reinterpret_cast<CUdeviceptr>(ptr));
    if (r == CUDA_SUCCESS) return check_within(ptr, bytes, base, size, name, "device");
    if (allow_host) return check_host_range(ptr, bytes, name);
    return fail(CC_ERR_INVALID, "%s=%p is not in a device allocation (CUresult %d)",
                name, ptr, static_cast<int>(r));
}

int ensure_device() {
    int major = 0, minor = 0;
    const cudaError_t e = check_device(&major, &minor);
    if (e != cudaSuccess) {
        if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver)
            return fail(CC_ERR_UNSUPPORTED, "no usable CUDA device: %s",
                        cudaGetErrorString(e));
        return fail_cuda(e, "device query");
    }
    if (major != 10 || minor != 3)
        return fail(CC_ERR_UNSUPPORTED,
                    "built for sm_103a (GB300); device is sm_%d%d", major, minor);
    return CC_OK;
}

int make_scalars(float lr, float beta1, float beta2, float eps,
                 float weight_decay, int step, float grad_scale,
                 AdamScalars *c) {
    if (!finite(lr) || lr < 0.0f) return fail(CC_ERR_INVALID, "lr=%g must be finite and >= 0", lr);
    if (!finite(beta1) || beta1 < 0.0f || beta1 >= 1.0f)
        return fail(CC_ERR_INVALID, "beta1=%g must be in [0, 1)", beta1);
    if (!finite(beta2) || beta2 < 0.0f || beta2 >= 1.0f)
        return fail(CC_ERR_INVALID, "beta2=%g must be in [0, 1)", beta2);
    if (!finite(eps) || eps < 0.0f) return fail(CC_ERR_INVALID, "eps=%g must be finite and >= 0", eps);
    if (!finite(weight_decay) || weight_decay < 0.0f)
        return fail(CC_ERR_INVALID, "weight_decay=%g must be finite and >= 0", weight_decay);
    if (step < 1) return fail(CC_ERR_INVALID, "step=%d must be >= 1", step);
    if (!finite(grad_scale) || grad_scale <= 0.0f)
        return fail(CC_ERR_INVALID, "grad_scale=%g must be finite and > 0", grad_scale);

    // Each scalar is one binary32 rounding of its definition (this file is
    // built with -ffp-contract=off, so nothing here fuses).
    c->beta1 = beta1;
    c->beta2 = beta2;
    c->one_minus_b1 = 1.0f - beta1;
    c->one_minus_b2 = 1.0f - beta2;
    const double t = static_cast<double>(step);
    c->bias_corr1 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta1), t));
    c->bias_corr2 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta2), t));
    c->lr = lr;
    c->eps = eps;
    const float lr_wd = lr * weight_decay;
    c->decay = 1.0f - lr_wd;
    c->inv_scale = 1.0f / grad_scale;
    if (!(c->bias_corr1 > 0.0f) || !(c->bias_corr2 > 0.0f))
        return fail(CC_ERR_INVALID, "bias correction underflows (beta too close to 1)");
    if (!finite(c->inv_scale))
        return fail(CC_ERR_INVALID, "1/grad_scale overflows (grad_scale=%g)", grad_scale);
    c->inv_bias_corr1 = 1.0f / c->bias_corr1;
    c->inv_bias_corr2 = 1.0f / c->bias_corr2;
    return CC_OK;
}

namespace {

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
    bool written;
    const char *name;
    int index;
    bool host_ok;      // may be page-locked host memory (replica slabs)
};

bool overlap(const Range &a, const Range &b) { return a.lo < b.hi && b.lo < a.hi; }

}  // namespace

int validate_slabs(const void *const *grads, const float *const *acc,
                   float *master, float *m, float *v, void *const *params_out,
                   size_t n, int R, bool need_acc, Slabs *s) {
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    if (!grads || !params_out) return fail(CC_ERR_INVALID, "grads/params_out arrays are NULL");
    if (need_acc && !acc) return fail(CC_ERR_INVALID, "acc array is NULL");
    if (!master || !m || !v) return fail(CC_ERR_INVALID, "master/m/v is NULL");
    if (n > (SIZE_MAX / 8)) return fail(CC_ERR_INVALID, "n=%zu too large", n);
    s->R = R;
    s->master = master;
    s->m = m;
    s->v = v;
    std::vector<Range> ranges;
    ranges.reserve(3 * CC_MAX_R + 3);
    auto add = [&](const void *p, size_t bytes, bool written, const char *name,
                   int idx, bool host_ok = false) -> int {
        if (!p) return fail(CC_ERR_INVALID, "%s[%d] is NULL", name, idx);
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
            return fail(CC_ERR_MISALIGNED, "%s[%d]=%p is not 16-byte aligned", name, idx, p);
        const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        ranges.push_back({lo, lo + bytes, written, name, idx, host_ok});
        return CC_OK;
    };
    int st;
    for (int r = 0; r < R; ++r) {
        s->grads[r] = grads[r];
        s->out[r] = params_out[r];
        s->acc[r] = need_acc ? acc[r] : nullptr;
        if ((st = add(grads[r], 2 * n, false, "grads", r, true)) != CC_OK) return st;
        if ((st = add(params_out[r], 2 * n, true, "params_out", r, true)) != CC_OK) return st;
        if (need_acc && (st = add(acc[r], 4 * n, false, "acc", r)) != CC_OK) return st;
    }
    for (int r = R; r < CC_MAX_R; ++r) {
        s->grads[r] = nullptr;
        s->out[r] = nullptr;
        s->acc[r] = nullptr;
    }
    if ((st = add(master, 4 * n, true, "master", 0)) != CC_OK) return st;
    if ((st = add(m, 4 * n, true, "m", 0)) != CC_OK) return st;
    if ((st = add(v, 4 * n, true, "v", 0)) != CC_OK) return st;
    for (size_t i = 0; i < ranges.size(); ++i)
        for (size_t j = i + 1; j < ranges.size(); ++j)
            if ((ranges[i].written || ranges[j].written) && overlap(ranges[i], ranges[j]))
                return fail(CC_ERR_ALIAS, "%s[%d] overlaps %s[%d]", ranges[i].name,
                            ranges[i].index, ranges[j].name, ranges[j].index);
    if ((st = ensure_device()) != CC_OK) return st;
    for (const Range &r : ranges)
        if ((st = check_slab_range(reinterpret_cast<const void *>(r.lo), r.hi - r.lo,
                                   r.name, r.host_ok)) != CC_OK)
            return st;
    return CC_OK;
}

size_t bucket_elems(size_t bucket_bytes, size_t n) {
    if (bucket_bytes == 0) return n;
    const size_t e = bucket_bytes / 16 * CC_PAD_ELEMS;
    return e < CC_PAD_ELEMS ? CC_PAD_ELEMS : e;
}

namespace {
// One-shot injected launch failure for this thread (cc_inject_launch_failure):
// -1 disarmed, otherwise the number of bucket launches still allowed.
thread_local int g_fail_after = -1;
}  // namespace

bool injected_failure() {
    if (g_fail_after < 0) return false;
    if (g_fail_after == 0) {
        g_fail_after = -1;
        return true;
    }
    --g_fail_after;
    return false;
}

int run_step(const Slabs &s, const AdamScalars &c, size_t n, size_t bucket_bytes,
             cudaStream_t stream) {
    const size_t per = bucket_elems(bucket_bytes, n);
    for (size_t b = 0; b < n; b += per) {
        const size_t e = std::min(n, b + per);
        if (injected_failure())
            return fail(CC_ERR_CUDA, "injected launch failure before the bucket at element %zu", b);
        TraceRange bucket("bucket", b);
        const cudaError_t err = launch_fused(s, c, b, e, 0, /*chain=*/b > 0, stream,
                                             /*wait_first=*/b == 0);
        if (err != cudaSuccess) return fail_cuda(err, "fused step launch");
    }
    return CC_OK;
}

}  // namespace ccdp

using namespace ccdp;

extern "C" {

const char *cc_status_string(int status) {
    switch (status) {
        case CC_OK: return "CC_OK";
        case CC_ERR_INVALID: return "CC_ERR_INVALID";
        case CC_ERR_ALIAS: return "CC_ERR_ALIAS";
        case CC_ERR_MISALIGNED: return "CC_ERR_MISALIGNED";
        case CC_ERR_CUDA: return "CC_ERR_CUDA";
        case CC_ERR_UNSUPPORTED: return "CC_ERR_UNSUPPORTED";
        case CC_ERR_CAPACITY: return "CC_ERR_CAPACITY";
        default: return "CC_ERR_UNKNOWN";
    }
}

const char *cc_last_error(void) { return last_error(); }

int cc_fused_dp_step_accum(const void *const *grads, const float *const *acc,
                           float *master, float *m, float *v,
                           void *const *params_out, size_t n, int R,
                           size_t bucket_bytes, float lr, float beta1,
                           float beta2, float eps, float weight_decay,
                           int step, float grad_scale, int accum_k,
                           void *stream) {
    TraceRange call(acc ? "cc_fused_dp_step_accum" : "cc_fused_dp_step", n);
    if (accum_k < 1) return fail(CC_ERR_INVALID, "accum_k=%d must be >= 1", accum_k);
    if (accum_k > 1 && !acc)
        return fail(CC_ERR_INVALID, "accum_k=%d needs the accumulators (acc is NULL)", accum_k);
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    AdamScalars c;
    int st = make_scalars(lr, beta1, beta2, eps, weight_decay, step, grad_scale, &c);
    if (st != CC_OK) return st;
    if (n == 0) return CC_OK;
    Slabs s;
    st = validate_slabs(grads, acc, master, m, v, params_out, n, R, acc != nullptr, &s);
    if (st != CC_OK) return st;
    return run_step(s, c, n, bucket_bytes, static_cast<cudaStream_t>(stream));
}

int cc_fused_dp_step(const void *const *grads, float *master, float *m,
                     float *v, void *const *params_out, size_t n, int R,
                     size_t bucket_bytes, float lr, float beta1, float beta2,
                     float eps, float weight_decay, int step, float grad_scale,
                     int accum_k, void *stream) {
    if (accum_k != 1)
        return fail(CC_ERR_INVALID,
                    "accum_k=%d: accumulated steps need cc_fused_dp_step_accum", accum_k);
    return cc_fused_dp_step_accum(grads, nullptr, master, m, v, params_out, n, R,
                                  bucket_bytes, lr, beta1, beta2, eps,
                                  weight_decay, step, grad_scale, 1, stream);
}

int cc_fused_dp_bucket(const void *const *grads, const float *const *acc,
                       float *master, float *m, float *v,
                       void *const *params_out, size_t n, int R, size_t begin,
                       size_t end, float lr, float beta1, float beta2,
                       float eps, float weight_decay, int step,
                       float grad_scale, int max_ctas, void *stream) {
    return cc_fused_dp_bucket_ex(grads, acc, master, m, v, params_out, n, R, begin, end, lr,
                                 beta1, beta2, eps, weight_decay, step, grad_scale, max_ctas,
                                 0u, stream);
}

int cc_fused_dp_bucket_ex(const void *const *grads, const float *const *acc,
                          float *master, float *m, float *v,
                          void *const *params_out, size_t n, int R, size_t begin,
                          size_t end, float lr, float beta1, float beta2,
                          float eps, float weight_decay, int step,
                          float grad_scale, int max_ctas, unsigned arith_flags,
                          void *stream) {
    TraceRange call("cc_fused_dp_bucket", begin);
    if (arith_flags & ~(CC_ARITH_FAST | CC_ENGINE_BULK_COPY))
        return fail(CC_ERR_INVALID, "arith_flags=%#x has unknown bits", arith_flags);
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    if (begin > end || end > n)
        return fail(CC_ERR_INVALID, "range [%zu, %zu) not inside [0, %zu)", begin, end, n);
    if (begin % CC_PAD_ELEMS != 0)
        return fail(CC_ERR_MISALIGNED, "begin=%zu is not a multiple of %d", begin, CC_PAD_ELEMS);
    if (max_ctas < 0) return fail(CC_ERR_INVALID, "max_ctas=%d must be >= 0", max_ctas);
    AdamScalars c;
    int st = make_scalars(lr, beta1, beta2, eps, weight_decay, step, grad_scale, &c);
    if (st != CC_OK) return st;
    if (begin == end) return CC_OK;
    Slabs s;
    st = validate_slabs(grads, acc, master, m, v, params_out, n, R, acc != nullptr, &s);
    if (st != CC_OK) return st;
    s.fast = (arith_flags & CC_ARITH_FAST) != 0;
    s.bulk_copy = (arith_flags & CC_ENGINE_BULK_COPY) != 0;
    const cudaError_t e =
        launch_step_range(s, c, begin, end, max_ctas, false, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CC_OK : fail_cuda(e, "fused bucket launch");
}

int cc_fused_dp_shard(const void *const *grads, const float *const *acc,
                      float *master, float *m, float *v,
                      void *const *params_out, size_t n, int R,
                      size_t shard_begin, size_t shard_end, size_t bucket_bytes,
                      float lr, float beta1, float beta2, float eps,
                      float weight_decay, int step, float grad_scale,
                      void *stream) {
    TraceRange call("cc_fused_dp_shard", shard_begin);
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    if (shard_begin > shard_end || shard_end > n)
        return fail(CC_ERR_INVALID, "shard [%zu, %zu) not inside [0, %zu)", shard_begin,
                    shard_end, n);
    if (shard_begin % CC_PAD_ELEMS != 0)
        return fail(CC_ERR_MISALIGNED, "shard_begin=%zu is not a multiple of %d", shard_begin,
                    CC_PAD_ELEMS);
    if (shard_begin == shard_end) {
        AdamScalars c;
        return make_scalars(lr, beta1, beta2, eps, weight_decay, step, grad_scale, &c);
    }
    if (!grads || !params_out) return fail(CC_ERR_INVALID, "grads/params_out arrays are NULL");
    // The shard's view of the replica slabs: the same step over
    // len = shard_end - shard_begin elements, with the state arrays as they
    // are.  shard_begin is a multiple of 8, so the views keep the 16-byte
    // alignment of the slabs.
    const void *g[CC_MAX_R];
    void *o[CC_MAX_R];
    const float *a[CC_MAX_R];
    for (int r = 0; r < R; ++r) {
        if (!grads[r] || !params_out[r] || (acc && !acc[r]))
            return fail(CC_ERR_INVALID, "replica %d slab is NULL", r);
        g[r] = static_cast<const char *>(grads[r]) + 2 * shard_begin;
        o[r] = static_cast<char *>(params_out[r]) + 2 * shard_begin;
        a[r] = acc ? acc[r] + shard_begin : nullptr;
    }
    return cc_fused_dp_step_accum(g, acc ? a : nullptr, master, m, v, o,
                                  shard_end - shard_begin, R, bucket_bytes, lr, beta1,
                                  beta2, eps, weight_decay, step, grad_scale, 1, stream);
}

int cc_shard_plan(const size_t *bucket_begin, const size_t *bucket_end, int num_buckets,
                  int world, size_t *shard_begin_out, size_t *shard_end_out,
                  size_t *state_offset_out, size_t *state_elems_out) {
    if (num_buckets < 0 || world < 1)
        return fail(CC_ERR_INVALID, "num_buckets=%d, world=%d", num_buckets, world);
    if (!state_elems_out || (num_buckets > 0 && (!bucket_begin || !bucket_end ||
                                                 !shard_begin_out || !shard_end_out ||
                                                 !state_offset_out)))
        return fail(CC_ERR_INVALID, "NULL array");
    for (int b = 0; b < num_buckets; ++b) {
        if (bucket_end[b] < bucket_begin[b] || (b > 0 && bucket_begin[b] < bucket_end[b - 1]))
            return fail(CC_ERR_INVALID, "bucket %d range is reversed or out of order", b);
        if (bucket_begin[b] % CC_PAD_ELEMS != 0)
            return fail(CC_ERR_MISALIGNED, "bucket %d begins at %zu, not a multiple of %d", b,
                        bucket_begin[b], CC_PAD_ELEMS);
    }
    for (int q = 0; q < world; ++q) state_elems_out[q] = 0;
    for (int b = 0; b < num_buckets; ++b) {
        // Cut the bucket in 8-element units: shard q holds units
        // [floor(u q / W), floor(u (q+1) / W)); the last shard also takes a
        // ragged tail.  Sizes differ by at most 8 elements (plus the tail).
        const size_t lo = bucket_begin[b], hi = bucket_end[b];
        const size_t units = (hi - lo) / CC_PAD_ELEMS;
        for (int q = 0; q < world; ++q) {
            const size_t i = static_cast<size_t>(b) * world + q;
            const size_t a = lo + CC_PAD_ELEMS * (units * q / world);
            const size_t e = q + 1 < world ? lo + CC_PAD_ELEMS * (units * (q + 1) / world) : hi;
            shard_begin_out[i] = a;
            shard_end_out[i] = e;
            state_offset_out[i] = state_elems_out[q];
            state_elems_out[q] += e - a;
        }
    }
    return CC_OK;
}

int cc_fused_dp_rank_step(const void *const *grad_slices, float *master, float *m, float *v,
                          void *param_out, size_t len, int R, float lr, float beta1,
                          float beta2, float eps, float weight_decay, int step,
                          float grad_scale, void *stream) {
    TraceRange call("cc_fused_dp_rank_step", len);
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    AdamScalars c;
    int st = make_scalars(lr, beta1, beta2, eps, weight_decay, step, grad_scale, &c);
    if (st != CC_OK) return st;
    if (len == 0) return CC_OK;
    if (!grad_slices) return fail(CC_ERR_INVALID, "grad_slices array is NULL");
    if (!param_out) return fail(CC_ERR_INVALID, "param_out is NULL");
    if (!master || !m || !v) return fail(CC_ERR_INVALID, "master/m/v is NULL");
    if (len > (SIZE_MAX / 8)) return fail(CC_ERR_INVALID, "len=%zu too large", len);
    std::vector<Range> ranges;
    auto add = [&](const void *p, size_t bytes, bool written, const char *name, int idx,
                   bool host_ok) -> int {
        if (!p) return fail(CC_ERR_INVALID, "%s[%d] is NULL", name, idx);
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
            return fail(CC_ERR_MISALIGNED, "%s[%d]=%p is not 16-byte aligned", name, idx, p);
        const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        ranges.push_back({lo, lo + bytes, written, name, idx, host_ok});
        return CC_OK;
    };
    for (int r = 0; r < R; ++r)
        if ((st = add(grad_slices[r], 2 * len, false, "grad_slices", r, true)) != CC_OK) return st;
    if ((st = add(param_out, 2 * len, true, "param_out", 0, true)) != CC_OK) return st;
    if ((st = add(master, 4 * len, true, "master", 0, false)) != CC_OK) return st;
    if ((st = add(m, 4 * len, true, "m", 0, false)) != CC_OK) return st;
    if ((st = add(v, 4 * len, true, "v", 0, false)) != CC_OK) return st;
    for (size_t i = 0; i < ranges.size(); ++i)
        for (size_t j = i + 1; j < ranges.size(); ++j)
            if ((ranges[i].written || ranges[j].written) && overlap(ranges[i], ranges[j]))
                return fail(CC_ERR_ALIAS, "%s[%d] overlaps %s[%d]", ranges[i].name,
                            ranges[i].index, ranges[j].name, ranges[j].index);
    if ((st = ensure_device()) != CC_OK) return st;
    for (const Range &r : ranges)
        if ((st = check_slab_range(reinterpret_cast<const void *>(r.lo), r.hi - r.lo, r.name,
                                   r.host_ok)) != CC_OK)
            return st;
    Slabs s;
    s.R = R;
    for (int r = 0; r < CC_MAX_R; ++r) {
        s.grads[r] = r < R ? grad_slices[r] : nullptr;
        s.acc[r] = nullptr;
        s.out[r] = r == 0 ? param_out : nullptr;
    }
    s.master = master;
    s.m = m;
    s.v = v;
    s.one_out = true;
    // A programmatic dependent of whatever precedes it (a previous rank step,
    // the exchange that filled the slices): resident early, reading nothing
    // before that grid has completed.
    const cudaError_t e = launch_fused(s, c, 0, len, 0, false, static_cast<cudaStream_t>(stream),
                                       /*wait_first=*/true);
    return e == cudaSuccess ? CC_OK : fail_cuda(e, "rank step launch");
}

int cc_accumulate_local(const void *const *grads, float *const *acc, size_t n,
                        int R, int first, void *stream) {
    TraceRange call(first ? "cc_accumulate_local(first)" : "cc_accumulate_local", n);
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    if (n == 0) return CC_OK;
    if (!grads || !acc) return fail(CC_ERR_INVALID, "grads/acc arrays are NULL");
    if (n > (SIZE_MAX / 8)) return fail(CC_ERR_INVALID, "n=%zu too large", n);
    std::vector<Range> ranges;
    for (int r = 0; r < R; ++r) {
        const void *ps[2] = {grads[r], acc[r]};
        const size_t bytes[2] = {2 * n, 4 * n};
        const char *names[2] = {"grads", "acc"};
        for (int k = 0; k < 2; ++k) {
            if (!ps[k]) return fail(CC_ERR_INVALID, "%s[%d] is NULL", names[k], r);
            if (reinterpret_cast<uintptr_t>(ps[k]) % 16 != 0)
                return fail(CC_ERR_MISALIGNED, "%s[%d]=%p is not 16-byte aligned",
                            names[k], r, ps[k]);
            const uintptr_t lo = reinterpret_cast<uintptr_t>(ps[k]);
            ranges.push_back({lo, lo + bytes[k], k == 1, names[k], r, false});
        }
    }
    for (size_t i = 0; i < ranges.size(); ++i)
        for (size_t j = i + 1; j < ranges.size(); ++j)
            if ((ranges[i].written || ranges[j].written) && overlap(ranges[i], ranges[j]))
                return fail(CC_ERR_ALIAS, "%s[%d] overlaps %s[%d]", ranges[i].name,
                            ranges[i].index, ranges[j].name, ranges[j].index);
    int st = ensure_device();
    if (st != CC_OK) return st;
    for (const Range &r : ranges)
        if ((st = check_device_range(reinterpret_cast<const void *>(r.lo), r.hi - r.lo,
                                     r.name)) != CC_OK)
            return st;
    const cudaError_t e =
        launch_accumulate(grads, acc, R, n, first != 0, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CC_OK : fail_cuda(e, "accumulate launch");
}

int cc_plan_buckets(const size_t *numel, int num_tensors, size_t bucket_bytes,
                    size_t *offsets_out, size_t *bucket_begin_out,
                    size_t *bucket_end_out, int capacity,
                    int *num_buckets_out, size_t *n_padded_out) {
    if (num_tensors < 1 || !numel || !offsets_out || !num_buckets_out)
        return fail(CC_ERR_INVALID, "need num_tensors >= 1, numel, offsets_out, num_buckets_out");
    if (capacity < 0 || (capacity > 0 && (!bucket_begin_out || !bucket_end_out)))
        return fail(CC_ERR_INVALID, "capacity=%d with NULL bucket arrays", capacity);
    // Slab position of the next tensor, start of the open bucket, and the
    // open bucket's bf16 bytes.  Walk from the last tensor to the first.
    size_t pos = 0, open_begin = 0, open_bytes = 0;
    int count = 0;
    auto emit = [&](size_t b, size_t e) {
        if (count < capacity) {
            bucket_begin_out[count] = b;
            bucket_end_out[count] = e;
        }
        ++count;
    };
    for (int t = num_tensors - 1; t >= 0; --t) {
        const size_t k = numel[t];
        if (k > SIZE_MAX / 4 - pos)
            return fail(CC_ERR_INVALID, "slab size overflows at tensor %d", t);
        const size_t span = (k + CC_PAD_ELEMS - 1) / CC_PAD_ELEMS * CC_PAD_ELEMS;
        offsets_out[t] = pos;
        pos += span;
        open_bytes += 2 * span;
        if (bucket_bytes != 0 && open_bytes >= bucket_bytes) {
            if (pos > open_begin) emit(open_begin, pos);
            open_begin = pos;
            open_bytes = 0;
        }
    }
    if (pos > open_begin) emit(open_begin, pos);
    *num_buckets_out = count;
    if (n_padded_out) *n_padded_out = pos;
    if (count > capacity)
        return fail(CC_ERR_CAPACITY, "%d buckets, capacity %d", count, capacity);
    return CC_OK;
}

int cc_bucket_ready_layers(const size_t *numel, const int *layer_of,
                           const size_t *offsets, int num_tensors,
                           const size_t *bucket_begin,
                           const size_t *bucket_end, int num_buckets,
                           int *ready_layer_out) {
    if (num_tensors < 1 || num_buckets < 1 || !numel || !layer_of || !offsets ||
        !bucket_begin || !bucket_end || !ready_layer_out)
        return fail(CC_ERR_INVALID, "NULL array or empty list");
    for (int b = 0; b < num_buckets; ++b) {
        if (bucket_end[b] <= bucket_begin[b] || (b > 0 && bucket_begin[b] < bucket_end[b - 1]))
            return fail(CC_ERR_INVALID, "bucket %d range is empty or out of order", b);
        ready_layer_out[b] = -1;
    }
    // Each non-empty tensor finds its bucket by binary search on the bucket
    // starts; the bucket keeps the lowest layer it has seen.
    for (int t = 0; t < num_tensors; ++t) {
        if (numel[t] == 0) continue;
        const size_t *it = std::upper_bound(bucket_begin, bucket_begin + num_buckets, offsets[t]);
        const int b = static_cast<int>(it - bucket_begin) - 1;
        if (b < 0 || offsets[t] >= bucket_end[b])
            return fail(CC_ERR_INVALID, "tensor %d at %zu lies in no bucket", t, offsets[t]);
        if (ready_layer_out[b] < 0 || layer_of[t] < ready_layer_out[b])
            ready_layer_out[b] = layer_of[t];
    }
    for (int b = 0; b < num_buckets; ++b)
        if (ready_layer_out[b] < 0) return fail(CC_ERR_INVALID, "bucket %d holds no tensor", b);
    return CC_OK;
}

int cc_unfused_dp_step(const void *const *grads, float *master, float *m, float *v,
                       void *const *params_out, float *workspace, size_t workspace_bytes,
                       size_t n, int R, size_t bucket_bytes, float lr, float beta1,
                       float beta2, float eps, float weight_decay, int step,
                       float grad_scale, void *stream) {
    TraceRange call("cc_unfused_dp_step", n);
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    AdamScalars c;
    int st = make_scalars(lr, beta1, beta2, eps, weight_decay, step, grad_scale, &c);
    if (st != CC_OK) return st;
    if (n == 0) return CC_OK;
    const size_t per = bucket_elems(bucket_bytes, n);
    const size_t need = 4 * (per < n ? per : n);
    if (!workspace) return fail(CC_ERR_INVALID, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return fail(CC_ERR_MISALIGNED, "workspace=%p is not 16-byte aligned", workspace);
    if (workspace_bytes < need)
        return fail(CC_ERR_INVALID, "workspace of %zu bytes, the largest bucket needs %zu",
                    workspace_bytes, need);
    // The workspace is written: it may overlap no slab.
    const uintptr_t wlo = reinterpret_cast<uintptr_t>(workspace), whi = wlo + need;
    auto hits = [&](const void *p, size_t bytes) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        return p && lo < whi && wlo < lo + bytes;
    };
    if (!grads || !params_out) return fail(CC_ERR_INVALID, "grads/params_out arrays are NULL");
    for (int r = 0; r < R; ++r)
        if (hits(grads[r], 2 * n) || hits(params_out[r], 2 * n))
            return fail(CC_ERR_ALIAS, "workspace overlaps replica %d's slabs", r);
    if (hits(master, 4 * n) || hits(m, 4 * n) || hits(v, 4 * n))
        return fail(CC_ERR_ALIAS, "workspace overlaps master/m/v");
    Slabs s;
    st = validate_slabs(grads, nullptr, master, m, v, params_out, n, R, false, &s);
    if (st != CC_OK) return st;
    if ((st = check_device_range(workspace, need, "workspace")) != CC_OK) return st;
    for (size_t b = 0; b < n; b += per) {
        const size_t e = std::min(n, b + per);
        if (injected_failure())
            return fail(CC_ERR_CUDA, "injected launch failure before the bucket at element %zu", b);
        TraceRange bucket("bucket", b);
        const cudaError_t err = launch_unfused_bucket(s, c, workspace, b, e,
                                                      static_cast<cudaStream_t>(stream));
        if (err != cudaSuccess) return fail_cuda(err, "unfused step launch");
    }
    return CC_OK;
}

int cc_inject_launch_failure(int after_launches) {
    if (after_launches < -1) return fail(CC_ERR_INVALID, "after_launches=%d must be >= -1",
                                         after_launches);
    g_fail_after = after_launches;
    return CC_OK;
}

int cc_inject_bulk_stall(long long tile, unsigned timeout_us) {
    if (tile < -1) return fail(CC_ERR_INVALID, "tile=%lld must be >= -1", tile);
    if (tile >= 0 && (timeout_us < 1 || timeout_us > 1000000))
        return fail(CC_ERR_INVALID, "timeout_us=%u must be in 1..1000000", timeout_us);
    arm_bulk_stall(tile, 1000ull * timeout_us);
    return CC_OK;
}

int cc_device_status(unsigned *status, int clear) {
    if (!status) return fail(CC_ERR_INVALID, "status is NULL");
    int st = ensure_device();
    if (st != CC_OK) return st;
    unsigned bulk = 0, tp = 0;
    cudaError_t e = read_bulk_status(&bulk, clear != 0);
    if (e == cudaSuccess) e = read_tp_status(&tp, clear != 0);
    if (e != cudaSuccess) return fail_cuda(e, "status read");
    *status = bulk | tp;
    return CC_OK;
}

int cc_l2_flush(void *buf, size_t bytes, void *stream) {
    if (!buf) return fail(CC_ERR_INVALID, "buf is NULL");
    if (reinterpret_cast<uintptr_t>(buf) % 16 != 0)
        return fail(CC_ERR_MISALIGNED, "buf=%p is not 16-byte aligned", buf);
    int st = ensure_device();
    if (st != CC_OK) return st;
    if ((st = check_device_range(buf, bytes, "buf")) != CC_OK) return st;
    const cudaError_t e = launch_l2_flush(buf, bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CC_OK : fail_cuda(e, "l2 flush launch");
}

}  // extern "C"
