// The unfused schedule of the same data-parallel step, for comparison with
// the fused kernel: what a data-parallel framework does when the collective
// and the optimizer are separate library calls ("LIT-735 (CoCoNet)", Key
// takeaways: the data-parallel result is that fusing the optimizer into the
// ReduceScatter/AllGather beats PyTorch DDP, whose bucketed AllReduce and
// optimizer step are separate kernels; "Communication Optimization ›
// Communication Overlap": the optimizer step reads the aggregated gradient
// only after the all-reduce has finished).
//
// Per bucket, three stream-ordered phases:
//   1. reduce_kernel   sums the R bf16 gradient slices (same order and
//                      rounding as the fused kernel) into an fp32 workspace
//                      (the all-reduced gradient),
//   2. adamw_kernel    reads the workspace and master/m/v, applies AdamW and
//                      writes master/m/v and replica 0's bf16 parameters,
//   3. R-1 copies      broadcast replica 0's parameters to the other
//                      replicas (the parameter all-gather / broadcast).
// The values are bit-identical to the fused step; only the schedule
// differs.  It moves (2R + 4) + (4 + 24 + 2) + 4(R - 1) = 6R + 30 bytes per
// parameter against the fused 4R + 24 (78 against 56 at R = 8).

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "cc_dp_device.cuh"
#include "cc_dp_internal.h"
#include "cc_trace.h"

namespace ccdp {
namespace {

using namespace dev;

constexpr int kThreads = 256;

struct ReduceParams {
    const uint4 *g[CC_MAX_R];
    float4 *red;          // workspace, indexed from the bucket start
    size_t vec_begin;     // first 8-element vector of the bucket
    size_t num_vec;
    size_t tail_begin;    // absolute element index of the partial vector
    int tail_len;
};

template <int R>
__global__ void __launch_bounds__(kThreads)
reduce_kernel(const __grid_constant__ ReduceParams p) {
    const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
    for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
         i < p.num_vec; i += stride) {
        uint4 gq[R];
#pragma unroll
        for (int r = 0; r < R; ++r) gq[r] = __ldcs(p.g[r] + p.vec_begin + i);
        float s[8];
        widen8(gq[0], s);
#pragma unroll
        for (int r = 1; r < R; ++r) add8_bf16(s, gq[r]);
        __stcs(p.red + 2 * i, make_float4(s[0], s[1], s[2], s[3]));
        __stcs(p.red + 2 * i + 1, make_float4(s[4], s[5], s[6], s[7]));
    }
    if (blockIdx.x == gridDim.x - 1 && static_cast<int>(threadIdx.x) < p.tail_len) {
        const size_t e = p.tail_begin + threadIdx.x;
        float s = bf16_at(p.g[0], e);
#pragma unroll
        for (int r = 1; r < R; ++r) s = __fadd_rn(s, bf16_at(p.g[r], e));
        reinterpret_cast<float *>(p.red)[8 * p.num_vec + threadIdx.x] = s;
    }
}

struct AdamParams {
    const float4 *red;
    float4 *master, *m, *v;
    uint4 *out0;
    AdamScalars c;
    size_t vec_begin, num_vec, tail_begin;
    int tail_len;
};

__global__ void __launch_bounds__(kThreads)
adamw_kernel(const __grid_constant__ AdamParams p) {
    const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
    for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
         i < p.num_vec; i += stride) {
        const size_t vi = p.vec_begin + i;
        const float4 r0 = __ldcs(p.red + 2 * i), r1 = __ldcs(p.red + 2 * i + 1);
        const float4 w0 = __ldcs(p.master + 2 * vi), w1 = __ldcs(p.master + 2 * vi + 1);
        const float4 m0 = __ldcs(p.m + 2 * vi), m1 = __ldcs(p.m + 2 * vi + 1);
        const float4 v0 = __ldcs(p.v + 2 * vi), v1 = __ldcs(p.v + 2 * vi + 1);
        const float s[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        float pw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        float mm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) adamw(s[k], pw[k], mm[k], vv[k], p.c);
        __stcs(p.master + 2 * vi, make_float4(pw[0], pw[1], pw[2], pw[3]));
        __stcs(p.master + 2 * vi + 1, make_float4(pw[4], pw[5], pw[6], pw[7]));
        __stcs(p.m + 2 * vi, make_float4(mm[0], mm[1], mm[2], mm[3]));
        __stcs(p.m + 2 * vi + 1, make_float4(mm[4], mm[5], mm[6], mm[7]));
        __stcs(p.v + 2 * vi, make_float4(vv[0], vv[1], vv[2], vv[3]));
        __stcs(p.v + 2 * vi + 1, make_float4(vv[4], vv[5], vv[6], vv[7]));
        __stcs(p.out0 + vi, make_uint4(pack_bf16x2(pw[0], pw[1]), pack_bf16x2(pw[2], pw[3]),
                                       pack_bf16x2(pw[4], pw[5]), pack_bf16x2(pw[6], pw[7])));
    }
    if (blockIdx.x == gridDim.x - 1 && static_cast<int>(threadIdx.x) < p.tail_len) {
        const size_t e = p.tail_begin + threadIdx.x;
        float *pm = reinterpret_cast<float *>(p.master);
        float *mm = reinterpret_cast<float *>(p.m);
        float *vv = reinterpret_cast<float *>(p.v);
        float pw = pm[e], m = mm[e], v = vv[e];
        adamw(reinterpret_cast<const float *>(p.red)[8 * p.num_vec + threadIdx.x], pw, m, v, p.c);
        pm[e] = pw;
        mm[e] = m;
        vv[e] = v;
        reinterpret_cast<__nv_bfloat16 *>(p.out0)[e] = __float2bfloat16_rn(pw);
    }
}

using ReduceKernel = void (*)(ReduceParams);

template <int R>
ReduceKernel reduce_for() { return reduce_kernel<R>; }

ReduceKernel reduce_kernel_for(int R) {
    switch (R) {
        case 1: return reduce_for<1>();   case 2: return reduce_for<2>();
        case 3: return reduce_for<3>();   case 4: return reduce_for<4>();
        case 5: return reduce_for<5>();   case 6: return reduce_for<6>();
        case 7: return reduce_for<7>();   case 8: return reduce_for<8>();
        case 9: return reduce_for<9>();   case 10: return reduce_for<10>();
        case 11: return reduce_for<11>(); case 12: return reduce_for<12>();
        case 13: return reduce_for<13>(); case 14: return reduce_for<14>();
        case 15: return reduce_for<15>(); case 16: return reduce_for<16>();
        default: return nullptr;
    }
}

unsigned grid_for(size_t num_vec, int sms) {
    size_t blocks = (num_vec + kThreads - 1) / kThreads;
    const size_t cap = static_cast<size_t>(sms) * 64;
    if (blocks > cap) blocks = cap;
    return static_cast<unsigned>(blocks == 0 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_unfused_bucket(const Slabs &s, const AdamScalars &c, float *workspace,
                                  size_t begin, size_t end, cudaStream_t stream) {
    if (end <= begin) return cudaSuccess;
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    const size_t num_vec = (end - begin) / CC_PAD_ELEMS;
    const size_t tail_begin = begin + num_vec * CC_PAD_ELEMS;
    const int tail_len = static_cast<int>(end - tail_begin);
    const unsigned grid = grid_for(num_vec, sms);

    ReduceParams rp{};
    for (int r = 0; r < s.R; ++r) rp.g[r] = static_cast<const uint4 *>(s.grads[r]);
    rp.red = reinterpret_cast<float4 *>(workspace);
    rp.vec_begin = begin / CC_PAD_ELEMS;
    rp.num_vec = num_vec;
    rp.tail_begin = tail_begin;
    rp.tail_len = tail_len;
    reduce_kernel_for(s.R)<<<grid, kThreads, 0, stream>>>(rp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    AdamParams ap{};
    ap.red = reinterpret_cast<const float4 *>(workspace);
    ap.master = reinterpret_cast<float4 *>(s.master);
    ap.m = reinterpret_cast<float4 *>(s.m);
    ap.v = reinterpret_cast<float4 *>(s.v);
    ap.out0 = static_cast<uint4 *>(s.out[0]);
    ap.c = c;
    ap.vec_begin = begin / CC_PAD_ELEMS;
    ap.num_vec = num_vec;
    ap.tail_begin = tail_begin;
    ap.tail_len = tail_len;
    adamw_kernel<<<grid, kThreads, 0, stream>>>(ap);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const size_t bytes = 2 * (end - begin);
    const char *src = static_cast<const char *>(s.out[0]) + 2 * begin;
    for (int r = 1; r < s.R; ++r) {
        // Default: replica slabs may be page-locked host memory.
        e = cudaMemcpyAsync(static_cast<char *>(s.out[r]) + 2 * begin, src, bytes,
                            cudaMemcpyDefault, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace ccdp

// ---------------------------------------------------------------------------
// The unfused step without a caller-provided workspace.
//
// Some callers cannot hand the library a scratch buffer or call cudaMalloc
// themselves: code that runs inside a framework whose caching allocator
// owns nearly all of the device memory (a raw cudaMalloc outside it can fail
// or fragment the pool), loops where an allocation or free would stall the
// device (cudaFree synchronises), and plugins that are given buffers but no
// right to allocate.  For them the reduced gradient of one bucket lives in a
// fixed array in the library's own device memory, which every GPU that
// loads the library holds until the process exits.
// ---------------------------------------------------------------------------

namespace ccdp {
namespace {

// Scratch of the allocation-free entry point: one bucket's fp32 reduced
// gradient, CC_NOALLOC_SCRATCH_ELEMS elements (64 MiB).
static __device__ __align__(256) float g_noalloc_scratch[CC_NOALLOC_SCRATCH_ELEMS];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
struct ScratchAddress {
    CUcontext ctx;   // the context the address was looked up in
    float *ptr;
};
ScratchAddress g_scratch_addr[kMaxScratchDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

// cuCtxGetCurrent through the runtime's driver entry points (no link-time
// libcuda), looked up once.
CtxGetCurrentFn ctx_get_current_fn() {
    static const CtxGetCurrentFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    return fn;
}

// The device address of g_noalloc_scratch on the current device.  In host
// code the array's name is only a host-side stand-in, so the address comes
// from cudaGetSymbolAddress, looked up once per device and context: a
// device reset destroys the primary context and the module with it, so a
// context other than the one of the last lookup means a new lookup.
int scratch_address(float **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxScratchDevices)
        return fail(CC_ERR_UNSUPPORTED, "device %d beyond the %d supported", dev,
                    kMaxScratchDevices);
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    if (!get_ctx) return fail(CC_ERR_UNSUPPORTED, "cuCtxGetCurrent unavailable");
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddress &a = g_scratch_addr[dev];
    if (!ctx || !a.ptr || a.ctx != ctx) {
        // The lookup makes the device's primary context current if no
        // context was; the context is then read again for the cache key.
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(scratch)");
        if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
        a.ptr = static_cast<float *>(p);
        a.ctx = ctx;
    }
    *out = a.ptr;
    return CC_OK;
}

}  // namespace
}  // namespace ccdp

extern "C" int cc_unfused_dp_step_noalloc(const void *const *grads, float *master, float *m,
                                          float *v, void *const *params_out, size_t n, int R,
                                          size_t bucket_bytes, float lr, float beta1,
                                          float beta2, float eps, float weight_decay,
                                          int step, float grad_scale, void *stream) {
    using namespace ccdp;
    TraceRange call("cc_unfused_dp_step_noalloc", n);
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    AdamScalars c;
    int st = make_scalars(lr, beta1, beta2, eps, weight_decay, step, grad_scale, &c);
    if (st != CC_OK) return st;
    if (n == 0) return CC_OK;
    const size_t per = bucket_elems(bucket_bytes, n);
    const size_t largest = per < n ? per : n;
    if (largest > CC_NOALLOC_SCRATCH_ELEMS) {
        if (bucket_bytes == 0 || per >= n)
            return fail(CC_ERR_INVALID,
                        "n=%zu elements in one bucket exceed the fixed scratch of %u "
                        "elements; cut the step into buckets of at most %u elements "
                        "(bucket_bytes < %u) or use cc_unfused_dp_step with a workspace",
                        n, static_cast<unsigned>(CC_NOALLOC_SCRATCH_ELEMS),
                        static_cast<unsigned>(CC_NOALLOC_SCRATCH_ELEMS),
                        static_cast<unsigned>(2u * CC_NOALLOC_SCRATCH_ELEMS + 16u));
        return fail(CC_ERR_INVALID,
                    "bucket_bytes=%zu gives buckets of %zu elements (floor(bucket_bytes/16)*8), "
                    "more than the fixed scratch of %u elements; use bucket_bytes < %u "
                    "or cc_unfused_dp_step with a workspace",
                    bucket_bytes, per, static_cast<unsigned>(CC_NOALLOC_SCRATCH_ELEMS),
                    static_cast<unsigned>(2u * CC_NOALLOC_SCRATCH_ELEMS + 16u));
    }
    Slabs s;
    st = validate_slabs(grads, nullptr, master, m, v, params_out, n, R, false, &s);
    if (st != CC_OK) return st;
    float *scratch = nullptr;
    if ((st = scratch_address(&scratch)) != CC_OK) return st;
    // The reduce kernel overwrites every scratch element a bucket uses before
    // the AdamW kernel reads it, so nothing needs clearing between calls.
    for (size_t b = 0; b < n; b += per) {
        const size_t e = b + per < n ? b + per : n;
        if (injected_failure())
            return fail(CC_ERR_CUDA, "injected launch failure before the bucket at element %zu", b);
        TraceRange bucket("bucket", b);
        const cudaError_t err = launch_unfused_bucket(s, c, scratch, b, e,
                                                      static_cast<cudaStream_t>(stream));
        if (err != cudaSuccess) return fail_cuda(err, "allocation-free step launch");
    }
    return CC_OK;
}
