// The tensor-parallel MatMul-then-AllReduce, overlapped in chunks ("LIT-735:
// Breaking the Computation and Communication Abstraction Barrier in
// Distributed Machine Learning Workloads", Key takeaways: for the
// model-parallel MatMul and the AllReduce that follows it, overlapping the
// two in chunks hides most of the MatMul's time).
//
// R tensor-parallel ranks are emulated in one GPU: rank r holds its shard
// X_r = X[:, K_r] and W_r = W[K_r, :] of a row-parallel linear layer and
// computes the partial product Y_r = X_r W_r (bf16 inputs, fp32 output).
// The AllReduce hands every rank the same Y = sum of the Y_r, summed in rank
// order in fp32 and rounded once to bf16: tp_allreduce_kernel reads the R
// partials of a range and writes the R bf16 replicas, 6R bytes per element.
// cc_tp_overlap_bench splits the rows into chunks; each chunk's AllReduce
// starts on a side stream as soon as that chunk's R GEMMs are done, while
// the next chunk's GEMMs run (stream events only, no device waits).  The
// GEMMs are cuBLAS (a plain library GEMM); the reduction is this file's.

#include <cublas_v2.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "cc_dp_device.cuh"
#include "cc_dp_internal.h"
#include "cc_trace.h"

namespace ccdp {
namespace {

using namespace dev;

constexpr int kThreads = 256;

struct TpParams {
    const float4 *part[CC_MAX_R];
    uint4 *out[CC_MAX_R];
    size_t vec_begin, num_vec, tail_begin;
    int tail_len;
};

template <int R>
__global__ void __launch_bounds__(kThreads)
tp_allreduce_kernel(const __grid_constant__ TpParams p) {
    const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
    for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
         i < p.num_vec; i += stride) {
        const size_t vi = p.vec_begin + i;
        float4 q[R][2];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            q[r][0] = __ldcs(p.part[r] + 2 * vi);
            q[r][1] = __ldcs(p.part[r] + 2 * vi + 1);
        }
        float s[8] = {q[0][0].x, q[0][0].y, q[0][0].z, q[0][0].w,
                      q[0][1].x, q[0][1].y, q[0][1].z, q[0][1].w};
#pragma unroll
        for (int r = 1; r < R; ++r) {
            s[0] = __fadd_rn(s[0], q[r][0].x); s[1] = __fadd_rn(s[1], q[r][0].y);
            s[2] = __fadd_rn(s[2], q[r][0].z); s[3] = __fadd_rn(s[3], q[r][0].w);
            s[4] = __fadd_rn(s[4], q[r][1].x); s[5] = __fadd_rn(s[5], q[r][1].y);
            s[6] = __fadd_rn(s[6], q[r][1].z); s[7] = __fadd_rn(s[7], q[r][1].w);
        }
        const uint4 o = make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]),
                                   pack_bf16x2(s[4], s[5]), pack_bf16x2(s[6], s[7]));
#pragma unroll
        for (int r = 0; r < R; ++r) __stcs(p.out[r] + vi, o);
    }
    if (blockIdx.x == gridDim.x - 1 && static_cast<int>(threadIdx.x) < p.tail_len) {
        const size_t e = p.tail_begin + threadIdx.x;
        float s = reinterpret_cast<const float *>(p.part[0])[e];
#pragma unroll
        for (int r = 1; r < R; ++r) s = __fadd_rn(s, reinterpret_cast<const float *>(p.part[r])[e]);
        const __nv_bfloat16 b = __float2bfloat16_rn(s);
#pragma unroll
        for (int r = 0; r < R; ++r) reinterpret_cast<__nv_bfloat16 *>(p.out[r])[e] = b;
    }
}

using TpKernel = void (*)(TpParams);

template <int R>
TpKernel tp_for() { return tp_allreduce_kernel<R>; }

TpKernel tp_kernel_for(int R) {
    switch (R) {
        case 1: return tp_for<1>();   case 2: return tp_for<2>();
        case 3: return tp_for<3>();   case 4: return tp_for<4>();
        case 5: return tp_for<5>();   case 6: return tp_for<6>();
        case 7: return tp_for<7>();   case 8: return tp_for<8>();
        case 9: return tp_for<9>();   case 10: return tp_for<10>();
        case 11: return tp_for<11>(); case 12: return tp_for<12>();
        case 13: return tp_for<13>(); case 14: return tp_for<14>();
        case 15: return tp_for<15>(); case 16: return tp_for<16>();
        default: return nullptr;
    }
}

// [begin, end) of R slabs; begin a multiple of 8.
cudaError_t launch_tp_allreduce(const float *const *part, void *const *out, int R,
                                size_t begin, size_t end, cudaStream_t stream) {
    if (end <= begin) return cudaSuccess;
    TpParams p{};
    for (int r = 0; r < R; ++r) {
        p.part[r] = reinterpret_cast<const float4 *>(part[r]);
        p.out[r] = static_cast<uint4 *>(out[r]);
    }
    p.vec_begin = begin / CC_PAD_ELEMS;
    p.num_vec = (end - begin) / CC_PAD_ELEMS;
    p.tail_begin = begin + p.num_vec * CC_PAD_ELEMS;
    p.tail_len = static_cast<int>(end - p.tail_begin);
    size_t blocks = (p.num_vec + kThreads - 1) / kThreads;
    if (blocks > 0x7FFFFFFFu) blocks = 0x7FFFFFFFu;
    if (blocks == 0) blocks = 1;
    tp_kernel_for(R)<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

struct Range2 {
    uintptr_t lo, hi;
    bool written;
};

// R, alignment, aliasing and device ranges of R partial and R output slabs.
int validate_tp(const float *const *part, void *const *out, size_t n, int R) {
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    if (!part || !out) return fail(CC_ERR_INVALID, "partials/out arrays are NULL");
    std::vector<Range2> rs;
    for (int r = 0; r < R; ++r) {
        const void *ps[2] = {part[r], out[r]};
        const size_t bytes[2] = {4 * n, 2 * n};
        for (int k = 0; k < 2; ++k) {
            if (!ps[k]) return fail(CC_ERR_INVALID, "%s[%d] is NULL", k ? "out" : "partials", r);
            if (reinterpret_cast<uintptr_t>(ps[k]) % 16 != 0)
                return fail(CC_ERR_MISALIGNED, "%s[%d]=%p is not 16-byte aligned",
                            k ? "out" : "partials", r, ps[k]);
            const uintptr_t lo = reinterpret_cast<uintptr_t>(ps[k]);
            rs.push_back({lo, lo + bytes[k], k == 1});
        }
    }
    for (size_t i = 0; i < rs.size(); ++i)
        for (size_t j = i + 1; j < rs.size(); ++j)
            if ((rs[i].written || rs[j].written) && rs[i].lo < rs[j].hi && rs[j].lo < rs[i].hi)
                return fail(CC_ERR_ALIAS, "partial/output slabs overlap");
    int st = ensure_device();
    if (st != CC_OK) return st;
    for (const Range2 &r : rs)
        if ((st = check_device_range(reinterpret_cast<const void *>(r.lo), r.hi - r.lo,
                                     r.written ? "out" : "partials")) != CC_OK)
            return st;
    return CC_OK;
}

struct TpResources {
    cudaStream_t comp = nullptr, side = nullptr;
    cudaEvent_t start = nullptr, stop = nullptr, side_done = nullptr;
    std::vector<cudaEvent_t> chunk;
    cublasHandle_t blas = nullptr;
    ~TpResources() {
        if (comp) cudaStreamSynchronize(comp);
        if (side) cudaStreamSynchronize(side);
        if (blas) cublasDestroy(blas);
        for (cudaEvent_t e : chunk)
            if (e) cudaEventDestroy(e);
        if (start) cudaEventDestroy(start);
        if (stop) cudaEventDestroy(stop);
        if (side_done) cudaEventDestroy(side_done);
        if (comp) cudaStreamDestroy(comp);
        if (side) cudaStreamDestroy(side);
    }
};

struct TpBench {
    const cc_tp_cfg &c;
    TpResources &res;
    size_t rows;   // rows per chunk
    size_t kr;     // K / R

    // Byte strides when the R shards of x, w and partials sit at equal
    // distances (one buffer cut into R slabs): then a chunk's R products are
    // one strided-batched GEMM instead of R small ones.
    bool batched = false;
    long long sx = 0, sw = 0, sp = 0;

    void find_strides() {
        if (c.R < 2) return;
        auto d = [](const void *a, const void *b) {
            return static_cast<long long>(reinterpret_cast<uintptr_t>(b)) -
                   static_cast<long long>(reinterpret_cast<uintptr_t>(a));
        };
        sx = d(c.x[0], c.x[1]);
        sw = d(c.w[0], c.w[1]);
        sp = d(c.partials[0], c.partials[1]);
        batched = sx % 2 == 0 && sw % 2 == 0 && sp % 4 == 0;
        for (int r = 2; r < c.R && batched; ++r)
            batched = d(c.x[r - 1], c.x[r]) == sx && d(c.w[r - 1], c.w[r]) == sw &&
                      d(c.partials[r - 1], c.partials[r]) == sp;
    }

    // The R partial products of one chunk of rows: Y_r = X_r W_r, row-major,
    // as the column-major C^T = B^T A^T.
    int gemms(int chunk) {
        const float alpha = 1.0f, beta = 0.0f;
        if (batched) {
            const char *x = static_cast<const char *>(c.x[0]) + 2 * chunk * rows * kr;
            char *y = reinterpret_cast<char *>(c.partials[0]) + 4 * chunk * rows * c.n;
            const cublasStatus_t st = cublasGemmStridedBatchedEx(
                res.blas, CUBLAS_OP_N, CUBLAS_OP_N, c.n, static_cast<int>(rows),
                static_cast<int>(kr), &alpha, c.w[0], CUDA_R_16BF, c.n, sw / 2, x,
                CUDA_R_16BF, static_cast<int>(kr), sx / 2, &beta, y, CUDA_R_32F, c.n,
                sp / 4, c.R, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
            if (st != CUBLAS_STATUS_SUCCESS)
                return fail(CC_ERR_CUDA, "cublasGemmStridedBatchedEx failed (status %d)",
                            static_cast<int>(st));
            return CC_OK;
        }
        for (int r = 0; r < c.R; ++r) {
            const char *x = static_cast<const char *>(c.x[r]) + 2 * chunk * rows * kr;
            char *y = reinterpret_cast<char *>(c.partials[r]) + 4 * chunk * rows * c.n;
            const cublasStatus_t st = cublasGemmEx(
                res.blas, CUBLAS_OP_N, CUBLAS_OP_N, c.n, static_cast<int>(rows),
                static_cast<int>(kr), &alpha, c.w[r], CUDA_R_16BF, c.n, x, CUDA_R_16BF,
                static_cast<int>(kr), &beta, y, CUDA_R_32F, c.n, CUBLAS_COMPUTE_32F,
                CUBLAS_GEMM_DEFAULT);
            if (st != CUBLAS_STATUS_SUCCESS)
                return fail(CC_ERR_CUDA, "cublasGemmEx failed (status %d)", static_cast<int>(st));
        }
        return CC_OK;
    }

    int reduce(int chunk, cudaStream_t s) {
        const size_t per = rows * static_cast<size_t>(c.n);
        const cudaError_t e = launch_tp_allreduce(c.partials, c.out, c.R, chunk * per,
                                                  (chunk + 1) * per, s);
        return e == cudaSuccess ? CC_OK : fail_cuda(e, "all-reduce launch");
    }

    int arm(int which, float *ms) {
        cudaError_t e = cudaEventRecord(res.start, res.comp);
        if (e != cudaSuccess) return fail_cuda(e, "start event");
        int st = CC_OK;
        if (which == 0) {                       // the GEMMs alone
            for (int k = 0; k < c.chunks && st == CC_OK; ++k) st = gemms(k);
        } else if (which == 1) {                // the AllReduce alone
            for (int k = 0; k < c.chunks && st == CC_OK; ++k) st = reduce(k, res.comp);
        } else if (which == 2) {                // MatMul, then AllReduce
            for (int k = 0; k < c.chunks && st == CC_OK; ++k) st = gemms(k);
            for (int k = 0; k < c.chunks && st == CC_OK; ++k) st = reduce(k, res.comp);
        } else {                                // chunked overlap
            if ((e = cudaStreamWaitEvent(res.side, res.start, 0)) != cudaSuccess)
                return fail_cuda(e, "side wait");
            for (int k = 0; k < c.chunks && st == CC_OK; ++k) {
                if ((st = gemms(k)) != CC_OK) break;
                if ((e = cudaEventRecord(res.chunk[k], res.comp)) != cudaSuccess ||
                    (e = cudaStreamWaitEvent(res.side, res.chunk[k], 0)) != cudaSuccess)
                    return fail_cuda(e, "chunk event");
                st = reduce(k, res.side);
            }
            if (st == CC_OK) {
                if ((e = cudaEventRecord(res.side_done, res.side)) != cudaSuccess ||
                    (e = cudaStreamWaitEvent(res.comp, res.side_done, 0)) != cudaSuccess)
                    return fail_cuda(e, "join");
            }
        }
        if (st != CC_OK) return st;
        if ((e = cudaEventRecord(res.stop, res.comp)) != cudaSuccess) return fail_cuda(e, "stop event");
        if ((e = cudaEventSynchronize(res.stop)) != cudaSuccess) return fail_cuda(e, "arm sync");
        if ((e = cudaEventElapsedTime(ms, res.start, res.stop)) != cudaSuccess)
            return fail_cuda(e, "elapsed time");
        return CC_OK;
    }

    int median(int which, float *out) {
        float ms = 0.0f;
        for (int i = 0; i < c.warmup; ++i) {
            const int st = arm(which, &ms);
            if (st != CC_OK) return st;
        }
        std::vector<float> t(c.iters);
        for (int i = 0; i < c.iters; ++i) {
            const int st = arm(which, &t[i]);
            if (st != CC_OK) return st;
        }
        std::sort(t.begin(), t.end());
        *out = (c.iters % 2) ? t[c.iters / 2] : 0.5f * (t[c.iters / 2 - 1] + t[c.iters / 2]);
        return CC_OK;
    }
};

}  // namespace
}  // namespace ccdp

using namespace ccdp;

extern "C" int cc_tp_allreduce(const float *const *partials, void *const *out, size_t n,
                               int R, void *stream) {
    TraceRange call("cc_tp_allreduce", n);
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    if (n == 0) return CC_OK;
    if (n > SIZE_MAX / 8) return fail(CC_ERR_INVALID, "n=%zu too large", n);
    int st = validate_tp(partials, out, n, R);
    if (st != CC_OK) return st;
    const cudaError_t e = launch_tp_allreduce(partials, out, R, 0, n,
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CC_OK : fail_cuda(e, "all-reduce launch");
}

extern "C" int cc_tp_overlap_bench(const cc_tp_cfg *cfg, cc_tp_result *out) {
    if (!cfg || !out) return fail(CC_ERR_INVALID, "cfg/out is NULL");
    const cc_tp_cfg &c = *cfg;
    if (c.R < 1 || c.R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", c.R, CC_MAX_R);
    if (c.m < 1 || c.n < 1 || c.k < 1 || c.k % c.R != 0)
        return fail(CC_ERR_INVALID, "need m, n, k >= 1 and k divisible by R=%d", c.R);
    if (c.chunks < 1 || c.chunks > 4096 || c.m % c.chunks != 0)
        return fail(CC_ERR_INVALID, "chunks=%d must divide m=%d (at most 4096)", c.chunks, c.m);
    const size_t rows = static_cast<size_t>(c.m / c.chunks), kr = static_cast<size_t>(c.k / c.R);
    if ((rows * c.n) % CC_PAD_ELEMS != 0 || kr % CC_PAD_ELEMS != 0)
        return fail(CC_ERR_MISALIGNED, "rows per chunk x n and k/R must be multiples of %d",
                    CC_PAD_ELEMS);
    if (c.iters < 1 || c.iters > 1000 || c.warmup < 0 || c.warmup > 1000)
        return fail(CC_ERR_INVALID, "iters=%d must be in 1..1000, warmup in 0..1000", c.iters);
    if (c.stream_priority < 0 || c.stream_priority > 2)
        return fail(CC_ERR_INVALID, "stream_priority=%d must be 0, 1 or 2", c.stream_priority);
    if (!c.x || !c.w) return fail(CC_ERR_INVALID, "x/w arrays are NULL");
    const size_t total = static_cast<size_t>(c.m) * c.n;
    int st = validate_tp(c.partials, c.out, total, c.R);
    if (st != CC_OK) return st;
    for (int r = 0; r < c.R; ++r) {
        if (!c.x[r] || !c.w[r]) return fail(CC_ERR_INVALID, "x[%d]/w[%d] is NULL", r, r);
        if ((st = check_device_range(c.x[r], 2 * static_cast<size_t>(c.m) * kr, "x")) != CC_OK ||
            (st = check_device_range(c.w[r], 2 * kr * c.n, "w")) != CC_OK)
            return st;
    }

    TpResources res;
    cudaError_t e;
    int lo = 0, hi = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess)
        return fail_cuda(e, "priority range");
    if ((e = cudaStreamCreateWithPriority(&res.comp, cudaStreamNonBlocking,
                                          c.stream_priority == 2 ? hi : lo)) != cudaSuccess ||
        (e = cudaStreamCreateWithPriority(&res.side, cudaStreamNonBlocking,
                                          c.stream_priority == 1 ? hi : lo)) != cudaSuccess)
        return fail_cuda(e, "stream create");
    if ((e = cudaEventCreate(&res.start)) != cudaSuccess ||
        (e = cudaEventCreate(&res.stop)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&res.side_done, cudaEventDisableTiming)) != cudaSuccess)
        return fail_cuda(e, "event create");
    res.chunk.assign(c.chunks, nullptr);
    for (int k = 0; k < c.chunks; ++k)
        if ((e = cudaEventCreateWithFlags(&res.chunk[k], cudaEventDisableTiming)) != cudaSuccess)
            return fail_cuda(e, "chunk event create");
    if (cublasCreate(&res.blas) != CUBLAS_STATUS_SUCCESS ||
        cublasSetStream(res.blas, res.comp) != CUBLAS_STATUS_SUCCESS)
        return fail(CC_ERR_CUDA, "cuBLAS set-up failed");

    TpBench bench{c, res, rows, kr};
    bench.find_strides();
    cc_tp_result r{};
    if ((st = bench.median(0, &r.t_gemm_ms)) != CC_OK) return st;
    if ((st = bench.median(1, &r.t_allreduce_ms)) != CC_OK) return st;
    if ((st = bench.median(2, &r.t_sequential_ms)) != CC_OK) return st;
    if ((st = bench.median(3, &r.t_overlap_ms)) != CC_OK) return st;
    *out = r;
    return CC_OK;
}
