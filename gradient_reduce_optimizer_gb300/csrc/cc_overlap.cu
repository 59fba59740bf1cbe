// Overlap measurement for the bucketed fused step (cc_overlap_bench in
// include/cc_dp.h).
//
// "Communication Optimization › Communication Overlap": DDP launches each
// bucket's reduction on a separate CUDA stream as soon as all gradients in it
// are ready, last layer first, and the step time is approximately
// T_fwd + T_bwd + max(0, T_comm - T_overlap).  Here the backward pass is a
// proxy of bf16 GEMMs on a compute stream that records one event per layer;
// the side stream waits on the event of each bucket's ready layer and then
// launches that bucket's fused reduce+AdamW+redistribute kernel.  The naive
// synchronous schedule (backward, then reduction and optimizer, in strict
// phases) is the sequential arm.  Stream ordering uses events only: no
// kernel waits on a flag.
//
// The reduction is an SM kernel that needs most SMs to stream at HBM speed,
// and cuBLAS's GEMMs occupy every SM, so left to the block scheduler the two
// take turns.  With comm_sms > 0 the overlapped arm runs on a spatial
// partition instead: two green contexts with disjoint SM sets, the buckets'
// stream on comm_sms SMs and the GEMMs' stream on the rest.  The other arms
// keep the whole GPU, so exposed time is still measured against the
// unpartitioned backward.

#include <cublasLt.h>
#include <cublas_v2.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "cc_dp_internal.h"
#include "cc_trace.h"

namespace ccdp {
namespace {

// Green-context driver calls, resolved through the runtime (no link-time
// libcuda).
struct GreenApi {
    decltype(&cuDeviceGetDevResource) get_resource = nullptr;
    decltype(&cuDevSmResourceSplitByCount) split = nullptr;
    decltype(&cuDevResourceGenerateDesc) make_desc = nullptr;
    decltype(&cuGreenCtxCreate) create = nullptr;
    decltype(&cuGreenCtxDestroy) destroy = nullptr;
    decltype(&cuGreenCtxStreamCreate) stream_create = nullptr;
    decltype(&cuStreamDestroy) stream_destroy = nullptr;
    bool ok = false;
};

template <typename F>
bool resolve(F *fn, const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 13000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return false;
    *fn = reinterpret_cast<F>(p);
    return true;
}

const GreenApi &green_api() {
    static const GreenApi api = [] {
        GreenApi a;
        a.ok = resolve(&a.get_resource, "cuDeviceGetDevResource") &&
               resolve(&a.split, "cuDevSmResourceSplitByCount") &&
               resolve(&a.make_desc, "cuDevResourceGenerateDesc") &&
               resolve(&a.create, "cuGreenCtxCreate") &&
               resolve(&a.destroy, "cuGreenCtxDestroy") &&
               resolve(&a.stream_create, "cuGreenCtxStreamCreate") &&
               resolve(&a.stream_destroy, "cuStreamDestroy");
        return a;
    }();
    return api;
}

struct Resources {
    cudaStream_t comp = nullptr, side = nullptr;
    cudaEvent_t start = nullptr, stop = nullptr, side_done = nullptr;
    std::vector<cudaEvent_t> layer;
    cublasHandle_t blas = nullptr;
    // gemm_algo > 0: the GEMMs through cuBLASLt with that heuristic candidate
    cublasLtHandle_t lt = nullptr;
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t lay_b = nullptr, lay_a = nullptr, lay_c = nullptr;
    cublasLtMatmulAlgo_t algo{};
    int algos = 0;
    // the spatial partition of the overlapped arm (comm_sms > 0)
    CUgreenCtx green_comp = nullptr, green_side = nullptr;
    CUstream gcomp = nullptr, gside = nullptr;
    int comm_sms = 0, compute_sms = 0;

    ~Resources() {
        if (comp) cudaStreamSynchronize(comp);
        if (side) cudaStreamSynchronize(side);
        const GreenApi &g = green_api();
        if (gcomp) cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(gcomp));
        if (gside) cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(gside));
        if (blas) cublasDestroy(blas);
        if (lay_a) cublasLtMatrixLayoutDestroy(lay_a);
        if (lay_b) cublasLtMatrixLayoutDestroy(lay_b);
        if (lay_c) cublasLtMatrixLayoutDestroy(lay_c);
        if (op) cublasLtMatmulDescDestroy(op);
        if (lt) cublasLtDestroy(lt);
        if (gcomp) g.stream_destroy(gcomp);
        if (gside) g.stream_destroy(gside);
        if (green_comp) g.destroy(green_comp);
        if (green_side) g.destroy(green_side);
        for (cudaEvent_t e : layer)
            if (e) cudaEventDestroy(e);
        if (start) cudaEventDestroy(start);
        if (stop) cudaEventDestroy(stop);
        if (side_done) cudaEventDestroy(side_done);
        if (comp) cudaStreamDestroy(comp);
        if (side) cudaStreamDestroy(side);
    }
};

// Split the current device's SMs into comm_sms (rounded up by the driver to
// its partition granularity) for the buckets and the rest for the GEMMs.
int make_partition(int want, int prio_comp, int prio_side, Resources &res) {
    const GreenApi &g = green_api();
    if (!g.ok) return fail(CC_ERR_UNSUPPORTED, "green contexts unavailable in this driver");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    CUdevResource all{}, part{}, rest{};
    if (g.get_resource(static_cast<CUdevice>(dev), &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS)
        return fail(CC_ERR_CUDA, "cuDeviceGetDevResource failed");
    if (want >= static_cast<int>(all.sm.smCount))
        return fail(CC_ERR_INVALID, "comm_sms=%d must be below the %u SMs", want,
                    all.sm.smCount);
    unsigned groups = 1;
    CUresult r = g.split(&part, &groups, &all, &rest, 0, static_cast<unsigned>(want));
    if (r != CUDA_SUCCESS || groups != 1 || rest.sm.smCount == 0)
        return fail(CC_ERR_INVALID, "cannot split %u SMs into %d + rest (CUresult %d)",
                    all.sm.smCount, want, static_cast<int>(r));
    CUdevResourceDesc dpart = nullptr, drest = nullptr;
    if (g.make_desc(&dpart, &part, 1) != CUDA_SUCCESS ||
        g.make_desc(&drest, &rest, 1) != CUDA_SUCCESS)
        return fail(CC_ERR_CUDA, "cuDevResourceGenerateDesc failed");
    if (g.create(&res.green_side, dpart, static_cast<CUdevice>(dev),
                 CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS ||
        g.create(&res.green_comp, drest, static_cast<CUdevice>(dev),
                 CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS)
        return fail(CC_ERR_CUDA, "cuGreenCtxCreate failed");
    if (g.stream_create(&res.gside, res.green_side, CU_STREAM_NON_BLOCKING, prio_side) !=
            CUDA_SUCCESS ||
        g.stream_create(&res.gcomp, res.green_comp, CU_STREAM_NON_BLOCKING, prio_comp) !=
            CUDA_SUCCESS)
        return fail(CC_ERR_CUDA, "cuGreenCtxStreamCreate failed");
    res.comm_sms = static_cast<int>(part.sm.smCount);
    res.compute_sms = static_cast<int>(rest.sm.smCount);
    return CC_OK;
}

// The proxy GEMM through cuBLASLt, column-major C^T[N,M] = B^T[N,K] A^T[K,M]
// (the same product as the cublasGemmEx call), with heuristic candidate
// gemm_algo (1-based) among those that need no workspace.  Candidates differ
// in tile shape and pipeline depth, and so in the registers and shared
// memory their CTAs hold -- what decides whether a reduction block can run
// on the same SM.
int pick_lt_algo(const cc_overlap_cfg &c, Resources &res) {
    const uint64_t M = c.gemm_m, N = c.gemm_n, K = c.gemm_k;
    if (cublasLtCreate(&res.lt) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulDescCreate(&res.op, CUBLAS_COMPUTE_32F, CUDA_R_32F) !=
            CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&res.lay_b, CUDA_R_16BF, N, K, N) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&res.lay_a, CUDA_R_16BF, K, M, K) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&res.lay_c, CUDA_R_16BF, N, M, N) != CUBLAS_STATUS_SUCCESS)
        return fail(CC_ERR_CUDA, "cuBLASLt descriptor setup failed");
    cublasLtMatmulPreference_t pref = nullptr;
    if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS)
        return fail(CC_ERR_CUDA, "cuBLASLt preference create failed");
    const size_t no_workspace = 0;
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES,
                                         &no_workspace, sizeof no_workspace);
    constexpr int kMaxAlgos = 32;
    cublasLtMatmulHeuristicResult_t cand[kMaxAlgos];
    int found = 0;
    const cublasStatus_t hs = cublasLtMatmulAlgoGetHeuristic(
        res.lt, res.op, res.lay_b, res.lay_a, res.lay_c, res.lay_c, pref, kMaxAlgos, cand,
        &found);
    cublasLtMatmulPreferenceDestroy(pref);
    if (hs != CUBLAS_STATUS_SUCCESS)
        return fail(CC_ERR_CUDA, "cuBLASLt heuristic failed (status %d)", static_cast<int>(hs));
    res.algos = found;
    if (c.gemm_algo > found)
        return fail(CC_ERR_INVALID, "gemm_algo=%d but cuBLASLt offers %d candidates",
                    c.gemm_algo, found);
    res.algo = cand[c.gemm_algo - 1].algo;
    return CC_OK;
}

struct Bench {
    const cc_overlap_cfg &cfg;
    const Slabs &slabs;
    const AdamScalars &scalars;
    Resources &res;

    // One layer's GEMMs: C[M,N] = A[M,K] B[K,N] in row-major terms, i.e.
    // C^T = B^T A^T for column-major cuBLAS.
    cublasStatus_t gemms() {
        const float alpha = 1.0f, beta = 0.0f;
        if (cfg.gemm_algo > 0) {
            for (int g = 0; g < cfg.gemms_per_layer; ++g) {
                const cublasStatus_t st = cublasLtMatmul(
                    res.lt, res.op, &alpha, cfg.gemm_b, res.lay_b, cfg.gemm_a, res.lay_a,
                    &beta, cfg.gemm_c, res.lay_c, cfg.gemm_c, res.lay_c, &res.algo, nullptr,
                    0, comp);
                if (st != CUBLAS_STATUS_SUCCESS) return st;
            }
            return CUBLAS_STATUS_SUCCESS;
        }
        for (int g = 0; g < cfg.gemms_per_layer; ++g) {
            const cublasStatus_t st = cublasGemmEx(
                res.blas, CUBLAS_OP_N, CUBLAS_OP_N, cfg.gemm_n, cfg.gemm_m, cfg.gemm_k,
                &alpha, cfg.gemm_b, CUDA_R_16BF, cfg.gemm_n, cfg.gemm_a, CUDA_R_16BF,
                cfg.gemm_k, &beta, cfg.gemm_c, CUDA_R_16BF, cfg.gemm_n,
                CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
            if (st != CUBLAS_STATUS_SUCCESS) return st;
        }
        return CUBLAS_STATUS_SUCCESS;
    }

    // Streams of the arm being run (the partitioned pair for the overlapped
    // arm when a partition exists, else the whole-GPU pair).
    cudaStream_t comp = nullptr, side = nullptr;

    int backward(bool record_layers) {
        for (int l = cfg.num_layers - 1; l >= 0; --l) {
            TraceRange layer("proxy backward layer", static_cast<uint64_t>(l));
            const cublasStatus_t st = gemms();
            if (st != CUBLAS_STATUS_SUCCESS)
                return fail(CC_ERR_CUDA, "cublasGemmEx failed (status %d)", static_cast<int>(st));
            if (record_layers) {
                const cudaError_t e = cudaEventRecord(res.layer[l], comp);
                if (e != cudaSuccess) return fail_cuda(e, "layer event record");
            }
        }
        return CC_OK;
    }

    int buckets(cudaStream_t s, bool wait_ready, int max_ctas) {
        for (int b = 0; b < cfg.num_buckets; ++b) {
            TraceRange bucket("bucket", cfg.bucket_begin[b]);
            // Past the budgeted buckets, a bucket waits for the end of the
            // backward (layer 0's event) and takes the whole GPU.
            const bool wide = wait_ready && cfg.budget_buckets > 0 && b >= cfg.budget_buckets;
            const int ready = wide ? 0 : cfg.bucket_ready_layer[b];
            cudaError_t e = cudaSuccess;
            if (wait_ready) e = cudaStreamWaitEvent(s, res.layer[ready], 0);
            if (e == cudaSuccess)
                e = launch_step_range(slabs, scalars, cfg.bucket_begin[b], cfg.bucket_end[b],
                                      wide ? 0 : max_ctas, /*chain=*/!wait_ready && b > 0, s);
            if (e != cudaSuccess) return fail_cuda(e, "bucket launch");
        }
        return CC_OK;
    }

    // Runs one arm once and returns its elapsed milliseconds in *ms.
    int arm(int which, float *ms) {
        static const char *const kArmNames[4] = {"arm: backward alone", "arm: buckets alone",
                                                 "arm: overlapped", "arm: sequential"};
        TraceRange range(kArmNames[which], static_cast<uint64_t>(which));
        const bool part = which == 2 && res.gcomp;
        comp = part ? reinterpret_cast<cudaStream_t>(res.gcomp) : res.comp;
        side = part ? reinterpret_cast<cudaStream_t>(res.gside) : res.side;
        if (cublasSetStream(res.blas, comp) != CUBLAS_STATUS_SUCCESS)
            return fail(CC_ERR_CUDA, "cublasSetStream failed");
        cudaError_t e = cudaEventRecord(res.start, comp);
        if (e != cudaSuccess) return fail_cuda(e, "start event");
        int st = CC_OK;
        switch (which) {
            case 0:  // backward alone
                st = backward(false);
                break;
            case 1:  // all buckets alone, on the compute stream
                st = buckets(comp, false, 0);
                break;
            case 2: {  // overlapped: ready-driven buckets on the side stream
                if ((e = cudaStreamWaitEvent(side, res.start, 0)) != cudaSuccess)
                    return fail_cuda(e, "side wait");
                if ((st = backward(true)) != CC_OK) return st;
                if ((st = buckets(side, true, part ? 0 : cfg.max_ctas)) != CC_OK) return st;
                if ((e = cudaEventRecord(res.side_done, side)) != cudaSuccess)
                    return fail_cuda(e, "side done event");
                if ((e = cudaStreamWaitEvent(comp, res.side_done, 0)) != cudaSuccess)
                    return fail_cuda(e, "join wait");
                break;
            }
            case 3:  // naive synchronous: backward, then every bucket
                if ((st = backward(false)) != CC_OK) return st;
                st = buckets(comp, false, 0);
                break;
        }
        if (st != CC_OK) return st;
        if ((e = cudaEventRecord(res.stop, comp)) != cudaSuccess) return fail_cuda(e, "stop event");
        if ((e = cudaEventSynchronize(res.stop)) != cudaSuccess) return fail_cuda(e, "arm sync");
        if ((e = cudaEventElapsedTime(ms, res.start, res.stop)) != cudaSuccess)
            return fail_cuda(e, "elapsed time");
        return CC_OK;
    }

    int median(int which, float *out) {
        float ms = 0.0f;
        for (int i = 0; i < cfg.warmup; ++i) {
            const int st = arm(which, &ms);
            if (st != CC_OK) return st;
        }
        std::vector<float> t(cfg.iters);
        for (int i = 0; i < cfg.iters; ++i) {
            const int st = arm(which, &t[i]);
            if (st != CC_OK) return st;
        }
        std::sort(t.begin(), t.end());
        *out = (cfg.iters % 2) ? t[cfg.iters / 2]
                               : 0.5f * (t[cfg.iters / 2 - 1] + t[cfg.iters / 2]);
        return CC_OK;
    }
};

}  // namespace
}  // namespace ccdp

using namespace ccdp;

extern "C" int cc_overlap_bench(const cc_overlap_cfg *cfg, cc_overlap_result *out) {
    if (!cfg || !out) return fail(CC_ERR_INVALID, "cfg/out is NULL");
    const cc_overlap_cfg &c = *cfg;
    if (c.num_layers < 1 || c.gemms_per_layer < 0 || c.gemm_m < 1 || c.gemm_n < 1 ||
        c.gemm_k < 1)
        return fail(CC_ERR_INVALID, "proxy backward shape must be positive");
    if (c.iters < 1 || c.iters > 1000 || c.warmup < 0 || c.warmup > 1000)
        return fail(CC_ERR_INVALID, "iters=%d must be in 1..1000, warmup in 0..1000", c.iters);
    if (c.max_ctas < 0) return fail(CC_ERR_INVALID, "max_ctas=%d must be >= 0", c.max_ctas);
    if (c.stream_priority < 0 || c.stream_priority > 2)
        return fail(CC_ERR_INVALID, "stream_priority=%d must be 0, 1 or 2", c.stream_priority);
    if (c.comm_sms < 0) return fail(CC_ERR_INVALID, "comm_sms=%d must be >= 0", c.comm_sms);
    if (c.gemm_algo < 0) return fail(CC_ERR_INVALID, "gemm_algo=%d must be >= 0", c.gemm_algo);
    if (c.budget_buckets < 0)
        return fail(CC_ERR_INVALID, "budget_buckets=%d must be >= 0", c.budget_buckets);
    if (c.arith_flags & ~(CC_ARITH_FAST | CC_ENGINE_BULK_COPY))
        return fail(CC_ERR_INVALID, "arith_flags=%#x has unknown bits", c.arith_flags);
    if (c.num_buckets < 1 || !c.bucket_begin || !c.bucket_end || !c.bucket_ready_layer)
        return fail(CC_ERR_INVALID, "need at least one bucket");
    for (int b = 0; b < c.num_buckets; ++b) {
        if (c.bucket_begin[b] % CC_PAD_ELEMS != 0)
            return fail(CC_ERR_MISALIGNED, "bucket %d begins at %zu", b, c.bucket_begin[b]);
        if (c.bucket_begin[b] >= c.bucket_end[b] || c.bucket_end[b] > c.n)
            return fail(CC_ERR_INVALID, "bucket %d range [%zu, %zu) invalid for n=%zu", b,
                        c.bucket_begin[b], c.bucket_end[b], c.n);
        if (c.bucket_ready_layer[b] < 0 || c.bucket_ready_layer[b] >= c.num_layers)
            return fail(CC_ERR_INVALID, "bucket %d ready layer %d out of range", b,
                        c.bucket_ready_layer[b]);
    }
    AdamScalars sc;
    int st = make_scalars(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay, c.step,
                          c.grad_scale, &sc);
    if (st != CC_OK) return st;
    if (c.n == 0) return fail(CC_ERR_INVALID, "n must be > 0");
    Slabs slabs;
    st = validate_slabs(c.grads, c.acc, c.master, c.m, c.v, c.params_out, c.n, c.R,
                        c.acc != nullptr, &slabs);
    if (st != CC_OK) return st;
    slabs.fast = (c.arith_flags & CC_ARITH_FAST) != 0;
    slabs.bulk_copy = (c.arith_flags & CC_ENGINE_BULK_COPY) != 0;
    if (c.gemms_per_layer > 0) {
        if (!c.gemm_a || !c.gemm_b || !c.gemm_c)
            return fail(CC_ERR_INVALID, "GEMM operand buffers are NULL");
        const size_t M = c.gemm_m, N = c.gemm_n, K = c.gemm_k;
        if ((st = check_device_range(c.gemm_a, 2 * M * K, "gemm_a")) != CC_OK) return st;
        if ((st = check_device_range(c.gemm_b, 2 * K * N, "gemm_b")) != CC_OK) return st;
        if ((st = check_device_range(c.gemm_c, 2 * M * N, "gemm_c")) != CC_OK) return st;
    }

    Resources res;
    cudaError_t e;
    int lo = 0, hi = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess)
        return fail_cuda(e, "priority range");
    // Larger numbers are lower priorities: lo is the default, hi the top.
    if ((e = cudaStreamCreateWithPriority(&res.comp, cudaStreamNonBlocking,
                                          c.stream_priority == 2 ? hi : lo)) != cudaSuccess)
        return fail_cuda(e, "compute stream");
    if ((e = cudaStreamCreateWithPriority(&res.side, cudaStreamNonBlocking,
                                          c.stream_priority == 1 ? hi : lo)) != cudaSuccess)
        return fail_cuda(e, "side stream");
    if ((e = cudaEventCreate(&res.start)) != cudaSuccess ||
        (e = cudaEventCreate(&res.stop)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&res.side_done, cudaEventDisableTiming)) != cudaSuccess)
        return fail_cuda(e, "event create");
    res.layer.assign(c.num_layers, nullptr);
    for (int l = 0; l < c.num_layers; ++l)
        if ((e = cudaEventCreateWithFlags(&res.layer[l], cudaEventDisableTiming)) != cudaSuccess)
            return fail_cuda(e, "layer event create");
    if (cublasCreate(&res.blas) != CUBLAS_STATUS_SUCCESS)
        return fail(CC_ERR_CUDA, "cublasCreate failed");
    if (c.gemm_algo > 0 && (st = pick_lt_algo(c, res)) != CC_OK) return st;
    if (c.comm_sms > 0 &&
        (st = make_partition(c.comm_sms, c.stream_priority == 2 ? hi : lo,
                             c.stream_priority == 1 ? hi : lo, res)) != CC_OK)
        return st;

    Bench bench{c, slabs, sc, res};
    cc_overlap_result r{};
    if ((st = bench.median(0, &r.t_bwd_ms)) != CC_OK) return st;
    if ((st = bench.median(1, &r.t_comm_ms)) != CC_OK) return st;
    if ((st = bench.median(2, &r.t_step_overlap_ms)) != CC_OK) return st;
    if ((st = bench.median(3, &r.t_step_seq_ms)) != CC_OK) return st;
    r.gemm_algos = res.algos;
    r.exposed_ms = r.t_step_overlap_ms - r.t_bwd_ms;
    r.exposed_bound_ms = std::max(0.0f, r.t_comm_ms - r.t_bwd_ms);
    // The step-time equation solved for the hidden part: T_overlap =
    // T_bwd + T_comm - T_step, as a fraction of the most that could hide.
    r.t_overlap_ms = r.t_bwd_ms + r.t_comm_ms - r.t_step_overlap_ms;
    const float hideable = std::min(r.t_comm_ms, r.t_bwd_ms);
    r.overlap_eff = hideable > 0.0f ? r.t_overlap_ms / hideable : 0.0f;
    r.num_buckets = c.num_buckets;
    r.comm_sms = res.comm_sms;
    r.compute_sms = res.compute_sms;
    *out = r;
    return CC_OK;
}

// ---------------------------------------------------------------------------
// Bucket-size tuning: the overlap bench over a list of bucket caps
// ---------------------------------------------------------------------------

namespace {

// Bucket caps tried when the caller gives none: the range that bucket-sizing
// guidance for DDP spans (25 MB to a few hundred), and two smaller caps.
constexpr size_t kDefaultCaps[] = {size_t(1) << 20, size_t(4) << 20, size_t(25) << 20,
                                   size_t(100) << 20, size_t(500) << 20};

// One candidate's launch list: the planner's buckets (or one rank's shard of
// each, empty shards dropped) and the layer after which each is ready.
struct CandidatePlan {
    std::vector<size_t> begin, end;
    std::vector<int> ready;
};

int plan_candidate(const cc_tune_cfg &t, size_t cap, CandidatePlan *out) {
    const int T = t.num_tensors;
    std::vector<size_t> offsets(T);
    int nb = 0;
    size_t n_padded = 0;
    int st = cc_plan_buckets(t.numel, T, cap, offsets.data(), nullptr, nullptr, 0, &nb,
                             &n_padded);
    if (st != CC_OK && st != CC_ERR_CAPACITY) return st;
    if (n_padded != t.overlap.n)
        return fail(CC_ERR_INVALID,
                    "the tensors' slab has %zu elements, the overlap config's n is %zu",
                    n_padded, t.overlap.n);
    std::vector<size_t> bb(nb), be(nb);
    if ((st = cc_plan_buckets(t.numel, T, cap, offsets.data(), bb.data(), be.data(), nb, &nb,
                              nullptr)) != CC_OK)
        return st;
    std::vector<int> ready(nb);
    if ((st = cc_bucket_ready_layers(t.numel, t.layer_of, offsets.data(), T, bb.data(),
                                     be.data(), nb, ready.data())) != CC_OK)
        return st;
    out->begin.clear();
    out->end.clear();
    out->ready.clear();
    if (t.rank < 0) {
        out->begin = bb;
        out->end = be;
        out->ready = ready;
        return CC_OK;
    }
    const int R = t.overlap.R;
    std::vector<size_t> sb(static_cast<size_t>(nb) * R), se(sb.size()), so(sb.size());
    std::vector<size_t> elems(R);
    if ((st = cc_shard_plan(bb.data(), be.data(), nb, R, sb.data(), se.data(), so.data(),
                            elems.data())) != CC_OK)
        return st;
    for (int b = 0; b < nb; ++b) {
        const size_t lo = sb[static_cast<size_t>(b) * R + t.rank];
        const size_t hi = se[static_cast<size_t>(b) * R + t.rank];
        if (hi > lo) {
            out->begin.push_back(lo);
            out->end.push_back(hi);
            out->ready.push_back(ready[b]);
        }
    }
    return CC_OK;
}

}  // namespace

extern "C" int cc_tune_bucket_bytes(const cc_tune_cfg *cfg, cc_overlap_result *results,
                                    cc_tune_result *out) {
    TraceRange call("cc_tune_bucket_bytes", 0);
    if (!cfg || !out) return fail(CC_ERR_INVALID, "cfg/out is NULL");
    const cc_tune_cfg &t = *cfg;
    if (t.num_tensors < 1 || !t.numel || !t.layer_of)
        return fail(CC_ERR_INVALID, "need at least one tensor with numel and layer_of");
    const size_t *caps = t.candidates ? t.candidates : kDefaultCaps;
    const int count = t.candidates ? t.num_candidates
                                   : static_cast<int>(sizeof(kDefaultCaps) / sizeof(size_t));
    if (count < 1 || count > CC_TUNE_MAX_CANDIDATES)
        return fail(CC_ERR_INVALID, "num_candidates=%d must be in 1..%d", count,
                    CC_TUNE_MAX_CANDIDATES);
    if (!results) return fail(CC_ERR_INVALID, "results is NULL");
    if (t.overlap.R < 1 || t.overlap.R > CC_MAX_R)
        return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", t.overlap.R, CC_MAX_R);
    if (t.rank < -1 || t.rank >= t.overlap.R)
        return fail(CC_ERR_INVALID, "rank=%d must be -1 or in 0..R-1", t.rank);
    // Every candidate is planned, and its plan checked, before anything runs.
    std::vector<CandidatePlan> plans(count);
    int st;
    for (int i = 0; i < count; ++i) {
        if ((st = plan_candidate(t, caps[i], &plans[i])) != CC_OK) return st;
        if (plans[i].begin.empty())
            return fail(CC_ERR_INVALID, "candidate %d (%zu bytes) gives rank %d no elements", i,
                        caps[i], t.rank);
        for (int r : plans[i].ready)
            if (r < 0 || r >= t.overlap.num_layers)
                return fail(CC_ERR_INVALID,
                            "candidate %d: a bucket is ready after layer %d, the proxy "
                            "backward has %d", i, r, t.overlap.num_layers);
    }
    int best = -1;
    for (int i = 0; i < count; ++i) {
        cc_overlap_cfg c = t.overlap;
        c.bucket_begin = plans[i].begin.data();
        c.bucket_end = plans[i].end.data();
        c.bucket_ready_layer = plans[i].ready.data();
        c.num_buckets = static_cast<int>(plans[i].begin.size());
        if ((st = cc_overlap_bench(&c, &results[i])) != CC_OK) return st;
        if (best < 0 || results[i].t_step_overlap_ms < results[best].t_step_overlap_ms)
            best = i;
    }
    out->best = best;
    out->best_bucket_bytes = caps[best];
    out->num_candidates = count;
    return CC_OK;
}
