/*
 * cc_dp.h -- C ABI of the GB300 fused data-parallel step.
 *
 * One pass over R emulated data-parallel replicas that does, per element:
 *   reduce   the R bf16 gradient replicas, summed in fixed order r = 0..R-1
 *            in fp32 (stands in for the ReduceScatter),
 *   update   one AdamW step in fp32 on the fp32 master weights and moments,
 *   gather   the bf16-rounded parameters stored to all R replica slabs
 *            (stands in for the AllGather),
 * launched bucket by bucket in reverse layer order.
 *
 * Sources.  "LIT-735: Breaking the Computation and Communication Abstraction
 * Barrier in Distributed Machine Learning Workloads" (CoCoNet), Key
 * takeaways: the data-parallel result is a fused ReduceScatter-optimizer-
 * AllGather, measured on BERT with the Adam optimizer.  "Communication Optimization ›
 * Communication Overlap": DDP groups parameters into fixed-size buckets
 * (default 25 MB), launches each bucket as soon as its gradients are ready on
 * a separate stream, last layer first; the step-time equation T_step ~
 * T_fwd + T_bwd + max(0, T_comm - T_overlap).  "Overlapping Communication and
 * Computation": with gradient accumulation, k-1 micro-steps only accumulate
 * locally and one step in k carries the whole reduction.
 *
 * Arithmetic (each operation a separately rounded IEEE binary32 op):
 *   s   = g[0] + g[1] + ... + g[R-1]          left to right, from g[0]
 *         (with accumulators: s = (acc[0]+g[0]) + (acc[1]+g[1]) + ...)
 *   g^  = s * fl(1/grad_scale)
 *   m'  = beta1*m + fl(1-beta1)*g^
 *   v'  = beta2*v + fl(1-beta2)*(g^*g^)
 *   p'  = p*fl(1 - lr*wd) - lr*((m'/bc1) / (sqrt(v'/bc2) + eps))
 *         with bcX = (float)(1 - betaX^step) computed in double
 *   out[r] = bf16 round-to-nearest-even of p', for every r
 * NaN and Inf propagate; no step is skipped.
 *
 * Conventions shared by every entry point:
 *  - Device pointers are caller-owned device memory (e.g. from torch).  The
 *    library never frees them.  Host pointer arrays (grads[], params_out[],
 *    acc[]) are read during the call only.
 *  - Every slab base must be 16-byte aligned (CC_ERR_MISALIGNED otherwise).
 *  - Each device range [ptr, ptr + bytes) must lie inside one device
 *    allocation; a range that does not is rejected with CC_ERR_INVALID
 *    before any launch.
 *  - Replica slabs (grads[r], params_out[r]) may instead live in page-locked
 *    host memory allocated or registered with CUDA and mapped at the same
 *    address (any pinned allocation under unified addressing).  The kernels
 *    then read and write them directly over the host link (NVLink-C2C on
 *    GB300), with no staging copy; the range must lie inside one such
 *    allocation.  Pageable host memory is rejected (CC_ERR_INVALID).
 *    master, m, v, accumulators and workspaces must be device memory.
 *  - Written ranges must not overlap one another nor any read range
 *    (CC_ERR_ALIAS); master, m and v are updated in place.  Read-only
 *    ranges (gradients, accumulators) may alias each other.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work and never synchronise.  The returned status covers host
 *    validation and launch errors; a fault inside a kernel surfaces at the
 *    caller's next synchronisation.
 *  - On any error nothing has been launched by that call, except
 *    CC_ERR_CUDA from a launch, which may follow earlier buckets' launches.
 *  - cc_last_error() gives a one-line reason for the last failing call on
 *    the calling thread.
 *  - Sizes are in elements unless the name says bytes.  "MB" in bucket sizes
 *    is MiB (2^20 bytes) of bf16 gradient per replica.
 */
#ifndef CC_DP_H
#define CC_DP_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of this ABI are exported; everything else in the library is
 * hidden. */
#if defined(__GNUC__)
#define CC_API __attribute__((visibility("default")))
#else
#define CC_API
#endif

/* Largest number of emulated replicas one call handles. */
#define CC_MAX_R 16
/* Every tensor span in a planned slab is padded to this many elements
 * (16 bytes of bf16), so every bucket starts on a 16-byte boundary. */
#define CC_PAD_ELEMS 8

typedef enum cc_status {
    CC_OK = 0,
    CC_ERR_INVALID = -1,      /* bad argument (pointer, size, hyper-parameter) */
    CC_ERR_ALIAS = -2,        /* a written range overlaps another range */
    CC_ERR_MISALIGNED = -3,   /* a slab base (or bucket start) is not 16-byte aligned */
    CC_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed */
    CC_ERR_UNSUPPORTED = -5,  /* no usable device, or not an sm_103 device */
    CC_ERR_CAPACITY = -6      /* an output array is too small; count reported */
} cc_status;

/* Name of a status code ("CC_OK", ...).  Never NULL. */
CC_API const char *cc_status_string(int status);

/* One-line reason for the last non-OK status returned on this thread. */
CC_API const char *cc_last_error(void);

/*
 * cc_fused_dp_step -- reduce R gradient replicas, take one AdamW step and
 * redistribute the parameters, bucket by bucket (CoCoNet's fused
 * ReduceScatter-Adam-AllGather, Key takeaways of LIT-735; DDP bucketing,
 * Communication Overlap).
 *
 *   grads[R]       bf16[n] each, read.  Replica r's gradient slab.
 *   master, m, v   fp32[n], read and written in place: master weights and
 *                  the two Adam moments.
 *   params_out[R]  bf16[n] each, written: every replica's parameter slab.
 *   n              elements per slab (0 is a no-op returning CC_OK; the
 *                  pointers are then not examined).
 *   R              replicas, 1..CC_MAX_R.
 *   bucket_bytes   bf16 gradient bytes per bucket and replica; [0, n) is
 *                  cut into consecutive buckets of floor(bucket_bytes/16)*8
 *                  elements (at least 8), launched in slab order, one kernel
 *                  launch per bucket.  0 = one bucket.  Slabs laid out by
 *                  cc_plan_buckets hold the last layer first, so slab order
 *                  is reverse layer order.  Values never depend on the cut.
 *   lr >= 0, 0 <= beta1 < 1, 0 <= beta2 < 1, eps >= 0, weight_decay >= 0:
 *                  finite AdamW hyper-parameters (decoupled decay).
 *   step >= 1      the step number t in the bias corrections.
 *   grad_scale     finite, > 0: the loss scale the gradients carry.
 *   accum_k        must be 1 here; accumulated steps (k > 1) need the
 *                  accumulators of cc_fused_dp_step_accum.
 *   stream         cudaStream_t.
 *
 * Returns CC_OK or a negative cc_status.  Allocates nothing.
 */
CC_API int cc_fused_dp_step(const void *const *grads, float *master, float *m,
                     float *v, void *const *params_out, size_t n, int R,
                     size_t bucket_bytes, float lr, float beta1, float beta2,
                     float eps, float weight_decay, int step, float grad_scale,
                     int accum_k, void *stream);

/*
 * cc_accumulate_local -- one of the k-1 local micro-steps of gradient
 * accumulation ("Overlapping Communication and Computation", paragraph on
 * accumulation): acc[r] = g[r] (first != 0) or acc[r] + g[r], elementwise in
 * fp32, for every replica; no value crosses replicas.
 *
 *   grads[R]  bf16[n] each, read.     acc[R]  fp32[n] each, written.
 *   n, R, stream as above.            first   nonzero on micro-step 1.
 */
CC_API int cc_accumulate_local(const void *const *grads, float *const *acc, size_t n,
                        int R, int first, void *stream);

/*
 * cc_fused_dp_step_accum -- the reducing k-th step of gradient accumulation:
 * as cc_fused_dp_step, but each replica's local total acc[r] + g[r] is formed
 * first and those totals are summed across replicas in order r = 0..R-1.
 *
 *   acc[R]    fp32[n] each, read (not modified): replica r's sum of micro-
 *             steps 1..k-1 from cc_accumulate_local.  May be NULL only
 *             when accum_k == 1 (then identical to cc_fused_dp_step).
 *   accum_k   >= 1, the number of micro-steps in this optimizer step.
 */
CC_API int cc_fused_dp_step_accum(const void *const *grads, const float *const *acc,
                           float *master, float *m, float *v,
                           void *const *params_out, size_t n, int R,
                           size_t bucket_bytes, float lr, float beta1,
                           float beta2, float eps, float weight_decay,
                           int step, float grad_scale, int accum_k,
                           void *stream);

/*
 * cc_fused_dp_bucket -- the fused step on one element range [begin, end) of
 * the slabs, as one kernel launch: the unit a scheduler launches when a
 * bucket's gradients become ready (DDP bucketing, Communication Overlap).
 * Slab pointers and n describe the whole slabs, as for cc_fused_dp_step_accum
 * (acc may be NULL).  begin must be a multiple of CC_PAD_ELEMS (else
 * CC_ERR_MISALIGNED) and begin <= end <= n.
 *   max_ctas  0: the plain kernel over the whole GPU.  > 0: a CTA budget that
 *             leaves SMs to concurrent compute -- the same kernel in wide
 *             CTAs (768 threads, one per SM) on at most max_ctas SMs, each
 *             thread striding over the range with every load of its vector
 *             in flight, so that few SMs reach HBM bandwidth (about 98 GB/s
 *             per SM on GB300 when master, m and v are 32-byte aligned and
 *             move in 32-byte accesses; 78 GB/s when they are only 16-byte
 *             aligned).  cc_fused_dp_bucket_ex can select the bulk-copy
 *             engine instead.  Same values either way.
 */
CC_API int cc_fused_dp_bucket(const void *const *grads, const float *const *acc,
                       float *master, float *m, float *v,
                       void *const *params_out, size_t n, int R, size_t begin,
                       size_t end, float lr, float beta1, float beta2,
                       float eps, float weight_decay, int step,
                       float grad_scale, int max_ctas, void *stream);

/*
 * cc_fused_dp_bucket_ex -- cc_fused_dp_bucket with a choice of arithmetic.
 *   arith_flags  0: the exact step above (every operation one IEEE rounding,
 *                bit-identical to any correctly rounded evaluation).
 *                CC_ARITH_FAST: a cheaper form for launches that share the
 *                GPU with compute (fewer instructions per element, so fewer
 *                SMs stream the bucket at HBM speed).  The sum, m and v are
 *                exactly as above; the bias corrections become
 *                multiplications by fl(1/bc1), fl(1/bc2), the square root
 *                stays IEEE, and m^/(sqrt(v^) + eps) is a fast division
 *                (2 ulp).  The parameter then differs from the exact step by
 *                a few ulp of its update (well inside a relative 1e-5 of the
 *                parameter unless the update cancels it), the bf16 copies by
 *                at most one bf16 ulp.  Requires eps > 0 for that bound.
 *                CC_ENGINE_BULK_COPY (or-ed in, with max_ctas > 0): the
 *                budget runs on the TMA bulk-copy engine instead of the wide
 *                CTAs -- one persistent CTA per SM whose producer warp
 *                streams tiles into a ring of shared-memory stages with
 *                cp.async.bulk and whose consumer warps reduce, update and
 *                store them; every pipeline wait is bounded (cc_device_status
 *                reports one that ran out).  It streams about 61 GB/s per SM
 *                (the copies of one replica slice are 2 KB, and a bulk copy's
 *                throughput falls with its size).  Same values.
 *                Other bits: CC_ERR_INVALID.
 */
#define CC_ARITH_FAST 1u
#define CC_ENGINE_BULK_COPY 2u
CC_API int cc_fused_dp_bucket_ex(const void *const *grads, const float *const *acc,
                                 float *master, float *m, float *v,
                                 void *const *params_out, size_t n, int R, size_t begin,
                                 size_t end, float lr, float beta1, float beta2,
                                 float eps, float weight_decay, int step,
                                 float grad_scale, int max_ctas, unsigned arith_flags,
                                 void *stream);

/*
 * cc_fused_dp_shard -- one rank's share of the sharded step, with the
 * optimizer state sharded ("LIT-735 (CoCoNet)", Key takeaways: the fused
 * ReduceScatter-optimizer-AllGather fits larger micro-batches by sharding
 * optimizer state).  The rank owns the master weights and Adam moments of
 * the slab elements [shard_begin, shard_end) only: it reduces the R
 * replicas' gradients of that range (its ReduceScatter share), updates its
 * state shard, and writes the range's bf16 parameters to all R replica
 * slabs (its AllGather share).  The R ranks' calls over a partition of
 * [0, n) give exactly the values of one cc_fused_dp_step_accum over [0, n).
 *
 *   grads[R], params_out[R]   whole replica slabs of n bf16 elements; only
 *                  [shard_begin, shard_end) is read / written.
 *   acc[R]         NULL, or whole fp32[n] accumulator slabs (read in the
 *                  range): the reducing step of gradient accumulation.
 *   master, m, v   fp32[shard_end - shard_begin]: element i is slab element
 *                  shard_begin + i.  Read and written in place.
 *   shard_begin    a multiple of CC_PAD_ELEMS (else CC_ERR_MISALIGNED);
 *                  shard_begin <= shard_end <= n (else CC_ERR_INVALID).  An
 *                  empty shard is a no-op returning CC_OK.
 *   bucket_bytes   the shard is cut into buckets as cc_fused_dp_step cuts
 *                  [0, n), counted from shard_begin.
 *   the rest       as cc_fused_dp_step.  Allocates nothing.
 */
CC_API int cc_fused_dp_shard(const void *const *grads, const float *const *acc,
                      float *master, float *m, float *v,
                      void *const *params_out, size_t n, int R,
                      size_t shard_begin, size_t shard_end, size_t bucket_bytes,
                      float lr, float beta1, float beta2, float eps,
                      float weight_decay, int step, float grad_scale,
                      void *stream);

/*
 * cc_shard_plan -- the shards of the real multi-GPU form of the step, one
 * ReduceScatter-AdamW-AllGather per bucket ("LIT-735 (CoCoNet)", Key
 * takeaways: the fused ReduceScatter-optimizer-AllGather, which shards the
 * optimizer state; "Communication Overlap": one collective per DDP bucket).
 * Each planned bucket is cut into `world` shards in rank order; rank q
 * reduces, updates and gathers shard q of every bucket, and owns the
 * optimizer state of those shards only, packed in launch order.  Host only.
 *
 *   bucket_begin/end[num_buckets]  element ranges in launch order (from
 *                  cc_plan_buckets: each begins on a multiple of CC_PAD_ELEMS,
 *                  else CC_ERR_MISALIGNED), non-decreasing.
 *   world          ranks, >= 1.
 *   shard_begin_out, shard_end_out [num_buckets * world]: shard q of bucket
 *                  b at index b * world + q.  The bucket is cut in units of
 *                  CC_PAD_ELEMS elements: shard q holds units
 *                  [floor(u q / world), floor(u (q + 1) / world)) of its u
 *                  units (the last shard also any ragged tail), so every shard
 *                  begins 16-byte aligned and sizes differ by at most 8.
 *   state_offset_out [num_buckets * world]: where shard q of bucket b starts
 *                  in rank q's master/m/v arrays.
 *   state_elems_out [world]: elements of master/m/v rank q owns.
 */
CC_API int cc_shard_plan(const size_t *bucket_begin, const size_t *bucket_end,
                         int num_buckets, int world, size_t *shard_begin_out,
                         size_t *shard_end_out, size_t *state_offset_out,
                         size_t *state_elems_out);

/*
 * cc_fused_dp_rank_step -- one rank's compute in the real multi-GPU form,
 * between the two exchanges of one bucket ("LIT-735 (CoCoNet)", Key
 * takeaways: the optimizer fused between the ReduceScatter and the
 * AllGather).  After the ReduceScatter exchange the rank holds every
 * replica's bf16 gradient of its shard; this call sums them in replica
 * (rank) order in fp32, takes the AdamW step on the rank's own state of
 * the shard, and writes the bf16 parameters of the shard once, into the
 * rank's own parameter slab, from where the AllGather exchange sends them
 * to every rank.  Values are exactly those of cc_fused_dp_step on the same
 * elements.
 *
 *   grad_slices[R]  bf16[len] each, read: replica r's gradient of the shard,
 *                   r = 0..R-1 (R = world size; the rank's own slice may point
 *                   into its own gradient slab).  May alias each other.
 *   master, m, v    fp32[len], read and written: the rank's state of the shard.
 *   param_out       bf16[len], written: the shard's parameters.
 *   len             elements of the shard (0 is a no-op).
 *   the rest        as cc_fused_dp_step.  One kernel launch; allocates nothing.
 *   Gradient slices and param_out may be page-locked host memory, as replica
 *   slabs may elsewhere; the state must be device memory.
 * The launch is a programmatic dependent of the work before it on the
 * stream: its blocks may become resident while that kernel finishes, but
 * read and write nothing before it has completed, so back-to-back rank
 * steps (one per bucket) overlap their launch gaps.
 */
CC_API int cc_fused_dp_rank_step(const void *const *grad_slices, float *master, float *m,
                                 float *v, void *param_out, size_t len, int R, float lr,
                                 float beta1, float beta2, float eps, float weight_decay,
                                 int step, float grad_scale, void *stream);

/*
 * cc_unfused_dp_step -- the same step as cc_fused_dp_step (bit-identical
 * results) in the unfused schedule a framework runs when the collective and
 * the optimizer are separate library calls, kept for comparison ("LIT-735
 * (CoCoNet)", Key takeaways: fusing the optimizer into the ReduceScatter/
 * AllGather beats PyTorch DDP's bucketed AllReduce followed by a separate
 * optimizer step).  Per bucket: a reduce kernel writes the fp32 sum of the
 * R gradients into `workspace`, an AdamW kernel reads it back and writes
 * master/m/v and replica 0's parameters, and R-1 device copies broadcast
 * replica 0's parameters.  (6R + 30 bytes per parameter against 4R + 24.)
 *
 *   workspace        caller-owned fp32 device scratch of workspace_bytes
 *                    >= 4 * (elements of the largest bucket) bytes, 16-byte
 *                    aligned, overlapping no slab; reused by every bucket
 *                    (the calls are stream-ordered).  Too small:
 *                    CC_ERR_INVALID.
 *   other arguments  as cc_fused_dp_step (no accumulators).
 */
CC_API int cc_unfused_dp_step(const void *const *grads, float *master, float *m,
                              float *v, void *const *params_out, float *workspace,
                              size_t workspace_bytes, size_t n, int R,
                              size_t bucket_bytes, float lr, float beta1, float beta2,
                              float eps, float weight_decay, int step,
                              float grad_scale, void *stream);

/*
 * cc_unfused_dp_step_noalloc -- cc_unfused_dp_step for callers that cannot
 * allocate device memory.  (The pages have no counterpart: this is a
 * convenience of this library.)  Some callers cannot pass a workspace or
 * call cudaMalloc: code whose device memory all belongs to a framework's
 * caching allocator, hot loops where an allocation or free would stall the
 * device, and plugins handed buffers but no right to allocate.  This entry
 * point takes only the inputs and outputs; the reduced gradient of one bucket
 * goes to a fixed array of CC_NOALLOC_SCRATCH_ELEMS fp32 elements (64 MiB)
 * inside the library's own device memory, which every GPU that loads the
 * library holds until the process exits.  It allocates nothing.
 *
 *  - The largest bucket, min(n, floor(bucket_bytes/16)*8) elements (n when
 *    bucket_bytes is 0), must fit the array: floor(bucket_bytes/16)*8 <=
 *    CC_NOALLOC_SCRATCH_ELEMS, i.e. bucket_bytes < 2*CC_NOALLOC_SCRATCH_ELEMS
 *    + 16 (32 MiB + 16 bytes), or n <= CC_NOALLOC_SCRATCH_ELEMS.  A larger
 *    bucket is rejected with CC_ERR_INVALID before any launch, and the
 *    reason names whichever of n and bucket_bytes set its size.
 *  - The first call on a device (and the first after a device reset, which
 *    makes a new context) looks up the array's device address
 *    (cudaGetSymbolAddress) for that device with it current; make that
 *    first call before any stream capture begins.
 *  - Every call shares the one array, and each bucket overwrites the part
 *    it uses before reading it, so no state carries over between calls.
 *    Calls that overlap on the GPU (on different streams, or from different
 *    threads without ordering) race on the array: order them.
 *  - Arguments and results are as for cc_fused_dp_step (bit-identical).
 */
#define CC_NOALLOC_SCRATCH_ELEMS (16u * 1024u * 1024u)
CC_API int cc_unfused_dp_step_noalloc(const void *const *grads, float *master, float *m,
                                      float *v, void *const *params_out, size_t n, int R,
                                      size_t bucket_bytes, float lr, float beta1,
                                      float beta2, float eps, float weight_decay,
                                      int step, float grad_scale, void *stream);

/*
 * cc_plan_buckets -- lay tensors out in reverse layer order and cut them into
 * buckets (Communication Overlap: backward produces the last layer's
 * gradients first, buckets hold a configurable size, default 25 MB, and the
 * last layer's bucket launches first; Overlapping Communication and
 * Computation: a very large single tensor is not split).  Host only: no
 * CUDA call.
 *
 *   numel[T]          tensor sizes in forward (layer) order.
 *   bucket_bytes      cap in bf16 bytes; a bucket closes as soon as its
 *                     padded spans reach the cap; 0 = one bucket.
 *   offsets_out[T]    written: tensor t's first slab element.  Spans are
 *                     padded to CC_PAD_ELEMS; tensor T-1 is at offset 0.
 *   bucket_begin_out, bucket_end_out [capacity]: written, element ranges
 *                     in launch order.  Buckets with no elements are not
 *                     emitted (a trailing run of empty tensors).
 *   capacity          length of the two bucket arrays.  If it is too small
 *                     the call writes *num_buckets_out and returns
 *                     CC_ERR_CAPACITY (pass 0 and NULLs to query).
 *   num_buckets_out   written: number of buckets.
 *   n_padded_out      written: slab length in elements (may be NULL).
 */
CC_API int cc_plan_buckets(const size_t *numel, int num_tensors, size_t bucket_bytes,
                    size_t *offsets_out, size_t *bucket_begin_out,
                    size_t *bucket_end_out, int capacity,
                    int *num_buckets_out, size_t *n_padded_out);

/*
 * cc_bucket_ready_layers -- for each bucket, the backward layer after which
 * all its gradients exist: the lowest layer index among its non-empty
 * tensors (backward runs from the highest layer down).  Host only.
 *
 *   layer_of[T]  layer of each tensor (forward order).  Other arrays as
 *                returned by cc_plan_buckets.  ready_layer_out[num_buckets]
 *                written.
 */
CC_API int cc_bucket_ready_layers(const size_t *numel, const int *layer_of,
                           const size_t *offsets, int num_tensors,
                           const size_t *bucket_begin,
                           const size_t *bucket_end, int num_buckets,
                           int *ready_layer_out);

/*
 * cc_overlap_bench -- measure how much of the bucketed fused step hides
 * behind a proxy backward pass ("Communication Overlap": step-time equation;
 * DDP launches each bucket on a separate stream once ready; "naive
 * synchronous data-parallel" runs backward, then the reduction, then the
 * optimizer, in strict phases).
 *
 * The proxy backward runs num_layers x gemms_per_layer bf16 GEMMs
 * (C[M,N] = A[M,K] B[K,N], fp32 accumulation, cuBLAS) on a compute stream,
 * layer num_layers-1 first, and records an event after each layer.  Bucket b
 * launches on a side stream once the event of bucket_ready_layer[b] has
 * fired.  Four arms are timed with CUDA events, each the median of `iters`
 * runs after `warmup` runs:
 *   t_bwd_ms          the GEMMs alone;
 *   t_comm_ms         all buckets alone, back to back;
 *   t_step_overlap_ms GEMMs and ready-driven buckets together;
 *   t_step_seq_ms     GEMMs, then all buckets, on one stream.
 * exposed_ms = t_step_overlap_ms - t_bwd_ms; exposed_bound_ms =
 * max(0, t_comm_ms - t_bwd_ms), the least any schedule can expose.
 * t_overlap_ms = t_bwd_ms + t_comm_ms - t_step_overlap_ms is the time the
 * step-time equation says was hidden (negative when the overlapped arm is
 * slower than the two parts back to back), and overlap_eff = t_overlap_ms /
 * min(t_comm_ms, t_bwd_ms) the fraction of what could hide that did.
 *
 * The slabs are stepped for real (master/m/v change on every run).  The GEMM
 * operands are caller-owned bf16 device buffers: A holds M*K, B K*N and C
 * M*N elements.  The call synchronises its own streams, creates and destroys
 * its streams, events and cuBLAS handle, and allocates no device memory of
 * its own beyond what cuBLAS takes for its handle.
 */
typedef struct cc_overlap_cfg {
    const void *const *grads;      /* [R] bf16[n] */
    const float *const *acc;       /* [R] fp32[n] or NULL */
    float *master, *m, *v;         /* fp32[n] */
    void *const *params_out;       /* [R] bf16[n] */
    size_t n;
    int R;
    const size_t *bucket_begin;    /* [num_buckets], launch order */
    const size_t *bucket_end;
    const int *bucket_ready_layer; /* [num_buckets], in [0, num_layers) */
    int num_buckets;
    float lr, beta1, beta2, eps, weight_decay;
    int step;
    float grad_scale;
    int num_layers, gemms_per_layer;
    int gemm_m, gemm_n, gemm_k;
    void *gemm_a, *gemm_b, *gemm_c;  /* bf16 device buffers */
    int warmup, iters;             /* iters in 1..1000 */
    int max_ctas;                  /* bucket kernels' CTA cap while overlapped; 0 = full */
    int stream_priority;           /* 0: equal; 1: side stream high; 2: compute stream high */
    int comm_sms;                  /* > 0: overlapped arm on a spatial partition (green
                                      contexts): buckets on comm_sms SMs (rounded up to the
                                      driver's granularity), GEMMs on the rest; 0: none */
    int budget_buckets;            /* > 0: in the overlapped arm only the first
                                      budget_buckets buckets take the max_ctas budget (the
                                      SMs the GEMMs leave free); the later ones wait for
                                      the whole backward and run on the whole GPU.
                                      0: every bucket takes max_ctas */
    int gemm_algo;                 /* 0: the proxy GEMMs through cublasGemmEx (cuBLAS's
                                      choice); k > 0: through cuBLASLt with the k-th
                                      candidate of its heuristic (no workspace) */
    unsigned arith_flags;          /* the buckets' arithmetic and budget engine: 0
                                      exact, or CC_ARITH_FAST and/or
                                      CC_ENGINE_BULK_COPY (see
                                      cc_fused_dp_bucket_ex) */
} cc_overlap_cfg;

typedef struct cc_overlap_result {
    float t_bwd_ms, t_comm_ms, t_step_overlap_ms, t_step_seq_ms;
    float exposed_ms, exposed_bound_ms;
    int num_buckets;
    int comm_sms, compute_sms;     /* the partition's SM counts (0 without one) */
    int gemm_algos;                /* cuBLASLt candidates offered (0 with gemm_algo 0) */
    float t_overlap_ms, overlap_eff;
} cc_overlap_result;

CC_API int cc_overlap_bench(const cc_overlap_cfg *cfg, cc_overlap_result *out);

/*
 * cc_tune_bucket_bytes -- choose the DDP bucket size by measurement
 * ("LIT-735 (CoCoNet)", Key takeaways: the schedule is autotuned;
 * "Communication Overlap", bucket sizing: caps of 25 to 500 MB work well,
 * larger models favouring larger buckets, so the best cap is measured, not
 * fixed).  For each candidate cap the tensors are planned with
 * cc_plan_buckets and cc_bucket_ready_layers (and, for one rank, cut with
 * cc_shard_plan), and cc_overlap_bench times that launch list; the
 * candidate whose overlapped step (t_step_overlap_ms) is shortest wins,
 * the first listed on a tie.
 *
 *   overlap        every cc_overlap_cfg field but the bucket arrays and
 *                  num_buckets, which are ignored: the slabs (n must be the
 *                  planner's slab length for numel), hyperparameters, proxy
 *                  backward and arm settings.  The slabs are stepped for real
 *                  by every candidate's runs.
 *   numel, layer_of [num_tensors]  the slab's tensors in forward order and
 *                  the backward layer of each (in [0, overlap.num_layers)
 *                  for every bucket's ready layer, else CC_ERR_INVALID).
 *   candidates     [num_candidates] caps in bf16 bytes (0: one bucket), or
 *                  NULL for 1, 4, 25, 100 and 500 MiB (num_candidates is
 *                  then ignored).  1..CC_TUNE_MAX_CANDIDATES.
 *   rank           -1: every bucket whole (the emulated R replicas);
 *                  0..R-1: only that rank's shard of each bucket (the
 *                  per-rank work of the multi-GPU form); a candidate that
 *                  leaves the rank no elements is CC_ERR_INVALID.
 *   results        [count] written: each candidate's cc_overlap_result.
 *   out            written: the winner's index and cap, and the count.
 * Every candidate is planned and checked on the host before the first
 * measurement; an error from a measurement stops the call there.
 */
#define CC_TUNE_MAX_CANDIDATES 64

typedef struct cc_tune_cfg {
    cc_overlap_cfg overlap;
    const size_t *numel;
    const int *layer_of;
    int num_tensors;
    const size_t *candidates;
    int num_candidates;
    int rank;
} cc_tune_cfg;

typedef struct cc_tune_result {
    int best;                      /* index into the candidates */
    size_t best_bucket_bytes;
    int num_candidates;            /* results written */
} cc_tune_result;

CC_API int cc_tune_bucket_bytes(const cc_tune_cfg *cfg, cc_overlap_result *results,
                                cc_tune_result *out);

/*
 * cc_tp_allreduce -- the AllReduce of a tensor-parallel row-parallel layer,
 * for R emulated ranks ("LIT-735 (CoCoNet)", Key takeaways: the
 * model-parallel MatMul and the AllReduce that follows it).  Every rank's
 * output becomes the bf16 rounding of the fp32 sum of the R partial products
 * in rank order r = 0..R-1 (one rounding).
 *
 *   partials[R]  fp32[n] each, read: rank r's partial product.
 *   out[R]       bf16[n] each, written: every rank's copy of the sum.
 *   n, R, stream as for cc_fused_dp_step.  Device memory only.
 */
CC_API int cc_tp_allreduce(const float *const *partials, void *const *out, size_t n,
                           int R, void *stream);

/*
 * cc_tp_overlap_bench -- the MatMul-then-AllReduce of a row-parallel layer,
 * sequential and overlapped in chunks of rows (LIT-735, Key takeaways:
 * overlapping the two in chunks hides most of the MatMul).  Rank r holds
 * x[r] (bf16, m x k/R, row-major) and w[r] (bf16, k/R x n, row-major) and
 * computes partials[r] = x[r] w[r] (fp32, m x n, cuBLAS with fp32
 * accumulation); out[r] receives the AllReduce (cc_tp_allreduce).  The rows
 * are cut into `chunks` equal chunks; in the overlapped arm each chunk's
 * AllReduce runs on a side stream as soon as that chunk's R GEMMs finish.
 * Four arms, each the median of `iters` runs after `warmup`: the GEMMs
 * alone, the AllReduce alone, GEMMs then AllReduce on one stream, and the
 * chunked overlap.  Requires k % R == 0, m % chunks == 0, (m/chunks)*n and
 * k/R multiples of 8.  When the R shards of x, w and partials lie at equal
 * strides (one buffer cut into R slabs), a chunk's R products run as one
 * strided-batched GEMM.  Buffers are caller-owned device memory; the call
 * synchronises its own streams and allocates nothing beyond cuBLAS's handle.
 */
typedef struct cc_tp_cfg {
    int R, m, n, k, chunks;
    const void *const *x;          /* [R] bf16 m x k/R */
    const void *const *w;          /* [R] bf16 k/R x n */
    float *const *partials;        /* [R] fp32 m x n */
    void *const *out;              /* [R] bf16 m x n */
    int warmup, iters;
    int stream_priority;           /* 0 equal, 1 side stream high, 2 compute high */
} cc_tp_cfg;

typedef struct cc_tp_result {
    float t_gemm_ms, t_allreduce_ms, t_sequential_ms, t_overlap_ms;
} cc_tp_result;

CC_API int cc_tp_overlap_bench(const cc_tp_cfg *cfg, cc_tp_result *out);

/*
 * cc_tp_matmul_allreduce -- the MatMul of a row-parallel layer and the
 * AllReduce that follows it, for R emulated tensor-parallel ranks, in one
 * kernel ("LIT-735 (CoCoNet)", Key takeaways: the model-parallel MatMul and
 * its AllReduce, which CoCoNet overlaps in chunks; here they are fused so
 * that no partial product reaches HBM).  Rank r computes Y_r = X_r W_r^T on
 * the tensor cores (tcgen05, bf16 inputs, fp32 accumulation); every rank's
 * output is the bf16 rounding (nearest-even, once) of the fp32 sum of the R
 * partial products in rank order r = 0..R-1 -- exactly cc_tp_allreduce
 * applied to those partial products.
 *
 *   x[R]         bf16, m x k/R each, row-major: rank r's activations.
 *   w[R]         bf16, n x k/R each, row-major (k/R contiguous: a linear
 *                layer's weight layout): rank r's weight shard.
 *   out[R]       bf16, m x n each, row-major, written: every rank's copy of
 *                the reduced output.
 *   partials     NULL, or [R] fp32 m x n each, written: each rank's partial
 *                product as the tensor cores accumulated it (for checking
 *                the reduction; costs 4R bytes per output element).
 *   m, n, k, R   k % R == 0; m % 128 == 0, n a multiple of 128 or 192, and
 *                (k/R) % 64 == 0 (the kernel's tiles), else CC_ERR_INVALID.
 *                R in 1..CC_MAX_R.
 *   stream       cudaStream_t.
 * Buffers are device memory, 16-byte aligned; written buffers overlap
 * nothing.  Allocates nothing.  A pipeline wait that runs out (each is
 * bounded to two seconds) is reported by cc_device_status (codes 8, 16, 32,
 * 64) instead of hanging.
 */
CC_API int cc_tp_matmul_allreduce(const void *const *x, const void *const *w,
                                  void *const *out, float *const *partials, int m, int n,
                                  int k, int R, void *stream);

/*
 * cc_tp_matmul_allreduce_ex -- cc_tp_matmul_allreduce with a caller
 * workspace and a CTA budget.  Same results, bit for bit, whatever the
 * workspace and budget.
 *
 * The kernel runs persistent CTA pairs, each taking one pair of 128-row
 * output tiles ("group") through all R ranks.  When a few groups are left
 * for a last wave (at most pairs / R of them), a workspace lets the kernel
 * split them into their R rank products, spread over the pairs, at most
 * one each: each product goes to the
 * workspace as fp32 and the pair that finishes a group's last product
 * (counted with one atomic per group half; no CTA waits for another) adds
 * the R products in rank order and writes the bf16 outputs.
 *
 *   workspace        NULL (or workspace_bytes 0): no group is split.  Else
 *                    device memory, 16-byte aligned, overlapping no other
 *                    buffer, of at least the bytes
 *                    cc_tp_matmul_allreduce_workspace gives for the same
 *                    shape and max_ctas on the same device
 *                    (CC_ERR_INVALID if smaller).  The call clears its
 *                    counters on the stream before the launch; calls that
 *                    share a workspace must be ordered (one stream).
 *   max_ctas         0: as many CTA pairs as fit the GPU at once; else at
 *                    most max_ctas CTAs (>= 2; 1 is CC_ERR_INVALID).
 * Other arguments and errors as cc_tp_matmul_allreduce.
 */
CC_API int cc_tp_matmul_allreduce_ex(const void *const *x, const void *const *w,
                                     void *const *out, float *const *partials, int m, int n,
                                     int k, int R, void *workspace, size_t workspace_bytes,
                                     int max_ctas, void *stream);

/*
 * cc_tp_matmul_allreduce_workspace -- the workspace bytes
 * cc_tp_matmul_allreduce_ex uses for this shape and max_ctas on the current
 * device: 0 when it splits nothing (R = 1, groups that fill every wave, a
 * leftover wave of more than pairs / R groups -- it is split only where
 * every CTA pair gets at most one rank product of it -- or an odd count of
 * row tiles).
 * Otherwise 256 bytes of counters per 32 split groups plus 2 x 128 x BN x R
 * fp32 products per split group (BN = 256, 192 or 128, the tile width the
 * kernel picks for n).  Shape errors as cc_tp_matmul_allreduce; max_ctas
 * as cc_tp_matmul_allreduce_ex (0, or >= 2).
 */
CC_API int cc_tp_matmul_allreduce_workspace(int m, int n, int k, int R, int max_ctas,
                                            size_t *bytes);

/*
 * cc_device_status -- the status word of the library's pipelined kernels on
 * the current device: 0, or an or of codes of pipeline waits that ran out
 * (every such wait is bounded, after which the kernel abandons its pipeline
 * and returns instead of hanging).  Bulk-copy engine (one second per wait):
 * 1 consumer, 2 producer, 4 drain of copies in flight.  Fused tensor-parallel
 * kernel (two seconds): 8 producer, 16 MMA, 32 epilogue, 64 drain.  Builds
 * with CC_DEBUG_BOUNDS=1 only: 128, an access of either kernel fell outside
 * the buffer or range its arguments describe and was skipped.  A non-zero
 * word means some launch did not finish its range.  Synchronises with the
 * device; clear != 0 resets the word.
 */
CC_API int cc_device_status(unsigned *status, int clear);

/*
 * cc_inject_launch_failure -- failure injection on the host, for testing how
 * errors propagate (no GPU fault is involved).  Arms a one-shot failure for
 * the calling thread: after `after_launches` more bucket launches by
 * cc_fused_dp_step, cc_fused_dp_step_accum, cc_unfused_dp_step or
 * cc_unfused_dp_step_noalloc, the next
 * bucket is not launched and the call returns CC_ERR_CUDA ("injected launch
 * failure ...") -- the documented partial-launch case: earlier buckets of
 * that call were enqueued, later ones were not.  -1 disarms.
 */
CC_API int cc_inject_launch_failure(int after_launches);

/*
 * cc_inject_bulk_stall -- failure injection on the GPU without a fault, for
 * testing the bulk-copy engine's bounded waits.  Arms a one-shot for the
 * calling thread: in the next bulk-engine launch it makes
 * (cc_fused_dp_bucket_ex with max_ctas > 0 and CC_ENGINE_BULK_COPY, or
 * cc_overlap_bench with a CTA budget and that flag), the producer never
 * issues tile `tile` (tiles of 1024, 512 or 256 elements, counted from the
 * launch's first element; the CTA tile % grid owns it), and that launch's
 * pipeline waits give up after timeout_us (1..1000000) instead of one
 * second.  The consumers waiting for the tile then give up (status code 1);
 * a producer that comes back to the tile's stage gives up too (code 2);
 * every copy issued still lands before the CTA exits.  The launch returns
 * with the skipped tile, and possibly later tiles of its CTA, not stepped
 * (each tile either stepped exactly or left as it was), and
 * cc_device_status reports the codes.  tile = -1 disarms.
 */
CC_API int cc_inject_bulk_stall(long long tile, unsigned timeout_us);

/*
 * cc_l2_flush -- overwrite `bytes` of the caller's device buffer `buf`
 * (16-byte aligned) so that a timed kernel that follows finds none of its
 * data in L2.  Measurement helper; not part of the step.
 */
CC_API int cc_l2_flush(void *buf, size_t bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CC_DP_H */
