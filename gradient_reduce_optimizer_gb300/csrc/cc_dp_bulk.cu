// Bulk-copy engine of the fused data-parallel step for sm_103a: the same
// per-element arithmetic as fused_step_kernel (cc_dp_device.cuh), organised
// to stream as many bytes per SM as possible, for launches that may use only
// part of the GPU (a CTA budget that leaves SMs to concurrent compute).
//
// The plain kernel keeps about 224 bytes in flight per thread and streams
// about 57 GB/s per 256-thread CTA, so it needs most of the 152 SMs to reach
// HBM bandwidth.  Here one persistent CTA per SM runs a warp-specialised
// pipeline over tiles of T elements:
//   * warp 0 (one elected lane) is the producer: for each tile it issues R+3
//     one-dimensional bulk copies (cp.async.bulk, the TMA engine) of the
//     gradient slices and the master/m/v slices into a stage of a ring of S
//     shared-memory stages, all signalling the stage's "full" mbarrier with
//     the byte count; up to S tiles (about 180 KB at R = 8) are in flight per
//     SM, independent of how many threads wait;
//   * the other warps are consumers, in groups of 8 that take the CTA's
//     tiles in turn (two groups: even and odd tiles).  Each warp owns a
//     fixed 128-element slice of a tile (four elements per lane): once the
//     stage is full it reads its slice and reduces the R gradient slices in
//     fixed order, arrives on the stage's "empty" mbarrier -- the stage goes
//     back to the producer when all 8 warps of the group have arrived --
//     and only then applies AdamW and stores master/m/v and the R bf16
//     parameter copies (the redistribution) straight to global memory with
//     coalesced vector stores.  Warps never wait for each other, and the
//     producer refills a stage while its consumers still compute.
//
// The stage count is a multiple of the group count, so every use of a
// stage falls to the same group: a group, taking its tiles in order, never
// waits on a stage whose previous use is still in flight (the mbarrier's
// parity test would let it through a phase early).
//
// Measured on GB300 (2^25 elements, R = 8): one 8-warp consumer group
// streams about 57 GB/s per SM with the IEEE-exact arithmetic; the SM is
// then issuing about half the time and otherwise waiting for its stages,
// not on its arithmetic pipes.  Loads carry an evict-first L2 policy and
// stores are streaming (.cs): the stream is used once.
//
// Every mbarrier wait is bounded by the global timer.  A wait that runs out
// records a code in a device status word (cc_device_status in
// include/cc_dp.h), abandons the pipeline, waits (bounded again) for its own
// copies in flight and returns, so a broken pipeline reports instead of
// hanging.  Nothing here waits on another CTA or another grid.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "cc_dp_device.cuh"
#include "cc_dp_internal.h"

namespace ccdp {

// Codes or-ed into the status word by a bulk-engine wait that ran out.
__device__ unsigned int g_bulk_status = 0;

namespace {

using namespace dev;

#ifndef CC_DP_BULK_GROUPS
#define CC_DP_BULK_GROUPS 2    // consumer groups of 8 warps, taking tiles in turn
#endif

constexpr int kConsumerWarps = 8;              // per group: one tile's consumers
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kGroups = CC_DP_BULK_GROUPS;
constexpr int kBulkThreads = kGroups * kConsumers + 32;  // + one producer warp
constexpr int kMaxStages = 16;
constexpr int kMaxTile = 1024;                 // a group's 256 threads x 4 elements
static_assert(kMaxTile == 4 * kConsumers, "one four-element slice per consumer thread");
constexpr int kSmemBudget = 200 * 1024;        // dynamic shared memory per CTA
constexpr unsigned kStatusConsumerTimeout = 1u;
constexpr unsigned kStatusProducerTimeout = 2u;
constexpr unsigned kStatusDrainTimeout = 4u;
constexpr unsigned kStatusBounds = 128u;        // debug builds: an access outside its range

#ifndef CC_DEBUG_BOUNDS
#define CC_DEBUG_BOUNDS 0   // 1: check the computed element ranges; skip and report
#endif
constexpr bool kDebugBounds = CC_DEBUG_BOUNDS != 0;

// Debug builds: whether [off, off + len) lies inside [0, limit); if not, the
// status word says so and the access is skipped.
__device__ __forceinline__ bool debug_in_bounds(size_t off, size_t len, size_t limit) {
    if constexpr (!kDebugBounds) return true;
    if (off + len <= limit) return true;
    atomicOr(&g_bulk_status, kStatusBounds);
    return false;
}

struct BulkParams {
    const uint16_t *g[CC_MAX_R];   // bf16 slabs
    const float *acc[CC_MAX_R];    // fp32 accumulators or null
    uint16_t *out[CC_MAX_R];
    float *master, *m, *v;
    AdamScalars c;
    size_t begin;        // first element of the tiled range (multiple of 8)
    size_t tiled;        // elements covered by tiles (multiple of 8)
    size_t num_tiles;
    size_t tail_begin;   // 0..7 elements after the tiled range
    int tail_len;
    int tile;            // T, elements per tile (multiple of 8)
    int stages;          // S
    unsigned long long timeout_ns;        // bound on a pipeline wait
    unsigned long long drain_timeout_ns;  // bound on the final wait for copies issued
    size_t skip_tile;    // failure injection: a tile the producer never issues
                         // (SIZE_MAX: none)
};

// Byte offsets of one stage's slices (all multiples of 16).
struct StageLayout {
    unsigned g, acc, master, m, v, bytes;
};

__host__ __device__ inline StageLayout stage_layout(int R, bool acc, int T) {
    StageLayout L;
    L.g = 0;
    L.acc = L.g + 2u * R * T;
    L.master = L.acc + (acc ? 4u * R * T : 0u);
    L.m = L.master + 4u * T;
    L.v = L.m + 4u * T;
    L.bytes = (L.v + 4u * T + 127u) / 128u * 128u;
    return L;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}

// Wait for the phase with this parity to complete, at most timeout_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long timeout_ns) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_test(bar, parity))
        if (global_ns() - t0 > timeout_ns) return false;
    return true;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}


// Four consecutive elements of one tile, read from their stage: the fixed-
// order sum of the R gradients (plus accumulators) and master/m/v.
struct Operands4 {
    float s[4];
    float4 p4, m4, v4;
};

template <int R, bool ACC>
__device__ __forceinline__ Operands4 read_reduce4(const unsigned char *st, const StageLayout &L,
                                                  int T, int j) {
    Operands4 x;
    uint2 gq[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
        gq[r] = *reinterpret_cast<const uint2 *>(st + L.g + 2u * (r * T + j));
    float *s = x.s;
    if constexpr (ACC) {
        const float4 a = *reinterpret_cast<const float4 *>(st + L.acc + 4u * j);
        s[0] = add_bf16_lo(a.x, gq[0].x); s[1] = add_bf16_hi(a.y, gq[0].x);
        s[2] = add_bf16_lo(a.z, gq[0].y); s[3] = add_bf16_hi(a.w, gq[0].y);
    } else {
        s[0] = bf16_lo(gq[0].x); s[1] = bf16_hi(gq[0].x);
        s[2] = bf16_lo(gq[0].y); s[3] = bf16_hi(gq[0].y);
    }
#pragma unroll
    for (int r = 1; r < R; ++r) {
        if constexpr (ACC) {
            const float4 a = *reinterpret_cast<const float4 *>(st + L.acc + 4u * (r * T + j));
            s[0] = __fadd_rn(s[0], add_bf16_lo(a.x, gq[r].x));
            s[1] = __fadd_rn(s[1], add_bf16_hi(a.y, gq[r].x));
            s[2] = __fadd_rn(s[2], add_bf16_lo(a.z, gq[r].y));
            s[3] = __fadd_rn(s[3], add_bf16_hi(a.w, gq[r].y));
        } else {
            s[0] = add_bf16_lo(s[0], gq[r].x); s[1] = add_bf16_hi(s[1], gq[r].x);
            s[2] = add_bf16_lo(s[2], gq[r].y); s[3] = add_bf16_hi(s[3], gq[r].y);
        }
    }
    x.p4 = *reinterpret_cast<const float4 *>(st + L.master + 4u * j);
    x.m4 = *reinterpret_cast<const float4 *>(st + L.m + 4u * j);
    x.v4 = *reinterpret_cast<const float4 *>(st + L.v + 4u * j);
    return x;
}

// AdamW on the four elements and their stores, straight to global memory
// (element e = tile start + j): needs nothing from the stage any more.
template <int R, bool FAST>
__device__ __forceinline__ void update_store4(Operands4 &x, size_t e, const BulkParams &p) {
    adamw_step<FAST>(x.s[0], x.p4.x, x.m4.x, x.v4.x, p.c);
    adamw_step<FAST>(x.s[1], x.p4.y, x.m4.y, x.v4.y, p.c);
    adamw_step<FAST>(x.s[2], x.p4.z, x.m4.z, x.v4.z, p.c);
    adamw_step<FAST>(x.s[3], x.p4.w, x.m4.w, x.v4.w, p.c);
    __stcs(reinterpret_cast<float4 *>(p.master + e), x.p4);
    __stcs(reinterpret_cast<float4 *>(p.m + e), x.m4);
    __stcs(reinterpret_cast<float4 *>(p.v + e), x.v4);
    const uint2 o = make_uint2(pack_bf16x2(x.p4.x, x.p4.y), pack_bf16x2(x.p4.z, x.p4.w));
#pragma unroll
    for (int r = 0; r < R; ++r) __stcs(reinterpret_cast<uint2 *>(p.out[r] + e), o);
}

// One element after the tiled range, straight from global memory.
template <int R, bool ACC, bool FAST>
__device__ void tail_element(const BulkParams &p, size_t i) {
    float s = bf16_at(p.g[0], i);
    if constexpr (ACC) s = __fadd_rn(p.acc[0][i], s);
#pragma unroll
    for (int r = 1; r < R; ++r) {
        const float t = bf16_at(p.g[r], i);
        if constexpr (ACC)
            s = __fadd_rn(s, __fadd_rn(p.acc[r][i], t));
        else
            s = __fadd_rn(s, t);
    }
    float pw = p.master[i], m = p.m[i], v = p.v[i];
    adamw_step<FAST>(s, pw, m, v, p.c);
    p.master[i] = pw;
    p.m[i] = m;
    p.v[i] = v;
    const __nv_bfloat16 b = __float2bfloat16_rn(pw);
#pragma unroll
    for (int r = 0; r < R; ++r) reinterpret_cast<__nv_bfloat16 *>(p.out[r])[i] = b;
}

template <int R, bool ACC, bool FAST>
__global__ void __launch_bounds__(kBulkThreads, 1)
fused_step_bulk_kernel(const __grid_constant__ BulkParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];

    const int T = p.tile;
    const int S = p.stages;
    const StageLayout L = stage_layout(R, ACC, T);
    const int tid = threadIdx.x;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 1);
            mbar_init(smem_addr(&empty_bar[s]), kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const uint64_t pol = evict_first_policy();
    if (tid < 32) {
        // ---------------- producer warp (lane 0 issues) ----------------
        if (tid == 0) {
            int issued_use[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) issued_use[s] = -1;
            size_t i = 0;
            for (size_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++i) {
                const int s = static_cast<int>(i % S);
                const int k = static_cast<int>(i / S);
                if (k > 0 &&
                    !mbar_wait(smem_addr(&empty_bar[s]), (k - 1) & 1, p.timeout_ns)) {
                    atomicOr(&g_bulk_status, kStatusProducerTimeout);
                    break;
                }
                // Failure injection: this tile is never issued, so its stage
                // never fills and the consumers' waits for it run out.
                if (t == p.skip_tile) continue;
                const size_t e0 = p.begin + t * static_cast<size_t>(T);
                const size_t left = p.tiled - t * static_cast<size_t>(T);
                const uint32_t len = static_cast<uint32_t>(left < static_cast<size_t>(T) ? left : T);
                unsigned char *st = smem + static_cast<size_t>(s) * L.bytes;
                const uint32_t bar = smem_addr(&full_bar[s]);
                // (debug builds) the copies stay inside the range and the stage
                debug_in_bounds(e0 - p.begin, len, p.tiled);
                debug_in_bounds(static_cast<size_t>(s) * L.bytes + L.v + 4u * T, 0,
                                static_cast<size_t>(S) * L.bytes);
                const uint32_t bytes = len * (2u * R + 12u + (ACC ? 4u * R : 0u));
                mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
                for (int r = 0; r < R; ++r)
                    bulk_load(smem_addr(st + L.g + 2u * r * T), p.g[r] + e0, 2u * len, bar, pol);
                if constexpr (ACC) {
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        bulk_load(smem_addr(st + L.acc + 4u * r * T), p.acc[r] + e0, 4u * len,
                                  bar, pol);
                }
                bulk_load(smem_addr(st + L.master), p.master + e0, 4u * len, bar, pol);
                bulk_load(smem_addr(st + L.m), p.m + e0, 4u * len, bar, pol);
                bulk_load(smem_addr(st + L.v), p.v + e0, 4u * len, bar, pol);
                issued_use[s] = k;
            }
            // Whether the loop ended normally or gave up, every copy issued
            // lands before this thread -- and so the CTA, whose shared memory
            // the copies write -- may exit: consumers that abandoned the
            // pipeline no longer wait for them.  A stage's last issued use
            // completes its full barrier's phase once its bytes have landed;
            // issued copies always land, so this wait keeps the long bound.
            for (int s = 0; s < S; ++s)
                if (issued_use[s] >= 0 &&
                    !mbar_wait(smem_addr(&full_bar[s]), issued_use[s] & 1, p.drain_timeout_ns))
                    atomicOr(&g_bulk_status, kStatusDrainTimeout);
        }
        return;
    }

    // ---------------- consumer warps ----------------
    // Group q of kGroups takes this CTA's tiles q, q + kGroups, ... (with S a
    // multiple of kGroups, every use of a stage belongs to one group); its warp
    // w (0..7) owns elements [128 w, 128 w + 128) of each, lane l the four
    // at 128 w + 4 l.  Several tiles are in arithmetic at once, so the
    // latency of one element's chain of operations hides behind the others.
    const int group = (tid - 32) / kConsumers;
    const int ct = (tid - 32) % kConsumers;
    const int j = 4 * ct;
    size_t i = static_cast<size_t>(group);
    for (size_t t = blockIdx.x + static_cast<size_t>(group) * gridDim.x; t < p.num_tiles;
         t += static_cast<size_t>(kGroups) * gridDim.x, i += kGroups) {
        const int s = static_cast<int>(i % S);
        const int k = static_cast<int>(i / S);
        const bool ready = mbar_wait(smem_addr(&full_bar[s]), k & 1, p.timeout_ns);
        // A warp-uniform decision: if any lane ran out of time the warp stops
        // (its stage is never released, so the producer stops too).
        if (!__all_sync(0xFFFFFFFFu, ready)) {
            if ((ct & 31) == 0) atomicOr(&g_bulk_status, kStatusConsumerTimeout);
            break;
        }
        const size_t left = p.tiled - t * static_cast<size_t>(T);
        const int len = static_cast<int>(left < static_cast<size_t>(T) ? left : T);
        const unsigned char *st = smem + static_cast<size_t>(s) * L.bytes;
        const size_t e0 = p.begin + t * static_cast<size_t>(T);
        // Read and reduce, hand the stage back, then update and store: the
        // producer refills the stage while this warp does the arithmetic.
        const bool mine = j < len && debug_in_bounds(e0 + j - p.begin, 4, p.tiled) &&
                          debug_in_bounds(j, 4, len);
        Operands4 x;
        if (mine) x = read_reduce4<R, ACC>(st, L, T, j);
        __syncwarp();
        if ((ct & 31) == 0) mbar_arrive(smem_addr(&empty_bar[s]));
        if (mine) update_store4<R, FAST>(x, e0 + j, p);
    }
    if (blockIdx.x == gridDim.x - 1 && group == 0 && ct < p.tail_len)
        tail_element<R, ACC, FAST>(p, p.tail_begin + ct);
}

using BulkKernel = void (*)(BulkParams);

template <int R>
BulkKernel pick_bulk(bool acc, bool fast) {
    if (fast) return acc ? fused_step_bulk_kernel<R, true, true> : fused_step_bulk_kernel<R, false, true>;
    return acc ? fused_step_bulk_kernel<R, true, false> : fused_step_bulk_kernel<R, false, false>;
}

BulkKernel bulk_kernel_for(int R, bool acc, bool fast) {
    switch (R) {
        case 1: return pick_bulk<1>(acc, fast);
        case 2: return pick_bulk<2>(acc, fast);
        case 3: return pick_bulk<3>(acc, fast);
        case 4: return pick_bulk<4>(acc, fast);
        case 5: return pick_bulk<5>(acc, fast);
        case 6: return pick_bulk<6>(acc, fast);
        case 7: return pick_bulk<7>(acc, fast);
        case 8: return pick_bulk<8>(acc, fast);
        case 9: return pick_bulk<9>(acc, fast);
        case 10: return pick_bulk<10>(acc, fast);
        case 11: return pick_bulk<11>(acc, fast);
        case 12: return pick_bulk<12>(acc, fast);
        case 13: return pick_bulk<13>(acc, fast);
        case 14: return pick_bulk<14>(acc, fast);
        case 15: return pick_bulk<15>(acc, fast);
        case 16: return pick_bulk<16>(acc, fast);
        default: return nullptr;
    }
}

// Tile length and stage count for R replicas: the largest tile (1024, 512
// or 256 elements) that still gives every consumer group a stage and three
// more stages in flight, within the budget.  The stage count is a multiple
// of the group count, so that a stage's consecutive uses (tiles i and i + S)
// always fall to the same group, which takes its tiles in order: a group
// then never waits on a stage whose previous use has not completed, where
// the parity test of the mbarrier would pass a phase early.  Returns false
// if no tile leaves at least one stage per group.
bool choose_tiling(int R, bool acc, int *tile, int *stages) {
    for (int T = kMaxTile; T >= 256; T /= 2) {
        int S = kSmemBudget / static_cast<int>(stage_layout(R, acc, T).bytes);
        if (S >= kGroups + 3 || T == 256) {
            S = S < kMaxStages ? S : kMaxStages;
            S -= S % kGroups;
            *tile = T;
            *stages = S;
            return S >= kGroups;
        }
    }
    return false;
}

constexpr int kMaxDevices = 64;
bool g_smem_attr_set[kMaxDevices][CC_MAX_R + 1][2][2];
std::mutex g_smem_attr_mutex;

// One-shot failure injection of the next bulk-engine launch on this thread
// (cc_inject_bulk_stall): the tile to skip, or -1, and the wait bound.
thread_local long long g_stall_tile = -1;
thread_local unsigned long long g_stall_timeout_ns = 0;

constexpr unsigned long long kWaitTimeoutNs = 1000000000ull;   // one second

}  // namespace

void arm_bulk_stall(long long tile, unsigned long long timeout_ns) {
    g_stall_tile = tile;
    g_stall_timeout_ns = timeout_ns;
}

cudaError_t launch_fused_bulk(const Slabs &s, const AdamScalars &c, size_t begin,
                              size_t end, int num_ctas, cudaStream_t stream) {
    if (end <= begin) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if ((e = device_sm_count(&sms)) != cudaSuccess) return e;
    const bool acc = s.acc[0] != nullptr;
    if (s.one_out) return cudaErrorInvalidValue;   // the bulk engine writes all R slabs
    BulkKernel kern = bulk_kernel_for(s.R, acc, s.fast);
    int T = 0, S = 0;
    if (!choose_tiling(s.R, acc, &T, &S)) return cudaErrorInvalidConfiguration;
    const unsigned smem = static_cast<unsigned>(S) * stage_layout(s.R, acc, T).bytes;
    {
        std::lock_guard<std::mutex> lock(g_smem_attr_mutex);
        if (!g_smem_attr_set[dev][s.R][acc ? 1 : 0][s.fast ? 1 : 0]) {
            e = cudaFuncSetAttribute(reinterpret_cast<const void *>(kern),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
            if (e != cudaSuccess) return e;
            g_smem_attr_set[dev][s.R][acc ? 1 : 0][s.fast ? 1 : 0] = true;
        }
    }
    BulkParams p{};
    for (int r = 0; r < s.R; ++r) {
        p.g[r] = static_cast<const uint16_t *>(s.grads[r]);
        p.acc[r] = s.acc[r];
        p.out[r] = static_cast<uint16_t *>(s.out[r]);
    }
    p.master = s.master;
    p.m = s.m;
    p.v = s.v;
    p.c = c;
    p.begin = begin;
    p.tiled = (end - begin) / CC_PAD_ELEMS * CC_PAD_ELEMS;
    p.tile = T;
    p.stages = S;
    p.num_tiles = (p.tiled + T - 1) / T;
    p.tail_begin = begin + p.tiled;
    p.tail_len = static_cast<int>(end - p.tail_begin);
    p.timeout_ns = kWaitTimeoutNs;
    p.drain_timeout_ns = kWaitTimeoutNs;
    p.skip_tile = SIZE_MAX;
    if (g_stall_tile >= 0) {
        p.skip_tile = static_cast<size_t>(g_stall_tile);
        p.timeout_ns = g_stall_timeout_ns;
        g_stall_tile = -1;
    }
    size_t grid = num_ctas > 0 ? static_cast<size_t>(num_ctas) : static_cast<size_t>(sms);
    if (grid > static_cast<size_t>(sms)) grid = sms;
    if (p.num_tiles > 0 && grid > p.num_tiles) grid = p.num_tiles;
    if (grid == 0) grid = 1;
    kern<<<static_cast<unsigned>(grid), kBulkThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t read_bulk_status(unsigned *status, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_bulk_status, sizeof(unsigned));
    if (e == cudaSuccess && clear) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_bulk_status, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace ccdp
