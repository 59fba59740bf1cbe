// The tensor-parallel MatMul and the AllReduce that follows it, fused into
// one tcgen05 kernel for sm_103a ("LIT-735: Breaking the Computation and
// Communication Abstraction Barrier in Distributed Machine Learning
// Workloads", Key takeaways: the model-parallel MatMul followed by an
// AllReduce, whose overlap CoCoNet exploits).
//
// R tensor-parallel ranks of a row-parallel linear layer are emulated in one
// GPU.  Rank r holds X_r (m x k/R, bf16, row-major) and its weight shard W_r
// (n x k/R, bf16, row-major: the K-contiguous layout of a linear layer's
// weight) and computes the partial product Y_r = X_r W_r^T with fp32
// accumulation.  The AllReduce gives every rank
//     out[r] = bf16_rne( (..((Y_0 + Y_1) + Y_2) .. ) + Y_{R-1} )
// summed in rank order in fp32, the same value for every r.
//
// Unfused, the R partial products go to HBM in fp32 and an AllReduce pass
// reads them back (4R bytes written + 4R read + 2R written per output
// element).  Here no partial product leaves the SM.  Persistent CTAs walk
// output tiles, and for each tile
//   * a producer warp streams 64-wide k-blocks of X_r and W_r for
//     r = 0..R-1 with TMA (cp.async.bulk.tensor, 128-byte swizzle) into a
//     ring of shared-memory stages;
//   * an MMA warp issues tcgen05.mma (bf16 in, fp32 accumulate) from those
//     stages into one of two TMEM accumulators, alternating per rank, so the
//     next rank's MMAs run while the epilogue drains the previous one;
//   * 4 * BN / 64 epilogue warps (each thread one row and 64 columns) read
//     each finished accumulator from TMEM (tcgen05.ld), add it to a running
//     fp32 sum in registers in rank order, and hand the accumulator back at
//     once.  After the last rank they round the sum to bf16 once and store
//     it to all R outputs through swizzled shared-memory boxes and TMA
//     stores -- the AllReduce's broadcast -- while the MMA warp already
//     works on the next tile.
// Only the operands are read and only the R bf16 outputs are written.
//
// Two kernels share this design.  The pair kernel (tp_fused_pair_kernel,
// used wherever the 128-row tiles pair up) runs one MMA over two SMs
// (tcgen05.mma.cta_group::2, M = 256): each CTA of a cluster of two loads
// its own 128 rows of X and half of the W tile, and the leader issues the
// MMAs for both.  Its tile width BN (256, 192 or 128) is chosen per shape
// by a model of its waves times its operand intake.  When a few groups of
// tiles are left for a last wave, a caller workspace lets it split them
// into their R rank products spread over the pairs: each product goes to
// the workspace in fp32 and the last of a group's R to finish, counted
// with an atomic ticket, sums them in rank order and stores the outputs.
// The single-CTA kernel (tp_fused_kernel, M = 128, optionally in clusters
// that share operand tiles by TMA multicast) takes odd row-tile counts.
//
// Every wait on an mbarrier is bounded by the global timer.  A wait that
// runs out records a code in this file's status word (read through
// cc_device_status), and its warp leaves its loop; the producer then waits,
// bounded again, for the copies it issued, the MMA warp for the MMAs it
// issued, and the TMEM is freed before the CTA exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "cc_dp_internal.h"
#include "cc_trace.h"

namespace ccdp {

// Codes or-ed in by a wait of the fused tensor-parallel kernel that ran out.
__device__ unsigned int g_tp_status = 0;

namespace {

constexpr int kBM = 128;                 // output rows per tile (MMA M)
constexpr int kBK = 64;                  // K per stage: 128 bytes of bf16
constexpr int kUmmaK = 16;               // K of one tcgen05.mma for 16-bit inputs
constexpr int kTileA = kBM * kBK * 2;    // 16 KiB
constexpr int kEpiCols = 64;             // output columns per epilogue thread
constexpr int kAccCols = 256;            // TMEM columns per accumulator
constexpr int kTmemCols = 2 * kAccCols;  // two accumulators: all 512 columns
constexpr int kChunk = 32;               // TMEM columns per epilogue load

#ifndef CC_TP_PREFETCH
#define CC_TP_PREFETCH 0    // k-blocks of L2 prefetch ahead of the loads (0: none;
                            // 8-32 measured no faster on the GPT-2 MLP shape)
#endif
constexpr int kPrefetch = CC_TP_PREFETCH;

#ifndef CC_TP_PAIR_BOX_COLS
#define CC_TP_PAIR_BOX_COLS 32   // columns of the pair kernel's output staging boxes
#endif

#ifndef CC_TP_STAGE_FENCE
#define CC_TP_STAGE_FENCE 1   // tcgen05 fence after each stage's full-barrier wait
#endif

// Shapes of one tile width BN (output columns per tile, the MMA's N).
template <int BN>
struct TileCfg {
    static_assert(BN % 64 == 0 && BN <= kAccCols, "BN: 128, 192 or 256");
    static constexpr int kTileB = BN * kBK * 2;
    static constexpr int kStageBytes = kTileA + kTileB;
    // Epilogue: one warp per 32 TMEM lanes and 64 columns, so that every
    // thread holds 64 running sums: 4 * BN / 64 warps, plus the producer and
    // MMA warps.  Each epilogue warp stages its 32 x 64 bf16 output block
    // (4 KiB) in shared memory for the TMA stores.
    static constexpr int kEpiWarps = 4 * (BN / kEpiCols);
    static constexpr int kThreads = 32 * (2 + kEpiWarps);
    static constexpr int kOutBox = 32 * kEpiCols * 2;
    static constexpr int kOutBytes = kEpiWarps * kOutBox;
    static constexpr int kStages =
        (220 * 1024 - kOutBytes) / kStageBytes < 8 ? (220 * 1024 - kOutBytes) / kStageBytes : 8;
    static constexpr int kSmemBytes = kStages * kStageBytes + kOutBytes + 1024;   // + align
    static constexpr int kChunks = kEpiCols / kChunk;
    static_assert(BN % kEpiCols == 0 && kTileB % 1024 == 0, "epilogue groups and swizzle atoms");
    // Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, both
    // K-major, fp32 accumulator, M = 128, N = BN.
    static constexpr uint32_t kInstrDesc = (1u << 4)                     // D: f32
                                         | (1u << 7)                     // A: bf16
                                         | (1u << 10)                    // B: bf16
                                         | (static_cast<uint32_t>(BN >> 3) << 17)
                                         | (static_cast<uint32_t>(kBM >> 4) << 24);
};

constexpr unsigned kStatusProducer = 8u;
constexpr unsigned kStatusMma = 16u;
constexpr unsigned kStatusEpilogue = 32u;
constexpr unsigned kStatusDrain = 64u;
constexpr unsigned kStatusBounds = 128u;   // debug builds: an access outside its buffer

#ifndef CC_DEBUG_BOUNDS
#define CC_DEBUG_BOUNDS 0   // 1: check the epilogue's computed offsets; skip and report
#endif
constexpr bool kDebugBounds = CC_DEBUG_BOUNDS != 0;
constexpr unsigned long long kTimeoutNs = 2000000000ull;   // two seconds per wait

struct TpFusedParams {
    CUtensorMap tx[CC_MAX_R];     // X_r: {k/R, m}, box {64, 128 / CN}
    CUtensorMap tw[CC_MAX_R];     // W_r: {k/R, n}, box {64, BN / CM}
    CUtensorMap tout[CC_MAX_R];   // out[r]: {n, m}, box {64, 32}
    __nv_bfloat16 *out[CC_MAX_R]; // m x n each
    float *partials[CC_MAX_R];    // m x n each, or all null
    int R, m, n, kb_per_rank;     // kb_per_rank = (k/R) / 64
    int tiles_n, num_tiles;
    // The pair kernel's last wave, balanced: groups [full_groups, all) are
    // cut into their R rank phases, spread over every cluster; each phase's
    // product goes to tail_ws as fp32 and the last phase of a group to
    // finish (tail_count) sums them in rank order.  tail_phases = 0: none.
    float *tail_ws;
    unsigned *tail_count;
    int full_groups, tail_phases;
    size_t tail_ws_floats;        // the slots' extent, for the debug bounds checks
};

// Debug builds: whether [off, off + len) lies inside a buffer of `limit`
// elements; if not, the status word says so and the access is skipped.
__device__ __forceinline__ bool debug_in_bounds(size_t off, size_t len, size_t limit) {
    if constexpr (!kDebugBounds) return true;
    if (off + len <= limit) return true;
    atomicOr(&g_tp_status, kStatusBounds);
    return false;
}

// The (group, rank) phases one cluster works through, numbered 0, 1, ...:
// first its whole groups (every rank of group first, then first + stride,
// ...), then its share of the split groups' single phases (q = first,
// first + stride, ... of full_groups * R + q).  Kept as one counter so that
// the schedule costs the epilogue no registers.
struct Phases {
    int first, stride, whole_jobs, jobs;
    __device__ Phases(const TpFusedParams &p, int first_, int stride_)
        : first(first_), stride(stride_) {
        const int whole = p.full_groups > first ? (p.full_groups - first + stride - 1) / stride : 0;
        const int split = p.tail_phases > first ? (p.tail_phases - first + stride - 1) / stride : 0;
        whole_jobs = whole * p.R;
        jobs = whole_jobs + split;
    }
    // group g and rank r of job j; whether the group is split
    __device__ bool at(const TpFusedParams &p, int j, int &g, int &r) const {
        if (j < whole_jobs) {
            g = first + (j / p.R) * stride;
            r = j % p.R;
            return false;
        }
        const int q = first + (j - whole_jobs) * stride;
        g = p.full_groups + q / p.R;
        r = q % p.R;
        return true;
    }
};

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
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
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
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

// Wait for the phase of this parity to complete, at most about kTimeoutNs.
// The timer is read once every 256 tries, so a wait that succeeds soon
// costs only the tries.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    unsigned long long t0 = 0;
    for (uint32_t tries = 1;; ++tries) {
        if (mbar_test(bar, parity)) return true;
        if ((tries & 255u) == 0) {
            const unsigned long long now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kTimeoutNs) return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x,
                                            int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// The same box delivered to the same shared-memory offset of every CTA in
// cta_mask (this GPU's own memory, within one cluster), each signalling its
// own mbarrier at the same offset.
__device__ __forceinline__ void tma_load_2d_multicast(uint32_t dst, const CUtensorMap *map,
                                                      int x, int y, uint32_t bar,
                                                      uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar),
          "h"(cta_mask)
        : "memory");
}

// Shared -> global tensor store of one box (bulk async group).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int x, int y,
                                             uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the bulk groups committed so far have read their shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until they have completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Make this thread's shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// A TMA load into this CTA's shared memory that signals an mbarrier of
// either CTA of the pair (the MMA pair's leader).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x,
                                                 int y, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".cta_group::2 [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// Arrive on an mbarrier given by its cluster address (here: the leader's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// The leader's own mbarrier, once every pair MMA issued before has
// completed (a kernel uses one CTA-group form throughout).
__device__ __forceinline__ void mma_commit_pair_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}

// Arrive on the mbarrier at this offset in both CTAs of the pair once every
// pair MMA issued before has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster"
                 ".multicast::cluster.b64 [%0], %1;"
                 ::"r"(bar), "h"(static_cast<uint16_t>(3)) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; orders shared-memory set-up
// (mbarrier initialisation) before any peer's use of it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bring a box of the tensor into L2 ahead of its load (no shared memory).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y) : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms of 1 KiB one after the
// other (stride-dimension offset 1024 B), start address in 16-byte units.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);       // start address
    d |= static_cast<uint64_t>(1) << 16;                      // leading offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;              // stride offset: 1 KiB
    d |= static_cast<uint64_t>(1) << 46;                      // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                      // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// The mbarrier arrives once every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}

// The same, arriving on the mbarrier at this offset in every CTA of cta_mask.
__device__ __forceinline__ void mma_commit_multicast(uint32_t bar, uint16_t cta_mask) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster"
                 ".multicast::cluster.b64 [%0], %1;"
                 ::"r"(bar), "h"(cta_mask) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

#define CC_TMEM_REGS32(r)                                                                  \
    "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),    \
    "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),             \
    "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),          \
    "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),          \
    "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])

// Start loading 32 consecutive fp32 columns of this warp's 32 TMEM lanes:
// lane i of the warp gets row (lane base + i), columns [col, col + 32).
// The values are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : CC_TMEM_REGS32(r)
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t a, uint32_t b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(a), __uint_as_float(b));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// CM x CN CTAs form a cluster working on CM x CN neighbouring tiles: CTA
// (a, b) (cluster rank a + CM b) computes the tile in row a and column b of
// the group.  The tiles of one row share their X tile and those of one
// column their W tile, so each CTA loads 1/CN of its X tile and 1/CM of its
// W tile and multicasts them to the CTAs that share them: every shared-
// memory stage is filled by the CTAs of its row and column.  A stage may be
// refilled only once all of those CTAs' MMAs have read it, so each MMA
// commit arrives on the empty barriers of its whole row and column.
// CM = CN = 1 is the plain single-CTA kernel.
template <int BN, int CM, int CN>
__global__ void __launch_bounds__(TileCfg<BN>::kThreads, 1)
tp_fused_kernel(const __grid_constant__ TpFusedParams p) {
    using C = TileCfg<BN>;
    constexpr int kStages = C::kStages;
    constexpr int kCluster = CM * CN;
    constexpr int kSliceA = kBM / CN;          // rows of the X tile this CTA loads
    constexpr int kSliceB = BN / CM;           // rows of the W tile this CTA loads
    static_assert(kSliceA % 8 == 0 && kSliceB % 8 == 0, "slices of whole 1 KiB atoms");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t acc_full[2];
    __shared__ __align__(8) uint64_t acc_empty[2];
    __shared__ __align__(8) uint64_t mma_done;
    __shared__ uint32_t tmem_base_slot;

    // The 128-byte swizzle wants 1 KiB-aligned tiles.
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int R = p.R;
    const int kb_per_rank = p.kb_per_rank;
    const uint32_t crank = kCluster > 1 ? cluster_ctarank() : 0u;
    const int ca = static_cast<int>(crank) % CM;     // row of the group
    const int cb = static_cast<int>(crank) / CM;     // column of the group
    uint16_t row_set = 0, col_set = 0;
#pragma unroll
    for (int b = 0; b < CN; ++b) row_set |= static_cast<uint16_t>(1u << (ca + CM * b));
#pragma unroll
    for (int a = 0; a < CM; ++a) col_set |= static_cast<uint16_t>(1u << (a + CM * cb));
    const uint16_t peers = row_set | col_set;         // who fills, and reads, this stage

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), CM + CN - 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&acc_full[a]), 1);
            mbar_init(smem_u32(&acc_empty[a]), C::kEpiWarps);
        }
        mbar_init(smem_u32(&mma_done), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (kCluster > 1) cluster_sync();       // peers' barriers exist
    if (warp == 0 && lane == 0) {
        for (int r = 0; r < R; ++r) {
            prefetch_map(&p.tx[r]);
            prefetch_map(&p.tw[r]);
        }
    }
    if (warp == 1) {
        // One warp allocates all 512 TMEM columns (one CTA per SM).
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_base_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_slot;
    // Groups of CM x CN tiles, one per cluster at a time.
    const int groups_n = p.tiles_n / CN;
    const int num_groups = (p.num_tiles / p.tiles_n / CM) * groups_n;
    const int first_group = static_cast<int>(blockIdx.x) / kCluster;
    const int group_stride = static_cast<int>(gridDim.x) / kCluster;

    if (warp == 0) {
        // ---------------- producer: TMA loads of X_r and W_r tiles --------
        if (lane == 0) {
            int issued_use[kStages];
            for (int s = 0; s < kStages; ++s) issued_use[s] = -1;
            uint32_t it = 0;
            bool ok = true;
            for (int g = first_group; ok && g < num_groups; g += group_stride) {
                const int m0 = ((g / groups_n) * CM + ca) * kBM;
                const int n0 = ((g % groups_n) * CN + cb) * BN;
                // L2 prefetch kPrefetch k-blocks ahead of the loads, within
                // the tile.
                int pf_r = 0, pf_kb = 0;
                for (int ahead = 0; ahead < kPrefetch && pf_r < R; ++ahead) {
                    tma_prefetch_2d(&p.tx[pf_r], pf_kb * kBK, m0);
                    tma_prefetch_2d(&p.tw[pf_r], pf_kb * kBK, n0);
                    if (++pf_kb == kb_per_rank) { pf_kb = 0; ++pf_r; }
                }
                for (int r = 0; ok && r < R; ++r) {
                    for (int kb = 0; kb < kb_per_rank; ++kb, ++it) {
                        if (pf_r < R) {
                            tma_prefetch_2d(&p.tx[pf_r], pf_kb * kBK, m0);
                            tma_prefetch_2d(&p.tw[pf_r], pf_kb * kBK, n0);
                            if (++pf_kb == kb_per_rank) { pf_kb = 0; ++pf_r; }
                        }
                        const int s = static_cast<int>(it % kStages);
                        const int use = static_cast<int>(it / kStages);
                        if (use > 0 && !mbar_wait(smem_u32(&empty_bar[s]), (use - 1) & 1)) {
                            atomicOr(&g_tp_status, kStatusProducer);
                            ok = false;
                            break;
                        }
                        const uint32_t sa = base + static_cast<uint32_t>(s) * C::kStageBytes;
                        const uint32_t bar = smem_u32(&full_bar[s]);
                        // the whole stage arrives: this CTA's slices and its
                        // row's and column's multicasts
                        mbar_arrive_expect_tx(bar, C::kStageBytes);
                        const uint32_t dst_a = sa + static_cast<uint32_t>(cb * kSliceA * 128);
                        const uint32_t dst_b =
                            sa + kTileA + static_cast<uint32_t>(ca * kSliceB * 128);
                        if constexpr (CN > 1)
                            tma_load_2d_multicast(dst_a, &p.tx[r], kb * kBK, m0 + cb * kSliceA,
                                                  bar, row_set);
                        else
                            tma_load_2d(dst_a, &p.tx[r], kb * kBK, m0, bar);
                        if constexpr (CM > 1)
                            tma_load_2d_multicast(dst_b, &p.tw[r], kb * kBK, n0 + ca * kSliceB,
                                                  bar, col_set);
                        else
                            tma_load_2d(dst_b, &p.tw[r], kb * kBK, n0, bar);
                        issued_use[s] = use;
                    }
                }
            }
            // Every copy into this CTA's shared memory lands, and every
            // peer MMA's arrival on its empty barriers happens, before the
            // CTA may exit.  Issued copies always land.
            for (int s = 0; s < kStages; ++s)
                if (issued_use[s] >= 0 &&
                    !mbar_wait(smem_u32(&full_bar[s]), issued_use[s] & 1))
                    atomicOr(&g_tp_status, kStatusDrain);
            if constexpr (kCluster > 1) {
                for (int s = 0; s < kStages; ++s)
                    if (issued_use[s] >= 0 &&
                        !mbar_wait(smem_u32(&empty_bar[s]), issued_use[s] & 1))
                        atomicOr(&g_tp_status, kStatusDrain);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer --------------------------------------
        if (lane == 0) {
            uint32_t it = 0, job = 0;
            bool ok = true;
            for (int g = first_group; ok && g < num_groups; g += group_stride) {
                for (int r = 0; ok && r < R; ++r, ++job) {
                    // Job j accumulates into buffer j % 2; that buffer's
                    // previous content (job j - 2's sum) must have been read.
                    const uint32_t acc = job & 1u;
                    const uint32_t acc_use = job >> 1;
                    if (acc_use > 0 && !mbar_wait(smem_u32(&acc_empty[acc]), (acc_use - 1) & 1)) {
                        atomicOr(&g_tp_status, kStatusMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + acc * kAccCols;
                    for (int kb = 0; kb < kb_per_rank; ++kb, ++it) {
                        const int s = static_cast<int>(it % kStages);
                        const int use = static_cast<int>(it / kStages);
                        if (!mbar_wait(smem_u32(&full_bar[s]), use & 1)) {
                            atomicOr(&g_tp_status, kStatusMma);
                            ok = false;
                            break;
                        }
#if CC_TP_STAGE_FENCE
                        tc_fence_after();
#endif
                        const uint32_t sa = base + static_cast<uint32_t>(s) * C::kStageBytes;
                        const uint64_t da = smem_desc_sw128(sa);
                        const uint64_t db = smem_desc_sw128(sa + kTileA);
#pragma unroll
                        for (int j = 0; j < kBK / kUmmaK; ++j) {
                            // K step j: 16 elements = 32 bytes further along the
                            // 128-byte swizzled rows (2 in 16-byte units).
                            mma_bf16(d_tmem, da + 2u * j, db + 2u * j, C::kInstrDesc,
                                     (kb > 0 || j > 0) ? 1u : 0u);
                        }
                        // the stage is free in every CTA that fills it once read
                        if constexpr (kCluster > 1)
                            mma_commit_multicast(smem_u32(&empty_bar[s]), peers);
                        else
                            mma_commit(smem_u32(&empty_bar[s]));
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&acc_full[acc]));      // rank r's product complete
                }
            }
            // Every MMA issued completes before the TMEM is freed.
            mma_commit(smem_u32(&mma_done));
            if (!mbar_wait(smem_u32(&mma_done), 0)) atomicOr(&g_tp_status, kStatusDrain);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: rank-order sum, bf16, R stores ---------
        const int e = warp - 2;                   // 0 .. kEpiWarps-1
        const int quarter = warp % 4;             // TMEM lanes 32*quarter.. (hardware rule)
        const int group = e / 4;                  // 64-column group of the tile
        const int row_in_tile = 32 * quarter + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * quarter) << 16;
        const uint32_t col_off = static_cast<uint32_t>(group * kEpiCols);
        const uint32_t out_box = base + static_cast<uint32_t>(kStages * C::kStageBytes) +
                                 static_cast<uint32_t>(e * C::kOutBox);
        // Rank-indexed pointers read through the parameter's own address
        // (a __grid_constant__ parameter is never copied).
        float *const *partials = p.partials;
        const bool keep_partials = partials[0] != nullptr;
        const size_t n = static_cast<size_t>(p.n);
        uint32_t job = 0;
        bool ok = true;
        for (int g = first_group; ok && g < num_groups; g += group_stride) {
            const int m0 = ((g / groups_n) * CM + ca) * kBM;
            const int n0 = ((g % groups_n) * CN + cb) * BN;
            const size_t off = static_cast<size_t>(m0 + row_in_tile) * n + n0 + col_off;
            float sum[kEpiCols];
            for (int r = 0; r < R; ++r, ++job) {
                const uint32_t acc = job & 1u;
                const bool ready = mbar_wait(smem_u32(&acc_full[acc]), (job >> 1) & 1);
                if (!__all_sync(0xFFFFFFFFu, ready)) {
                    if (lane == 0) atomicOr(&g_tp_status, kStatusEpilogue);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t y_addr = tmem + lane_addr + acc * kAccCols + col_off;
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) {
                    uint32_t y[32];
                    tmem_ld32(y_addr + kChunk * c, y);
                    tmem_wait_ld();
                    if (keep_partials) {
                        // rank r's partial product as the tensor cores made it
                        float4 *dst = reinterpret_cast<float4 *>(partials[r] + off + kChunk * c);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[q] = make_float4(__uint_as_float(y[4 * q]),
                                                 __uint_as_float(y[4 * q + 1]),
                                                 __uint_as_float(y[4 * q + 2]),
                                                 __uint_as_float(y[4 * q + 3]));
                    }
                    // rank order: S_0 = Y_0, S_r = S_{r-1} + Y_r
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        sum[kChunk * c + i] = r == 0 ? __uint_as_float(y[i])
                                                     : __fadd_rn(sum[kChunk * c + i],
                                                                 __uint_as_float(y[i]));
                }
                // The accumulator has been read: rank r + 2 may reuse it.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&acc_empty[acc]));
            }
            if (!ok) break;
            // Round the sum once to bf16 into this warp's 32 x 64 staging box
            // (the 128-byte swizzle: 16-byte chunk j of row i at chunk
            // j ^ (i % 8), no bank conflicts beyond the minimum), then TMA
            // stores the box to every rank's output -- the AllReduce's
            // result on every rank -- in whole lines, while the MMA warp
            // already accumulates the next tile.
            if (lane == 0) bulk_wait_read_all();     // the last tile's stores have read it
            __syncwarp();
#pragma unroll
            for (int q = 0; q < kEpiCols / 8; ++q) {
                const uint4 pk = make_uint4(
                    pack_bf16x2(__float_as_uint(sum[8 * q]), __float_as_uint(sum[8 * q + 1])),
                    pack_bf16x2(__float_as_uint(sum[8 * q + 2]), __float_as_uint(sum[8 * q + 3])),
                    pack_bf16x2(__float_as_uint(sum[8 * q + 4]), __float_as_uint(sum[8 * q + 5])),
                    pack_bf16x2(__float_as_uint(sum[8 * q + 6]), __float_as_uint(sum[8 * q + 7])));
                const uint32_t chunk = static_cast<uint32_t>(q) ^ static_cast<uint32_t>(lane & 7);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                             ::"r"(out_box + static_cast<uint32_t>(lane) * 128u + chunk * 16u),
                               "r"(pk.x), "r"(pk.y), "r"(pk.z), "r"(pk.w) : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int x = n0 + static_cast<int>(col_off);
                const int y = m0 + 32 * quarter;
                for (int o = 0; o < R; ++o) tma_store_2d(&p.tout[o], x, y, out_box);
                bulk_commit_group();
            }
        }
        if (lane == 0) bulk_wait_all();               // stores done before exit
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (kCluster > 1) cluster_sync();       // no peer still writes here
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// ---------------------------------------------------------------------------
// The pair form: one MMA over two SMs (tcgen05 cta_group::2, M = 256).
//
// Two CTAs of a cluster compute two vertically adjacent 128 x BN tiles as
// one 256 x BN product.  Each CTA loads its own 128 rows of X and half of the
// W tile (BN/2 rows) into its own shared memory; the leader CTA (rank 0)
// issues the MMAs, which read A from each CTA's own stage and B from both,
// and accumulate each CTA's 128 rows in that CTA's TMEM.  So each SM takes in
// 16 KiB of X and BN/2 x 128 bytes of W per k-block of 64, against 16 KiB +
// BN x 128 bytes for the single-CTA kernel: 30% fewer operand bytes per
// FLOP at BN = 192, where one SM's operand intake is the bound.
//   * Both CTAs' TMA loads signal the leader's "full" barrier (expecting both
//     CTAs' bytes); the leader's MMA commits arrive on the "empty" barriers
//     and the accumulator barriers of both CTAs.
//   * Each CTA's epilogue reads its own TMEM lanes, keeps the rank-order sum
//     in registers and hands the accumulator back on the leader's barrier
//     (both CTAs' epilogue warps must arrive); the output leaves through the
//     same per-warp TMA stores as the single-CTA kernel.
// TMEM is allocated for the pair (both CTAs' allocating warps take part).
// ---------------------------------------------------------------------------

#ifndef CC_TP_PAIR_SMEM
#define CC_TP_PAIR_SMEM (220 * 1024)  // stages + output boxes of the pair kernel (226 KB, a
                                      // sixth stage at 256 columns, measured no faster)
#endif

template <int BN>
struct PairCfg {
    static_assert(BN % 64 == 0 && BN <= kAccCols, "BN: 128, 192 or 256");
    static constexpr int kHalfB = BN / 2;                 // W rows this CTA loads
    static constexpr int kTileB = kHalfB * kBK * 2;
    static constexpr int kStageBytes = kTileA + kTileB;
    static constexpr int kEpiWarps = 4 * (BN / kEpiCols);
    static constexpr int kThreads = 32 * (2 + kEpiWarps);
    // Each epilogue warp stages 32 rows x kBoxCols of bf16 output at a time
    // (64-byte swizzle for 32 columns, 128-byte for 64), stored twice per
    // tile with 32 columns: the smaller boxes leave room for one more stage.
    static constexpr int kBoxCols = CC_TP_PAIR_BOX_COLS;
    static constexpr int kOutBox = 32 * kBoxCols * 2;
    static constexpr int kOutBytes = kEpiWarps * kOutBox;
    static constexpr int kStagesFit = (CC_TP_PAIR_SMEM - kOutBytes) / kStageBytes;
    static constexpr int kStages = kStagesFit < 8 ? kStagesFit : 8;
    static constexpr int kSmemBytes = kStages * kStageBytes + kOutBytes + 1024;
    static constexpr int kChunks = kEpiCols / kChunk;
    static_assert(kTileB % 1024 == 0, "swizzle atoms");
    static_assert(kBoxCols == 32 || kBoxCols == 64, "output boxes of 32 or 64 columns");
    static_assert(kSmemBytes <= 227 * 1024 - 1024, "dynamic shared memory beside the barriers");
    // tcgen05.mma kind::f16, bf16 A and B (K-major), fp32 accumulator,
    // M = 256 (the pair), N = BN.
    static constexpr uint32_t kInstrDesc = (1u << 4) | (1u << 7) | (1u << 10)
                                         | (static_cast<uint32_t>(BN >> 3) << 17)
                                         | (static_cast<uint32_t>(256 >> 4) << 24);
};

// Columns 4q .. 4q+3 of a TMEM load as a float4.
__device__ __forceinline__ float4 quad(const uint32_t (&y)[32], int q) {
    return make_float4(__uint_as_float(y[4 * q]), __uint_as_float(y[4 * q + 1]),
                       __uint_as_float(y[4 * q + 2]), __uint_as_float(y[4 * q + 3]));
}

// Convert 64 running sums of one row to bf16 (nearest-even) into this warp's
// staging box and TMA-store it to every rank's output, kBoxCols columns at a
// time.  Swizzle: 16-byte chunk j of row i at chunk j ^ (i % 8) in 128-byte
// rows, j ^ ((i / 2) % 4) in 64-byte rows.
template <int kBoxCols>
__device__ __forceinline__ void store_sums_bf16(const float (&sum)[kEpiCols], int lane,
                                                uint32_t out_box, const CUtensorMap *tout,
                                                int R, int x0, int y) {
#pragma unroll
    for (int h = 0; h < kEpiCols / kBoxCols; ++h) {
        if (lane == 0) bulk_wait_read_all();         // the box is free again
        __syncwarp();
        constexpr int kq = kBoxCols / 8;             // 16-byte chunks per row
#pragma unroll
        for (int j = 0; j < kq; ++j) {
            const int q = h * kq + j;
            const uint4 pk = make_uint4(
                pack_bf16x2(__float_as_uint(sum[8 * q]), __float_as_uint(sum[8 * q + 1])),
                pack_bf16x2(__float_as_uint(sum[8 * q + 2]), __float_as_uint(sum[8 * q + 3])),
                pack_bf16x2(__float_as_uint(sum[8 * q + 4]), __float_as_uint(sum[8 * q + 5])),
                pack_bf16x2(__float_as_uint(sum[8 * q + 6]), __float_as_uint(sum[8 * q + 7])));
            const uint32_t sw = kBoxCols == 64 ? static_cast<uint32_t>(lane & 7)
                                               : static_cast<uint32_t>((lane >> 1) & 3);
            const uint32_t chunk = static_cast<uint32_t>(j) ^ sw;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         ::"r"(out_box + static_cast<uint32_t>(lane * kBoxCols * 2) + chunk * 16u),
                           "r"(pk.x), "r"(pk.y), "r"(pk.z), "r"(pk.w) : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            for (int o = 0; o < R; ++o) tma_store_2d(&tout[o], x0 + h * kBoxCols, y, out_box);
            bulk_commit_group();
        }
    }
}

#ifndef CC_TP_FIXUP_RANKS
#define CC_TP_FIXUP_RANKS 1   // ranks' loads in flight per thread in a fixup
#endif

// The fixup of a split group: this thread's 64 output columns of one row
// are the rank-order sums of the R fp32 products in the workspace (slot r at
// slot0 + r * rank_stride float4s; column quad c of the row at c * 128).
// Sixteen columns at a time, with up to four ranks' loads in flight, packed
// to bf16 straight into the warp's staging box and TMA-stored to every
// rank's output as store_sums_bf16 does.
template <int kBoxCols>
__device__ __forceinline__ void fixup_store_bf16(const float4 *slot0, size_t rank_stride, int lane,
                                                 uint32_t out_box, const CUtensorMap *tout,
                                                 int R, int x0, int y) {
    constexpr int kRanksInFlight = CC_TP_FIXUP_RANKS;
#pragma unroll 1
    for (int h = 0; h < kEpiCols / kBoxCols; ++h) {
        if (lane == 0) bulk_wait_read_all();         // the box is free again
        __syncwarp();
#pragma unroll 1
        for (int part = 0; part < kBoxCols / 16; ++part) {
            const float4 *base = slot0 + static_cast<size_t>(h * kBoxCols / 4 + part * 4) * kBM;
            float acc[16];
#pragma unroll 1
            for (int r0 = 0; r0 < R; r0 += kRanksInFlight) {
                float4 v[kRanksInFlight][4];
#pragma unroll
                for (int i = 0; i < kRanksInFlight; ++i)
                    if (r0 + i < R) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            v[i][q] = __ldcg(base + (r0 + i) * rank_stride + q * kBM);
                    }
#pragma unroll
                for (int i = 0; i < kRanksInFlight; ++i)
                    if (r0 + i < R) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float e4[4] = {v[i][q].x, v[i][q].y, v[i][q].z, v[i][q].w};
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                acc[4 * q + c] = r0 + i == 0 ? e4[c]
                                                             : __fadd_rn(acc[4 * q + c], e4[c]);
                        }
                    }
            }
            const uint32_t sw = kBoxCols == 64 ? static_cast<uint32_t>(lane & 7)
                                               : static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const uint32_t chunk = static_cast<uint32_t>(part * 2 + jj) ^ sw;
                const float *a = acc + 8 * jj;
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                             ::"r"(out_box + static_cast<uint32_t>(lane * kBoxCols * 2) +
                                   chunk * 16u),
                               "r"(pack_bf16x2(__float_as_uint(a[0]), __float_as_uint(a[1]))),
                               "r"(pack_bf16x2(__float_as_uint(a[2]), __float_as_uint(a[3]))),
                               "r"(pack_bf16x2(__float_as_uint(a[4]), __float_as_uint(a[5]))),
                               "r"(pack_bf16x2(__float_as_uint(a[6]), __float_as_uint(a[7])))
                             : "memory");
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            for (int o = 0; o < R; ++o) tma_store_2d(&tout[o], x0 + h * kBoxCols, y, out_box);
            bulk_commit_group();
        }
    }
}

template <int BN>
__global__ void __launch_bounds__(PairCfg<BN>::kThreads, 1)
tp_fused_pair_kernel(const __grid_constant__ TpFusedParams p) {
    using C = PairCfg<BN>;
    constexpr int kStages = C::kStages;
    constexpr int kSlotFloats = kBM * BN;                  // one CTA's half of a tile
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages];    // the leader's is used
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t acc_full[2];
    __shared__ __align__(8) uint64_t acc_empty[2];         // the leader's is used
    __shared__ __align__(8) uint64_t mma_done;
    __shared__ __align__(8) uint64_t tail_in;              // epilogue warps wrote a phase
    __shared__ __align__(8) uint64_t tail_out;             // ... and whether it was the last
    __shared__ uint32_t tmem_base_slot;
    __shared__ int tail_last;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int R = p.R;
    const int kb_per_rank = p.kb_per_rank;
    const uint32_t crank = cluster_ctarank();               // 0: the leader
    const bool leader = crank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&acc_full[a]), 1);
            mbar_init(smem_u32(&acc_empty[a]), 2 * C::kEpiWarps);
        }
        mbar_init(smem_u32(&mma_done), 1);
        mbar_init(smem_u32(&tail_in), C::kEpiWarps);
        mbar_init(smem_u32(&tail_out), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    cluster_sync();                                          // the pair's barriers exist
    if (warp == 0 && lane == 0) {
        for (int r = 0; r < R; ++r) {
            prefetch_map(&p.tx[r]);
            prefetch_map(&p.tw[r]);
        }
    }
    if (warp == 1) {
        // One warp of each CTA of the pair allocates, together, all 512
        // columns in both CTAs.
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_base_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_slot;
    // Pairs of row tiles ("groups"), one pair per cluster at a time.
    const int first_group = static_cast<int>(blockIdx.x) / 2;
    const int group_stride = static_cast<int>(gridDim.x) / 2;

    if (warp == 0) {
        // ---------------- producer (both CTAs) --------------------------
        if (lane == 0) {
            int issued_use[kStages];
            for (int s = 0; s < kStages; ++s) issued_use[s] = -1;
            uint32_t it = 0;
            bool ok = true;
            const Phases ph(p, first_group, group_stride);
            for (int j = 0; ok && j < ph.jobs; ++j) {
                int g, r;
                ph.at(p, j, g, r);
                const int m0 = ((g / p.tiles_n) * 2 + static_cast<int>(crank)) * kBM;
                const int n0 = (g % p.tiles_n) * BN;
                for (int kb = 0; kb < kb_per_rank; ++kb, ++it) {
                    const int s = static_cast<int>(it % kStages);
                    const int use = static_cast<int>(it / kStages);
                    if (use > 0 && !mbar_wait(smem_u32(&empty_bar[s]), (use - 1) & 1)) {
                        atomicOr(&g_tp_status, kStatusProducer);
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + static_cast<uint32_t>(s) * C::kStageBytes;
                    const uint32_t leader_full = map_to_cta(smem_u32(&full_bar[s]), 0);
                    if (leader)   // both CTAs' bytes land before the stage is full
                        mbar_arrive_expect_tx(smem_u32(&full_bar[s]), 2 * C::kStageBytes);
                    tma_load_2d_pair(sa, &p.tx[r], kb * kBK, m0, leader_full);
                    tma_load_2d_pair(sa + kTileA, &p.tw[r], kb * kBK,
                                     n0 + static_cast<int>(crank) * C::kHalfB, leader_full);
                    issued_use[s] = use;
                }
            }
            // The leader's MMAs have read every stage this CTA filled (and so
            // every copy into it has landed) before the CTA may exit.
            for (int s = 0; s < kStages; ++s)
                if (issued_use[s] >= 0 &&
                    !mbar_wait(smem_u32(&empty_bar[s]), issued_use[s] & 1))
                    atomicOr(&g_tp_status, kStatusDrain);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (the leader only) ------------------
        if (leader && lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            const Phases ph(p, first_group, group_stride);
            for (uint32_t job = 0; ok && job < static_cast<uint32_t>(ph.jobs); ++job) {
                const uint32_t acc = job & 1u;
                const uint32_t acc_use = job >> 1;
                if (acc_use > 0 && !mbar_wait(smem_u32(&acc_empty[acc]), (acc_use - 1) & 1)) {
                    atomicOr(&g_tp_status, kStatusMma);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + acc * kAccCols;
                for (int kb = 0; kb < kb_per_rank; ++kb, ++it) {
                    const int s = static_cast<int>(it % kStages);
                    const int use = static_cast<int>(it / kStages);
                    if (!mbar_wait(smem_u32(&full_bar[s]), use & 1)) {
                        atomicOr(&g_tp_status, kStatusMma);
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + static_cast<uint32_t>(s) * C::kStageBytes;
                    const uint64_t da = smem_desc_sw128(sa);
                    const uint64_t db = smem_desc_sw128(sa + kTileA);
#pragma unroll
                    for (int j = 0; j < kBK / kUmmaK; ++j)
                        mma_bf16_pair(d_tmem, da + 2u * j, db + 2u * j, C::kInstrDesc,
                                      (kb > 0 || j > 0) ? 1u : 0u);
                    mma_commit_pair(smem_u32(&empty_bar[s]));   // free in both CTAs
                }
                if (!ok) break;
                mma_commit_pair(smem_u32(&acc_full[acc]));      // both halves complete
            }
            mma_commit_pair_local(smem_u32(&mma_done));
            if (!mbar_wait(smem_u32(&mma_done), 0)) atomicOr(&g_tp_status, kStatusDrain);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (both CTAs, own rows) -----------------
        const int e = warp - 2;
        const int quarter = warp % 4;
        const int group = e / 4;
        const int row_in_tile = 32 * quarter + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * quarter) << 16;
        const uint32_t col_off = static_cast<uint32_t>(group * kEpiCols);
        const uint32_t out_box = base + static_cast<uint32_t>(kStages * C::kStageBytes) +
                                 static_cast<uint32_t>(e * C::kOutBox);
        float *const *partials = p.partials;
        const bool keep_partials = partials[0] != nullptr;
        const size_t n = static_cast<size_t>(p.n);
        const uint32_t leader_acc_empty[2] = {map_to_cta(smem_u32(&acc_empty[0]), 0),
                                              map_to_cta(smem_u32(&acc_empty[1]), 0)};
        // A tail slot holds one CTA's 128 x BN fp32 product as BN / 4 column
        // quads, each 128 rows of float4: a warp's lanes (rows) touch 512
        // consecutive bytes.  This thread's first quad:
        const size_t slot_off = (static_cast<size_t>(col_off / 4) * kBM + row_in_tile) * 4;
        const Phases ph(p, first_group, group_stride);
        bool ok = true;
        int job = 0;
        // Wait for job j's accumulator; its TMEM address (this warp's lanes
        // and columns), or false if the wait ran out.
        auto wait_acc = [&](int j, uint32_t &y_addr) {
            const uint32_t acc = static_cast<uint32_t>(j) & 1u;
            const bool ready = mbar_wait(smem_u32(&acc_full[acc]), (j >> 1) & 1);
            if (!__all_sync(0xFFFFFFFFu, ready)) {
                if (lane == 0) atomicOr(&g_tp_status, kStatusEpilogue);
                return false;
            }
            tc_fence_after();
            y_addr = tmem + lane_addr + acc * kAccCols + col_off;
            return true;
        };
        auto release_acc = [&](int j) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(leader_acc_empty[j & 1]);
        };
        {
            // Whole groups: the running sum over the R ranks in registers,
            // stored once the last rank is in.
            float sum[kEpiCols];
            for (; ok && job < ph.whole_jobs; ++job) {
                int g, r;
                ph.at(p, job, g, r);
                const int m0 = ((g / p.tiles_n) * 2 + static_cast<int>(crank)) * kBM;
                const int n0 = (g % p.tiles_n) * BN;
                const size_t off = static_cast<size_t>(m0 + row_in_tile) * n + n0 + col_off;
                uint32_t y_addr;
                if (!(ok = wait_acc(job, y_addr))) break;
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) {
                    uint32_t y[32];
                    tmem_ld32(y_addr + kChunk * c, y);
                    tmem_wait_ld();
                    if (keep_partials &&
                        debug_in_bounds(off + kChunk * c, kChunk, static_cast<size_t>(p.m) * n)) {
                        float4 *dst = reinterpret_cast<float4 *>(partials[r] + off + kChunk * c);
#pragma unroll
                        for (int q = 0; q < 8; ++q) dst[q] = quad(y, q);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        sum[kChunk * c + i] = r == 0 ? __uint_as_float(y[i])
                                                     : __fadd_rn(sum[kChunk * c + i],
                                                                 __uint_as_float(y[i]));
                }
                release_acc(job);
                if (r == R - 1)
                    store_sums_bf16<C::kBoxCols>(sum, lane, out_box, p.tout, R,
                                                 n0 + static_cast<int>(col_off), m0 + 32 * quarter);
            }
        }
        // Split groups: each phase's product, as is, to its workspace slot;
        // the group's last phase to finish (an atomic ticket per group half)
        // sums the R slots in rank order.  No CTA waits for another: only
        // this CTA's epilogue warps meet, on bounded waits.
        uint32_t tail_parity = 0;
        for (; ok && job < ph.jobs; ++job) {
            int g, r;
            ph.at(p, job, g, r);
            const int tg = g - p.full_groups;
            const int m0 = ((g / p.tiles_n) * 2 + static_cast<int>(crank)) * kBM;
            const int n0 = (g % p.tiles_n) * BN;
            const size_t off = static_cast<size_t>(m0 + row_in_tile) * n + n0 + col_off;
            const float *slots = p.tail_ws + static_cast<size_t>(tg) * R * 2 * kSlotFloats +
                                 static_cast<size_t>(crank) * kSlotFloats + slot_off;
            float *slot = const_cast<float *>(slots) + static_cast<size_t>(r) * 2 * kSlotFloats;
            uint32_t y_addr;
            if (!(ok = wait_acc(job, y_addr))) break;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
                uint32_t y[32];
                tmem_ld32(y_addr + kChunk * c, y);
                tmem_wait_ld();
                if (keep_partials &&
                    debug_in_bounds(off + kChunk * c, kChunk, static_cast<size_t>(p.m) * n)) {
                    float4 *dst = reinterpret_cast<float4 *>(partials[r] + off + kChunk * c);
#pragma unroll
                    for (int q = 0; q < 8; ++q) dst[q] = quad(y, q);
                }
                float4 *dst = reinterpret_cast<float4 *>(slot) + (kChunk / 4) * c * kBM;
                // the chunk's last float4 lies 7 * kBM float4s past its first
                if (debug_in_bounds(static_cast<size_t>(reinterpret_cast<float *>(dst) - p.tail_ws),
                                    4 * (7 * kBM + 1), p.tail_ws_floats)) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) dst[q * kBM] = quad(y, q);
                }
            }
            release_acc(job);
            __threadfence();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tail_in));
            if (e == 0 && lane == 0) {
                int last = 0;
                if (mbar_wait(smem_u32(&tail_in), tail_parity)) {
                    const unsigned ticket = atomicAdd(&p.tail_count[tg * 2 + crank], 1u);
                    last = ticket == static_cast<unsigned>(R - 1);
                    __threadfence();
                } else {
                    atomicOr(&g_tp_status, kStatusEpilogue);
                }
                tail_last = last;
                mbar_arrive(smem_u32(&tail_out));
            }
            const bool told = mbar_wait(smem_u32(&tail_out), tail_parity);
            tail_parity ^= 1u;
            if (!__all_sync(0xFFFFFFFFu, told)) {
                if (lane == 0) atomicOr(&g_tp_status, kStatusEpilogue);
                ok = false;
                break;
            }
            // the fixup reads R slots, each 16 column quads of 128 rows deep
            if (tail_last &&
                debug_in_bounds(static_cast<size_t>(slots - p.tail_ws),
                                static_cast<size_t>(R - 1) * 2 * kSlotFloats +
                                    4 * (15 * kBM + 1),
                                p.tail_ws_floats))
                fixup_store_bf16<C::kBoxCols>(reinterpret_cast<const float4 *>(slots),
                                              2 * kSlotFloats / 4, lane, out_box, p.tout, R,
                                              n0 + static_cast<int>(col_off), m0 + 32 * quarter);
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();                                          // the peer is done with us
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and the launch
// ---------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// A bf16 row-major matrix of `rows` x `cols` (cols contiguous), moved in
// boxes of box_cols columns x box_rows rows: 64 columns (128 bytes) with the
// 128-byte swizzle, or 32 columns (64 bytes) with the 64-byte swizzle.
int encode_bf16_map(CUtensorMap *map, const void *ptr, int rows, int cols, int box_rows,
                    const char *name, int r, int box_cols = kBK) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return fail(CC_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols),
                               static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr),
                            dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                           : CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS)
        return fail(CC_ERR_INVALID, "%s[%d]: tensor map rejected (CUresult %d)", name, r,
                    static_cast<int>(res));
    return CC_OK;
}

constexpr int kMaxDevices = 64;
std::mutex g_attr_mutex;

template <int BN, int CM, int CN>
int launch_cfg(TpFusedParams &p, const void *const *x, const void *const *w, int m, int n,
               int kr, int R, int max_ctas, cudaStream_t stream) {
    static bool attr_set[kMaxDevices];
    constexpr int kCluster = CM * CN;
    auto kernel = tp_fused_kernel<BN, CM, CN>;
    int st;
    for (int r = 0; r < R; ++r) {
        if ((st = encode_bf16_map(&p.tx[r], x[r], m, kr, kBM / CN, "x", r)) != CC_OK) return st;
        if ((st = encode_bf16_map(&p.tw[r], w[r], n, kr, BN / CM, "w", r)) != CC_OK) return st;
        if ((st = encode_bf16_map(&p.tout[r], p.out[r], m, n, 32, "out", r)) != CC_OK) return st;
    }
    p.tiles_n = n / BN;
    p.num_tiles = (m / kBM) * p.tiles_n;
    const int num_groups = p.num_tiles / kCluster;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(CC_ERR_UNSUPPORTED, "device %d beyond the %d supported", dev, kMaxDevices);
    if ((e = device_sm_count(&sms)) != cudaSuccess) return fail_cuda(e, "SM count");
    {
        std::lock_guard<std::mutex> lock(g_attr_mutex);
        if (!attr_set[dev]) {
            e = cudaFuncSetAttribute(reinterpret_cast<const void *>(kernel),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     TileCfg<BN>::kSmemBytes);
            if (e != cudaSuccess) return fail_cuda(e, "shared memory attribute");
            attr_set[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(TileCfg<BN>::kThreads);
    cfg.dynamicSmemBytes = TileCfg<BN>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // One CTA per SM: as many clusters as the GPU holds at once (clusters
    // need their CTAs on SMs of one GPC), at most one per group.
    int clusters = sms / kCluster;
    if (kCluster > 1) {
        cfg.gridDim = dim3(static_cast<unsigned>(kCluster * clusters));
        int active = 0;
        e = cudaOccupancyMaxActiveClusters(&active, kernel, &cfg);
        if (e != cudaSuccess) return fail_cuda(e, "cluster occupancy");
        if (active > 0 && active < clusters) clusters = active;
    }
    if (max_ctas > 0 && clusters * kCluster > max_ctas) clusters = max_ctas / kCluster;
    if (clusters > num_groups) clusters = num_groups;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(kCluster * clusters));
    e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? CC_OK : fail_cuda(e, "fused tensor-parallel launch");
}

// Bytes of the tail workspace before the slots: one arrival counter per
// (split group, CTA of the pair), rounded up to 256.
size_t tail_counter_bytes(int tail_groups) {
    return (static_cast<size_t>(tail_groups) * 2 * sizeof(unsigned) + 255) / 256 * 256;
}

// The pair kernel's schedule: how many clusters run, and which groups are
// split into rank phases.  The last wave is split when its groups do not
// fill every cluster and each cluster then has at most one split phase:
// tail * R <= clusters (and R > 1).  A split phase costs far more than its
// share of the MMAs -- its product goes out in fp32 and the last of the R
// reads them all back and stores the R outputs -- so on the GPT-2 MLP
// layer (m = 8192, 4 groups left over) it gains 0.035 ms, while spreading
// 40 leftover groups over 5 phases per cluster (m = 4096) loses 0.12 ms.
struct PairPlan {
    int clusters, full_groups, tail_phases;
    size_t ws_bytes;                                     // 0: nothing split
};

template <int BN>
int pair_plan(int m, int n, int R, int max_ctas, bool split, PairPlan *plan) {
    static bool attr_set[kMaxDevices];
    using C = PairCfg<BN>;
    auto kernel = tp_fused_pair_kernel<BN>;
    const int num_groups = (m / kBM / 2) * (n / BN);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(CC_ERR_UNSUPPORTED, "device %d beyond the %d supported", dev, kMaxDevices);
    if ((e = device_sm_count(&sms)) != cudaSuccess) return fail_cuda(e, "SM count");
    {
        std::lock_guard<std::mutex> lock(g_attr_mutex);
        if (!attr_set[dev]) {
            e = cudaFuncSetAttribute(reinterpret_cast<const void *>(kernel),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::kSmemBytes);
            if (e != cudaSuccess) return fail_cuda(e, "shared memory attribute");
            attr_set[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = sms / 2;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    int active = 0;
    e = cudaOccupancyMaxActiveClusters(&active, kernel, &cfg);
    if (e != cudaSuccess) return fail_cuda(e, "cluster occupancy");
    if (active > 0 && active < clusters) clusters = active;
    if (max_ctas > 0 && 2 * clusters > max_ctas) clusters = max_ctas / 2;
    if (clusters < 1) clusters = 1;
    const int tail = num_groups % clusters;
    if (split && tail > 0 && R > 1 && tail * R <= clusters) {
        plan->full_groups = num_groups - tail;
        plan->tail_phases = tail * R;
        plan->clusters = plan->full_groups > 0 ? clusters : std::min(clusters, tail * R);
        plan->ws_bytes = tail_counter_bytes(tail) +
                         static_cast<size_t>(tail) * R * 2 * kBM * BN * sizeof(float);
    } else {
        plan->full_groups = num_groups;
        plan->tail_phases = 0;
        plan->clusters = std::min(clusters, num_groups);
        plan->ws_bytes = 0;
    }
    return CC_OK;
}

template <int BN>
int launch_pair(TpFusedParams &p, const void *const *x, const void *const *w, int m, int n,
                int kr, int R, int max_ctas, void *ws, size_t ws_bytes, cudaStream_t stream) {
    using C = PairCfg<BN>;
    int st;
    for (int r = 0; r < R; ++r) {
        if ((st = encode_bf16_map(&p.tx[r], x[r], m, kr, kBM, "x", r)) != CC_OK) return st;
        if ((st = encode_bf16_map(&p.tw[r], w[r], n, kr, C::kHalfB, "w", r)) != CC_OK) return st;
        if ((st = encode_bf16_map(&p.tout[r], p.out[r], m, n, 32, "out", r, C::kBoxCols)) !=
            CC_OK)
            return st;
    }
    p.tiles_n = n / BN;
    p.num_tiles = (m / kBM) * p.tiles_n;
    PairPlan plan;
    if ((st = pair_plan<BN>(m, n, R, max_ctas, ws != nullptr, &plan)) != CC_OK) return st;
    p.full_groups = plan.full_groups;
    p.tail_phases = plan.tail_phases;
    cudaError_t e;
    if (plan.tail_phases > 0) {
        if (ws_bytes < plan.ws_bytes)
            return fail(CC_ERR_INVALID, "workspace of %zu bytes, this shape needs %zu", ws_bytes,
                        plan.ws_bytes);
        const int tail_groups = plan.tail_phases / R;
        p.tail_count = static_cast<unsigned *>(ws);
        p.tail_ws = reinterpret_cast<float *>(static_cast<unsigned char *>(ws) +
                                              tail_counter_bytes(tail_groups));
        p.tail_ws_floats = (plan.ws_bytes - tail_counter_bytes(tail_groups)) / sizeof(float);
        e = cudaMemsetAsync(ws, 0, static_cast<size_t>(tail_groups) * 2 * sizeof(unsigned),
                            stream);
        if (e != cudaSuccess) return fail_cuda(e, "tail counters");
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * plan.clusters));
    e = cudaLaunchKernelEx(&cfg, tp_fused_pair_kernel<BN>, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? CC_OK : fail_cuda(e, "fused tensor-parallel launch");
}

#ifndef CC_TP_PAIR
#define CC_TP_PAIR 1   // 1: the pair form (cta_group::2) wherever row tiles pair up
#endif

// The cluster shape for a tile grid: pairs along M (2 x 1, sharing the W
// tile) where the row-tile count is even, else one CTA.  Measured on the
// GPT-2 MLP shape (R = 8, m = 8192, n = 3072, k = 12288, BN = 192): 1 x 1,
// 2 x 1 and 1 x 2 all 0.597 ms, 2 x 2 0.682 ms (fewer 4-CTA clusters fit at
// once than 152 / 4), so multicast halves the W tile's L2 reads at no cost
// but buys no time: one SM's operand intake, not L2, is the bound.
#if defined(CC_TP_CLUSTER_M) && defined(CC_TP_CLUSTER_N)
template <int BN>
int launch_bn(TpFusedParams &p, const void *const *x, const void *const *w, int m, int n,
              int kr, int R, int max_ctas, void *, size_t, cudaStream_t stream) {
    if ((m / kBM) % CC_TP_CLUSTER_M != 0 || (n / BN) % CC_TP_CLUSTER_N != 0)
        return launch_cfg<BN, 1, 1>(p, x, w, m, n, kr, R, max_ctas, stream);
    return launch_cfg<BN, CC_TP_CLUSTER_M, CC_TP_CLUSTER_N>(p, x, w, m, n, kr, R, max_ctas,
                                                            stream);
}
#else
template <int BN>
int launch_bn(TpFusedParams &p, const void *const *x, const void *const *w, int m, int n,
              int kr, int R, int max_ctas, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if ((m / kBM) % 2 == 0) {
        if (CC_TP_PAIR)
            return launch_pair<BN>(p, x, w, m, n, kr, R, max_ctas, ws, ws_bytes, stream);
        return launch_cfg<BN, 2, 1>(p, x, w, m, n, kr, R, max_ctas, stream);
    }
    return launch_cfg<BN, 1, 1>(p, x, w, m, n, kr, R, max_ctas, stream);
}
#endif

// The single-CTA kernel's tile width for n output columns: 192 (16 column
// tiles for n = 3072), then 256, then 128.  The pair kernel's is chosen by
// pick_pair_bn.
int pick_bn(int n, bool) {
#ifdef CC_TP_BN
    return n % CC_TP_BN == 0 ? CC_TP_BN : 0;
#else
    return n % 192 == 0 ? 192 : n % 256 == 0 ? 256 : n % 128 == 0 ? 128 : 0;
#endif
}

// The pair kernel's modelled time at tile width BN: its waves (a split last
// wave counted as half) times one wave's operand intake per CTA and k-block,
// X 128 x 64 plus half of W (BN/2 x 64) in bf16 = 16384 + 64 BN bytes.  One
// SM's operand intake bounds a wave, so this ranks the widths: on the GPT-2
// MLP layer (R = 8, n = 3072, k = 12288) it picks 256 at m = 4096 and 8192
// (measured 0.228 / 0.4155 ms against 0.264 / 0.457 at 192) and 192 at
// m = 2048 (0.137 against 0.154), where both widths take two waves.
template <int BN>
int pair_cost(int m, int n, int R, int max_ctas, bool split, double *cost) {
    *cost = -1.0;
    if (n % BN != 0) return CC_OK;
    PairPlan plan;
    const int st = pair_plan<BN>(m, n, R, max_ctas, split, &plan);
    if (st != CC_OK) return st;
    const int full_waves = plan.full_groups / plan.clusters;
    const double waves = full_waves + (plan.tail_phases > 0 ? 0.5
                                       : plan.full_groups % plan.clusters ? 1.0 : 0.0);
    *cost = waves * (16384.0 + 64.0 * BN);
    return CC_OK;
}

// The pair kernel's tile width for this shape and budget (0: n fits none).
int pick_pair_bn(int m, int n, int R, int max_ctas, bool split, int *bn) {
#ifdef CC_TP_BN
    (void)m; (void)R; (void)max_ctas; (void)split;
    *bn = n % CC_TP_BN == 0 ? CC_TP_BN : 0;
    return CC_OK;
#else
    double c256, c192, c128;
    int st;
    if ((st = pair_cost<256>(m, n, R, max_ctas, split, &c256)) != CC_OK) return st;
    if ((st = pair_cost<192>(m, n, R, max_ctas, split, &c192)) != CC_OK) return st;
    if ((st = pair_cost<128>(m, n, R, max_ctas, split, &c128)) != CC_OK) return st;
    *bn = 0;
    double best = 0.0;
    const int widths[3] = {256, 192, 128};
    const double costs[3] = {c256, c192, c128};
    for (int i = 0; i < 3; ++i)
        if (costs[i] >= 0.0 && (*bn == 0 || costs[i] < best)) {
            *bn = widths[i];
            best = costs[i];
        }
    return CC_OK;
#endif
}

}  // namespace

int launch_tp_fused(const void *const *x, const void *const *w, void *const *out,
                    float *const *partials, int m, int n, int k, int R, int max_ctas,
                    void *ws, size_t ws_bytes, cudaStream_t stream) {
    TpFusedParams p{};
    const int kr = k / R;
    for (int r = 0; r < R; ++r) {
        p.out[r] = static_cast<__nv_bfloat16 *>(out[r]);
        p.partials[r] = partials ? partials[r] : nullptr;
    }
    p.R = R;
    p.m = m;
    p.n = n;
    p.kb_per_rank = kr / kBK;
    const bool pair = CC_TP_PAIR && (m / kBM) % 2 == 0;
    int bn = pick_bn(n, false);
    if (pair) {
        const int st = pick_pair_bn(m, n, R, max_ctas, ws != nullptr, &bn);
        if (st != CC_OK) return st;
    }
    switch (bn) {
        case 128: return launch_bn<128>(p, x, w, m, n, kr, R, max_ctas, ws, ws_bytes, stream);
        case 192: return launch_bn<192>(p, x, w, m, n, kr, R, max_ctas, ws, ws_bytes, stream);
        case 256: return launch_bn<256>(p, x, w, m, n, kr, R, max_ctas, ws, ws_bytes, stream);
        default: return fail(CC_ERR_INVALID, "n=%d is not a multiple of 128 or 192", n);
    }
}

bool tp_fused_shape_ok(int m, int n, int kr) {
    return m % kBM == 0 && kr % kBK == 0 && pick_bn(n, false) != 0;
}

int tp_fused_workspace(int m, int n, int R, int max_ctas, size_t *bytes) {
    *bytes = 0;
    if (!CC_TP_PAIR || (m / kBM) % 2 != 0) return CC_OK;   // the single-CTA kernel
    PairPlan plan;
    int bn = 0;
    int st = pick_pair_bn(m, n, R, max_ctas, true, &bn);
    if (st != CC_OK) return st;
    switch (bn) {
        case 128: st = pair_plan<128>(m, n, R, max_ctas, true, &plan); break;
        case 192: st = pair_plan<192>(m, n, R, max_ctas, true, &plan); break;
        case 256: st = pair_plan<256>(m, n, R, max_ctas, true, &plan); break;
        default: return fail(CC_ERR_INVALID, "n=%d is not a multiple of 128 or 192", n);
    }
    if (st == CC_OK) *bytes = plan.ws_bytes;
    return st;
}


cudaError_t read_tp_status(unsigned *status, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_tp_status, sizeof(unsigned));
    if (e == cudaSuccess && clear) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_tp_status, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace ccdp

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

namespace {

struct Span {
    uintptr_t lo, hi;
    bool written;
    const char *name;
    int index;
};

}  // namespace

namespace {

int tp_check_shape(int m, int n, int k, int R) {
    using namespace ccdp;
    if (R < 1 || R > CC_MAX_R) return fail(CC_ERR_INVALID, "R=%d must be in 1..%d", R, CC_MAX_R);
    if (m <= 0 || n <= 0 || k <= 0) return fail(CC_ERR_INVALID, "m, n, k must be > 0");
    if (k % R != 0) return fail(CC_ERR_INVALID, "k=%d is not a multiple of R=%d", k, R);
    const int kr = k / R;
    if (!tp_fused_shape_ok(m, n, kr))
        return fail(CC_ERR_INVALID,
                    "shape m=%d n=%d k/R=%d: needs m %% 128 == 0, n a multiple of 128 or "
                    "192, and k/R %% 64 == 0", m, n, kr);
    return CC_OK;
}

}  // namespace

extern "C" int cc_tp_matmul_allreduce_workspace(int m, int n, int k, int R, int max_ctas,
                                                size_t *bytes) {
    using namespace ccdp;
    if (!bytes) return fail(CC_ERR_INVALID, "bytes is NULL");
    *bytes = 0;
    if (max_ctas < 0) return fail(CC_ERR_INVALID, "max_ctas=%d must be >= 0", max_ctas);
    if (max_ctas == 1) return fail(CC_ERR_INVALID, "max_ctas=1: the kernel runs CTA pairs");
    int st;
    if ((st = tp_check_shape(m, n, k, R)) != CC_OK) return st;
    if ((st = ensure_device()) != CC_OK) return st;
    return tp_fused_workspace(m, n, R, max_ctas, bytes);
}

extern "C" int cc_tp_matmul_allreduce_ex(const void *const *x, const void *const *w,
                                         void *const *out, float *const *partials, int m,
                                         int n, int k, int R, void *workspace,
                                         size_t workspace_bytes, int max_ctas, void *stream) {
    using namespace ccdp;
    TraceRange call("cc_tp_matmul_allreduce", static_cast<uint64_t>(m));
    int st;
    if ((st = tp_check_shape(m, n, k, R)) != CC_OK) return st;
    if (max_ctas < 0) return fail(CC_ERR_INVALID, "max_ctas=%d must be >= 0", max_ctas);
    if (max_ctas == 1) return fail(CC_ERR_INVALID, "max_ctas=1: the kernel runs CTA pairs");
    if (!x || !w || !out) return fail(CC_ERR_INVALID, "x/w/out arrays are NULL");
    const int kr = k / R;
    const size_t mn = static_cast<size_t>(m) * n;
    std::vector<Span> spans;
    auto add = [&](const void *ptr, size_t bytes, bool written, const char *name, int r) {
        if (!ptr) return fail(CC_ERR_INVALID, "%s[%d] is NULL", name, r);
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
            return fail(CC_ERR_MISALIGNED, "%s[%d]=%p is not 16-byte aligned", name, r, ptr);
        const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
        spans.push_back({lo, lo + bytes, written, name, r});
        return static_cast<int>(CC_OK);
    };
    for (int r = 0; r < R; ++r) {
        if ((st = add(x[r], 2 * static_cast<size_t>(m) * kr, false, "x", r)) != CC_OK) return st;
        if ((st = add(w[r], 2 * static_cast<size_t>(n) * kr, false, "w", r)) != CC_OK) return st;
        if ((st = add(out[r], 2 * mn, true, "out", r)) != CC_OK) return st;
        if (partials && (st = add(partials[r], 4 * mn, true, "partials", r)) != CC_OK)
            return st;
    }
    if (workspace && workspace_bytes > 0 &&
        (st = add(workspace, workspace_bytes, true, "workspace", 0)) != CC_OK)
        return st;
    for (size_t i = 0; i < spans.size(); ++i)
        for (size_t j = i + 1; j < spans.size(); ++j)
            if ((spans[i].written || spans[j].written) && spans[i].lo < spans[j].hi &&
                spans[j].lo < spans[i].hi)
                return fail(CC_ERR_ALIAS, "%s[%d] overlaps %s[%d]", spans[i].name,
                            spans[i].index, spans[j].name, spans[j].index);
    if ((st = ensure_device()) != CC_OK) return st;
    for (const Span &sp : spans)
        if ((st = check_device_range(reinterpret_cast<const void *>(sp.lo), sp.hi - sp.lo,
                                     sp.name)) != CC_OK)
            return st;
    return launch_tp_fused(x, w, out, partials, m, n, k, R, max_ctas,
                           workspace_bytes > 0 ? workspace : nullptr, workspace_bytes,
                           static_cast<cudaStream_t>(stream));
}

extern "C" int cc_tp_matmul_allreduce(const void *const *x, const void *const *w,
                                      void *const *out, float *const *partials, int m, int n,
                                      int k, int R, void *stream) {
    return cc_tp_matmul_allreduce_ex(x, w, out, partials, m, n, k, R, nullptr, 0, 0, stream);
}
