// fwd_pair_sm103.cu -- the forward (prefill) kernel on CTA pairs: tcgen05
// MMAs of the cta_group::2 kind, M = 256, issued by one warp for two SMs.
//
// Same computation as fwd_sm103.cu -- O = softmax(scale * Q K^T) V and lse
// per query row ("Optimizing Attention on GPUs by Exploiting GPU
// Architectural NUMA Effects", detail page, section 4 equation), FA2
// partitioning (Figure 4) and the online softmax with running (m, l, O)
// (kernbench2 "Fused Grouped-Query Attention", short-context section) -- with
// the work of two SMs fused into one MMA stream.  The pages place the
// workgroups that share one head's K/V on one chiplet (detail page, section 2
// Q1-Q2); here the two CTAs of a cluster (one GPC) share every K/V block
// through the pair MMA instead of each loading it.
//
// A cluster of two CTAs (ranks 0 and 1) owns a unit of 512 query rows of one
// head.  Pair tile t (t = 0, 1) is rows [256 t, 256 t + 256) of the unit;
// CTA c holds rows [256 t + 128 c, +128) of it in shared memory (Q) and in
// its tensor memory (S/P and O).  Per 128-key block j:
//   S(t) = Q(t) K_j^T   M = 256, N = 128, K = d: each CTA supplies its 128
//                        query rows (A) and 64 of the 128 keys (B); each
//                        CTA's TMEM receives its rows' scores for all keys;
//   O(t) += P(t) V_j    M = 256, N = d, K = 128: P from each CTA's TMEM (A),
//                        each CTA supplies d/2 of V's columns (B); each CTA's
//                        TMEM receives its rows' O for all d columns.
// So each SM loads half of every K/V block (16 KiB of K, 16 KiB of V at
// d = 128) and the pair's MMA warp issues one instruction per 256 rows.
//
// Roles (384 threads per CTA, as in the one-CTA kernel):
//   warp 0      TMA producer of this CTA's halves (both CTAs).  Copies complete
//               on the rank-0 CTA's barriers (the .cta_group::2 form of the
//               tensor copy), which count both halves' bytes.
//   warp 1      rank 0: the MMA warp of the pair (the whole warp runs the loop,
//               an elected lane issues); rank 1: TMEM only.
//   warps 4-11  softmax / epilogue of this CTA's rows of pair tiles 0 and 1.
// Rank 0 fetches the units and hands them to rank 1 through its shared
// memory.  The MMA warp's commits arrive on both CTAs' barriers
// (multicast); the softmax warps of both CTAs hand P to the MMA warp on
// rank 0's barriers.  Every wait is bounded in time; a wait that gives up
// sets both CTAs' abort flags.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.h"
#include "sm103_ptx.cuh"
#include "tile_order.cuh"

namespace attn {

static __device__ int g_fwd_pair_status;

// Work counters, one slot per launch as in the one-CTA kernel ({next unit
// (die 0), next unit of die 1, CTAs finished, unused}), in an array of their
// own: the two kernels never share a slot.
constexpr int kPairSchedSlots = 64;
constexpr int kPairWorkDone = 2;
static __device__ unsigned int g_fwd_pair_work[kPairSchedSlots][4];
static std::atomic<unsigned int> g_fwd_pair_launch_seq{0};

namespace fwd2 {

constexpr int D = 128;
constexpr int kTileM = 128;           // query rows of a pair tile held by one CTA
constexpr int kUnitRowsPair = 512;    // query rows of one pair unit
constexpr int kBlockN = 128;          // keys per K/V block
constexpr int kNT = 2;                // pair tiles per unit
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 120;  // the warp-wide MMA issue loop spills at 104
constexpr int kSoftmaxRegs = 192;
static_assert(128 * kCtrlRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kTmemCols = 512;
constexpr int kChunks = D / 64;                 // 128-byte column chunks of a Q or K row
constexpr int kQChunkBytes = kTileM * 128;      // 128 rows x 128 bytes
constexpr int kQBytes = kTileM * D * 2;         // one CTA's rows of one pair tile
constexpr int kKChunkBytes = (kBlockN / 2) * 128;  // 64 keys x 128 bytes
constexpr int kHalfBytes = kBlockN * D;         // 16 KiB: half a K block or half a V block
constexpr int kStages = 8;                      // ring slots (K and V halves alternate)
constexpr int kOCol = 2 * kTileM;               // first O column in TMEM
// barriers (same offsets in both CTAs; "r0" = waited on in rank 0 only)
constexpr int kBarQFull = 0,          // [2] r0: both CTAs' Q halves landed
    kBarQEmpty = 2,                   // [2] both: Q buffer free (MMA commit, multicast)
    kBarSFull = 4,                    // [2] both: S ready (multicast)
    kBarPFull = 6,                    // [2] r0: P written by the 8 softmax warps of the pair
    kBarOFull = 8,                    // [2] both: O final (multicast)
    kBarOEmpty = 10,                  // [2] r0: O read by the 8 epilogue warps of the pair
    kBarKVFull = 12,                  // [S] r0: both halves of a ring fill landed
    kBarKVEmpty = 12 + kStages,       // [S] both: this CTA's half of the slot free
    kBarDrain = 12 + 2 * kStages,     // r0: every MMA complete (teardown)
    kBarUQFull = 13 + 2 * kStages,    // [2] both: unit queue entry written
    kBarUQEmpty = 15 + 2 * kStages,   // [2] r0: entry read by every role of the pair
    kNumBars = 17 + 2 * kStages;
constexpr int kUQConsumers = 2 * (1 + 8);  // per CTA: producer or MMA warp, and 8 softmax warps
constexpr int kDataBytes = kNT * kQBytes + kStages * kHalfBytes;
constexpr int kSmemBytes = kDataBytes + kNumBars * 8 + 32 + 1024;
constexpr uint16_t kBothCtas = 0x3;

struct Params {
    __nv_bfloat16 *o;
    float *lse;
    int B, N, Hq, Hkv, G, d_store, causal, order, nb;  // nb: pair units per head
    long long total_units;
    float scale_log2;
    unsigned long long wait_ns;
    int sched_slot;
    const int *die_of_sm;
};

struct UnitWork {
    int b, h, kvh;
    int row0[kNT];  // first row of pair tile t
    int nkv[kNT];   // K/V blocks pair tile t visits (0: it lies past N)
    int nmax;
};

template <bool kGrouped>
__device__ __forceinline__ UnitWork unit_work(const Params &p, long long u) {
    const Tile t = kGrouped ? unit_to_tile_grouped_causal(u, p.Hq, p.G, p.nb)
                            : unit_to_tile(p.order, u, p.Hq, p.nb, p.causal);
    UnitWork w;
    w.b = t.b;
    w.h = t.h;
    w.kvh = t.h / p.G;
    const int nkv_all = (p.N + kBlockN - 1) / kBlockN;
    w.nmax = 0;
#pragma unroll
    for (int tt = 0; tt < kNT; ++tt) {
        const int r0 = t.m * kUnitRowsPair + tt * 2 * kTileM;
        w.row0[tt] = r0;
        int n = 0;
        // causal: up to the block of the pair tile's last row (rank 1's rows);
        // rank 0 sees that block fully masked
        if (r0 < p.N) n = p.causal ? min(nkv_all, min(r0 + 2 * kTileM - 1, p.N - 1) / kBlockN + 1) : nkv_all;
        w.nkv[tt] = n;
        w.nmax = max(w.nmax, n);
    }
    return w;
}

__device__ __forceinline__ long long fetch_unit(const Params &p, long long i, int my_die) {
    if (p.order == kNaiveHeadFirst) return i == 0 ? (long long)(blockIdx.x >> 1) : -1;
    if (p.order == kDieSplitHeadFirst) {
        for (int s = 0; s < kDies; ++s) {
            const int die = (my_die + s) % kDies;
            const unsigned int k = atomicAdd(&g_fwd_pair_work[p.sched_slot][die], 1u);
            const long long u = die_split_unit(die, (long long)k, p.B, p.Hkv, p.G, p.nb);
            if (u >= 0) return u;
        }
        return -1;
    }
    const unsigned int u = atomicAdd(&g_fwd_pair_work[p.sched_slot][0], 1u);
    return (long long)u < p.total_units ? (long long)u : -1;
}

__device__ __forceinline__ int last_user(const UnitWork &w, int j) {
    int last = -1;
#pragma unroll
    for (int t = 0; t < kNT; ++t)
        if (j < w.nkv[t]) last = t;
    return last;
}

// ------------------------------------------------------ cluster primitives
__device__ __forceinline__ uint32_t cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void store_remote(uint32_t cluster_addr, int v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool test_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Tensor copy of this CTA's half, completing on a barrier of the rank-0 CTA
// (cluster address): the .cta_group::2 form lets the barrier sit in the peer.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrive on the barrier at this offset in both CTAs once every pair MMA
// issued so far by this thread is complete.
__device__ __forceinline__ void commit_both(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(kBothCtas)
        : "memory");
}
// The same, on this CTA's barrier only.
__device__ __forceinline__ void commit_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void mma_ss_x4_pair(uint32_t d, const uint64_t (&a)[4], const uint64_t (&b)[4],
                                               uint32_t idesc, uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p0, p1;\n\t"
        "setp.ne.b32 p0, %9, 0;\n\t"
        "setp.eq.b32 p1, %9, %9;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %5, %10, p0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %2, %6, %10, p1;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %3, %7, %10, p1;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %4, %8, %10, p1;\n\t}" ::"r"(d),
        "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(acc0),
        "r"(idesc)
        : "memory");
}
__device__ __forceinline__ void mma_ts_x4_pair(uint32_t d, const uint32_t (&a)[4], const uint64_t (&b)[4],
                                               uint32_t idesc, uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p0, p1;\n\t"
        "setp.ne.b32 p0, %9, 0;\n\t"
        "setp.eq.b32 p1, %9, %9;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %5, %10, p0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%2], %6, %10, p1;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%3], %7, %10, p1;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%4], %8, %10, p1;\n\t}" ::"r"(d),
        "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(acc0),
        "r"(idesc)
        : "memory");
}

// Warp-collective forms of the above: all 32 lanes execute them and the lane
// that elect.sync picks (the lowest, the same one every time) issues.
__device__ __forceinline__ void commit_both_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}"
        ::"r"(bar), "h"(kBothCtas)
        : "memory");
}
__device__ __forceinline__ void commit_local_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void mma_ss_x4_pair_elect(uint32_t d, const uint64_t (&a)[4], const uint64_t (&b)[4],
                                                     uint32_t idesc, uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p0, p1, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %9, 0;\n\t"
        "setp.eq.b32 p1, %9, %9;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %5, %10, p0;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %2, %6, %10, p1;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %3, %7, %10, p1;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %4, %8, %10, p1;\n\t}" ::"r"(d),
        "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(acc0),
        "r"(idesc)
        : "memory");
}
__device__ __forceinline__ void mma_ts_x4_pair_elect(uint32_t d, const uint32_t (&a)[4], const uint64_t (&b)[4],
                                                     uint32_t idesc, uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p0, p1, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %9, 0;\n\t"
        "setp.eq.b32 p1, %9, %9;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %5, %10, p0;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%2], %6, %10, p1;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%3], %7, %10, p1;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%4], %8, %10, p1;\n\t}" ::"r"(d),
        "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(acc0),
        "r"(idesc)
        : "memory");
}

// Bounded waits of the pair kernel: as mbar_wait_bounded / mbar_wait_warp
// (sm103_ptx.cuh) with cluster-scope acquire (some arrivals come from the
// other CTA); on giving up they also set the other CTA's abort flag, so the
// pair leaves together.
struct PairAbort {
    volatile int *local;
    uint32_t peer_flag;  // cluster address of the other CTA's flag
    int *status;
    __device__ __forceinline__ void raise() const {
        *local = 1;
        store_remote(peer_flag, 1);
        atomicOr(status, kStatusTimeout);
    }
};

__device__ __forceinline__ bool wait_pair(uint32_t bar, uint32_t parity, uint64_t limit_ns, const PairAbort &ab) {
    if (limit_ns == 0) {
        if (test_wait_cluster(bar, parity)) return true;
        ab.raise();
        return false;
    }
    if (try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (try_wait_cluster(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (*ab.local) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                ab.raise();
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_pair_warp(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                               const PairAbort &ab) {
    if (limit_ns == 0) {
        if (__all_sync(0xffffffffu, test_wait_cluster(bar, parity))) return true;
        if ((threadIdx.x & 31) == 0) ab.raise();
        __syncwarp();
        return false;
    }
    bool done = try_wait_cluster(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (!done) done = try_wait_cluster(bar, parity);
        if (__all_sync(0xffffffffu, done)) return true;
        if ((it & 15u) == 0) {
            int give_up = 0;
            if ((threadIdx.x & 31) == 0) {
                if (*ab.local) {
                    give_up = 1;
                } else if (global_timer_ns() - t0 > limit_ns) {
                    ab.raise();
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
    }
}

// Spin for `ns` nanoseconds (the teardown grace period of a producer whose
// copies complete on the other CTA's barriers).
__device__ __forceinline__ void spin_ns(uint64_t ns) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) {
    }
}

template <bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sQ = smem;
    uint8_t *sKV = smem + kNT * kQBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kDataBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *unit_q = reinterpret_cast<volatile int *>(tmem_slot + 2);  // 2 entries

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cta_rank();
    auto bar = [&](int i) { return smem_u32(bars + i); };
    // rank 0's copy of barrier i (a cluster address; rank 0's own address on rank 0)
    auto bar0 = [&](int i) { return map_to(smem_u32(bars + i), 0); };

    if (threadIdx.x == 0) {
        for (int t = 0; t < kNT; ++t) {
            mbar_init(bar(kBarQFull + t), 1);
            mbar_init(bar(kBarQEmpty + t), 1);
            mbar_init(bar(kBarSFull + t), 1);
            mbar_init(bar(kBarPFull + t), 8);   // 4 softmax warps of each CTA
            mbar_init(bar(kBarOFull + t), 1);
            mbar_init(bar(kBarOEmpty + t), 8);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarKVFull + s), 1);
            mbar_init(bar(kBarKVEmpty + s), 1);
        }
        mbar_init(bar(kBarDrain), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarUQFull + i), 1);
            mbar_init(bar(kBarUQEmpty + i), kUQConsumers);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);  // one warp of each CTA, together
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int *status = &g_fwd_pair_status;
    const PairAbort ab{abort_flag, map_to(smem_u32(const_cast<int *>(abort_flag)), rank ^ 1u), status};

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
      if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            long long fills = 0;
            int q_loads[kNT] = {0, 0};
            bool ok = true;
            int my_die = 0;
            if (p.die_of_sm && rank == 0) {
                uint32_t smid;
                asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
                if (smid < uint32_t(kDieMapMaxSms)) my_die = p.die_of_sm[smid] & 1;
            }
            const uint32_t uq_peer = map_to(smem_u32(const_cast<int *>(unit_q)), 1);
            for (long long qi = 0; ok; ++qi) {
                const int qs = int(qi & 1);
                long long u;
                if (rank == 0) {
                    u = fetch_unit(p, qi, my_die);
                    if (qi >= 2 && !wait_pair(bar(kBarUQEmpty + qs), uint32_t(((qi >> 1) - 1) & 1), p.wait_ns, ab)) {
                        ok = false;
                        break;
                    }
                    unit_q[qs] = int(u);
                    store_remote(uq_peer + 4u * qs, int(u));
                    mbar_arrive(bar(kBarUQFull + qs));
                    arrive_remote(map_to(bar(kBarUQFull + qs), 1));
                } else {
                    if (!wait_pair(bar(kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns, ab)) {
                        ok = false;
                        break;
                    }
                    u = unit_q[qs];
                    arrive_remote(bar0(kBarUQEmpty + qs));
                }
                if (u < 0) break;
                const UnitWork w = unit_work<kGrouped>(p, u);
                for (int t = 0; t < kNT && ok; ++t) {
                    if (w.nkv[t] == 0) continue;
                    if (q_loads[t] > 0)
                        ok = wait_pair(bar(kBarQEmpty + t), (q_loads[t] - 1) & 1, p.wait_ns, ab);
                    if (!ok) break;
                    if (rank == 0) mbar_arrive_expect_tx(bar(kBarQFull + t), 2 * kQBytes);
                    const uint32_t qb = bar0(kBarQFull + t);
                    const int row = w.row0[t] + int(rank) * kTileM;
                    for (int c = 0; c < kChunks; ++c)
                        tma_load_3d_pair(smem_u32(sQ + t * kQBytes + c * kQChunkBytes), &tmQ, qb, c * 64, row,
                                         w.b * p.Hq + w.h);
                    ++q_loads[t];
                }
                for (int j = 0; ok && j < w.nmax; ++j) {
                    for (int kv = 0; kv < 2; ++kv) {
                        const int slot = int(fills % kStages);
                        const long long round = fills / kStages;
                        if (round > 0) {
                            ok = wait_pair(bar(kBarKVEmpty + slot), uint32_t((round - 1) & 1), p.wait_ns, ab);
                            if (!ok) break;
                        }
                        if (rank == 0) mbar_arrive_expect_tx(bar(kBarKVFull + slot), 2 * kHalfBytes);
                        const uint32_t fb = bar0(kBarKVFull + slot);
                        const uint32_t dst = smem_u32(sKV + slot * kHalfBytes);
                        const int plane = w.b * p.Hkv + w.kvh;
                        if (kv == 0) {
                            // K: keys [128 j + 64 rank, +64), all d columns
                            for (int c = 0; c < kChunks; ++c)
                                tma_load_3d_pair(dst + c * kKChunkBytes, &tmK, fb, c * 64,
                                                 j * kBlockN + int(rank) * (kBlockN / 2), plane);
                        } else {
                            // V: all 128 keys, d columns [64 rank, +64)
                            tma_load_3d_pair(dst, &tmV, fb, int(rank) * 64, j * kBlockN, plane);
                        }
                        ++fills;
                    }
                }
            }
            if (!ok) {
                // Rank 0 waits (bounded) for the fills and Q loads it armed; a
                // half the other CTA never sent leaves its phase open, so these
                // waits are short.  Rank 1's copies complete on rank 0's
                // barriers, out of its sight: it gives them a grace period.
                // Either way no copy is still writing shared memory when the
                // pair passes the final cluster barrier.
                volatile int no_abort = 0;
                if (rank == 0) {
                    const unsigned long long drain_ns = 2000000ull;
                    for (int s = 0; s < kStages; ++s) {
                        long long last = fills - 1 - ((fills - 1 - s) % kStages + kStages) % kStages;
                        if (fills == 0 || last < 0) continue;
                        if (!mbar_wait_bounded(bar(kBarKVFull + int(last % kStages)),
                                               uint32_t((last / kStages) & 1), drain_ns, &no_abort, status))
                            atomicOr(status, kStatusDrainTimeout);
                    }
                    for (int t = 0; t < kNT; ++t)
                        if (q_loads[t] > 0 && !mbar_wait_bounded(bar(kBarQFull + t), (q_loads[t] - 1) & 1,
                                                                 drain_ns, &no_abort, status))
                            atomicOr(status, kStatusDrainTimeout);
                } else {
                    spin_ns(2000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        // Rank 0's whole warp runs the issue loop (its state is warp-uniform);
        // each MMA, commit and arrival goes out from one elected lane.
        if (rank == 0) {
            constexpr uint32_t kIdescQK = idesc_bf16_f32(2 * kTileM, kBlockN, 0);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(2 * kTileM, D, 1);
            long long fills = 0;
            int q_used[kNT] = {0, 0};
            int p_waits[kNT] = {0, 0};
            int units_done[kNT] = {0, 0};
            bool ok = true;

            auto wait_slot = [&](long long f) {
                return wait_pair_warp(bar(kBarKVFull + int(f % kStages)), uint32_t((f / kStages) & 1), p.wait_ns, ab);
            };
            const uint64_t dQ = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dK = smem_desc_sw128(smem_u32(sKV), 16, 1024);
            const uint64_t dV = smem_desc_sw128(smem_u32(sKV), kHalfBytes, 1024);
            auto slot_off = [&](long long f) { return uint64_t(int(f % kStages) * (kHalfBytes >> 4)); };
            auto issue_qk = [&](int t, long long fK) {
                const uint64_t a0 = dQ + uint64_t(t * (kQBytes >> 4));
                const uint64_t b0 = dK + slot_off(fK);
                const uint32_t d_tmem = tmem_base + t * kTileM;
#pragma unroll
                for (int g = 0; g < kChunks; ++g) {
                    uint64_t a[4], b[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        a[i] = a0 + uint64_t((g * kQChunkBytes + i * 32) >> 4);
                        b[i] = b0 + uint64_t((g * kKChunkBytes + i * 32) >> 4);
                    }
                    mma_ss_x4_pair_elect(d_tmem, a, b, kIdescQK, g > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, long long fV, bool acc) {
                const uint64_t b0 = dV + slot_off(fV);
                const uint32_t d_tmem = tmem_base + kOCol + t * D;
                const uint32_t a_tmem = tmem_base + t * kTileM;
#pragma unroll
                for (int g = 0; g < kBlockN / 64; ++g) {
                    uint32_t a[4];
                    uint64_t b[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int kk = g * 4 + i;
                        a[i] = a_tmem + kk * 8;
                        b[i] = b0 + uint64_t((kk * 16 * 128) >> 4);
                    }
                    mma_ts_x4_pair_elect(d_tmem, a, b, kIdescPV, (acc || g > 0) ? 1u : 0u);
                }
            };

            for (long long qi = 0; ok; ++qi) {
                const int qs = int(qi & 1);
                ok = wait_pair_warp(bar(kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns, ab);
                if (!ok) break;
                const long long u = __shfl_sync(0xffffffffu, int(unit_q[qs]), 0);
                mbar_arrive_elect(bar(kBarUQEmpty + qs));
                if (u < 0) break;
                const UnitWork w = unit_work<kGrouped>(p, u);
                const long long f0 = fills;
                ok = wait_slot(f0);
                for (int t = 0; ok && t < kNT; ++t) {
                    if (w.nkv[t] == 0) continue;
                    ok = wait_pair_warp(bar(kBarQFull + t), q_used[t] & 1, p.wait_ns, ab);
                    if (!ok) break;
                    ++q_used[t];
                    tc_fence_after();
                    issue_qk(t, f0);
                    commit_both_elect(bar(kBarSFull + t));
                }
                for (int j = 0; ok && j < w.nmax; ++j) {
                    const long long fV = f0 + 2 * j + 1, fK = f0 + 2 * j + 2;
                    bool v_ready = false, k_ready = false;
                    for (int t = 0; ok && t < kNT; ++t) {
                        if (j >= w.nkv[t]) continue;
                        ok = wait_pair_warp(bar(kBarPFull + t), p_waits[t] & 1, p.wait_ns, ab);
                        if (!ok) break;
                        ++p_waits[t];
                        if (j == 0 && units_done[t] > 0) {
                            ok = wait_pair_warp(bar(kBarOEmpty + t), (units_done[t] - 1) & 1, p.wait_ns, ab);
                            if (!ok) break;
                        }
                        if (!v_ready) {
                            ok = wait_slot(fV);
                            if (!ok) break;
                            v_ready = true;
                        }
                        tc_fence_after();
                        issue_pv(t, fV, j > 0);
                        if (t == last_user(w, j)) commit_both_elect(bar(kBarKVEmpty + int(fV % kStages)));
                        if (j + 1 < w.nkv[t]) {
                            if (!k_ready) {
                                ok = wait_slot(fK);
                                if (!ok) break;
                                k_ready = true;
                            }
                            issue_qk(t, fK);
                            commit_both_elect(bar(kBarSFull + t));
                        } else {
                            commit_both_elect(bar(kBarOFull + t));
                            commit_both_elect(bar(kBarQEmpty + t));
                            ++units_done[t];
                        }
                    }
                }
                fills = f0 + 2 * (long long)w.nmax;
            }
            commit_local_elect(bar(kBarDrain));
            volatile int no_abort = 0;
            if (!mbar_wait_warp(bar(kBarDrain), 0, 1000000000ull, &no_abort, status) && lane == 0)
                atomicOr(status, kStatusDrainTimeout);
        }
        __syncwarp();
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
        // ------------------------------------------------- softmax / epilogue
        const int t = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        const uint32_t tS = tmem_base + lane_off + t * kTileM;
        const uint32_t tO = tmem_base + lane_off + kOCol + t * D;
        const float sl2 = p.scale_log2;
        int s_waits = 0, o_waits = 0;
        long long kv_base = 0;
        const bool frees_slots = (quarter == 0 && lane == 0);
        // rank 0's P-full, O-empty and unit-queue-empty barriers
        const uint32_t p_full = bar0(kBarPFull + t), o_empty = bar0(kBarOEmpty + t);
        bool ok = true;

        for (long long qi = 0; ok; ++qi) {
            const int qs = int(qi & 1);
            ok = wait_pair_warp(bar(kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns, ab);
            if (!ok) break;
            const long long u = unit_q[qs];
            __syncwarp();
            if (lane == 0) arrive_remote(bar0(kBarUQEmpty + qs));
            if (u < 0) break;
            const UnitWork w = unit_work<kGrouped>(p, u);
            const long long f0 = kv_base;
            kv_base += 2 * (long long)w.nmax;
            const int nkv = w.nkv[t];
            if (nkv == 0) continue;
            const int row0 = w.row0[t] + int(rank) * kTileM;  // this CTA's first row of pair tile t
            const int row = row0 + r;
            float m_run = -INFINITY, l_run = 0.f;

            for (int j = 0; j < nkv; ++j) {
                ok = wait_pair_warp(bar(kBarSFull + t), s_waits & 1, p.wait_ns, ab);
                if (!ok) break;
                ++s_waits;
                // this CTA's K half of block j is free once S(t, j) is complete
                if (frees_slots && t == last_user(w, j))
                    mbar_arrive(bar(kBarKVEmpty + int((f0 + 2 * j) % kStages)));
                tc_fence_after();
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
                tmem_wait_ld();
                float s[128];
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(sr[c][i]);

                const int kv0 = j * kBlockN;
                const bool ragged = kv0 + kBlockN > p.N;
                const bool diag = p.causal && (kv0 + kBlockN - 1 > row0);
                if (ragged || diag) {
                    int lim = p.N - kv0;
                    if (p.causal) lim = min(lim, row + 1 - kv0);
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                auto block_max = [&]() {
                    float mq[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float m = fmax3(s[32 * c], s[32 * c + 1], s[32 * c + 2]);
#pragma unroll
                        for (int i = 3; i < 31; i += 2) m = fmax3(m, s[32 * c + i], s[32 * c + i + 1]);
                        mq[c] = fmaxf(m, s[32 * c + 31]);
                    }
                    return fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
                };
                auto exp_block = [&](float neg_m) {
                    float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float x0, x1;
                            ffma2(x0, x1, s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1], sl2, sl2, neg_m, neg_m);
                            const float p0 = fast_exp2(x0);
                            const float p1 = fast_exp2(x1);
                            const int a = (i & 3) * 2;
                            fadd2(ls[a], ls[a + 1], p0, p1);
                            pk[i] = pack_bf16x2(p0, p1);
                        }
                        tmem_st16(tS + c * 16, pk);
                    }
                    return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                };
                // Kept reference maximum with the 2^60 block-sum guard, as in the
                // one-CTA kernel.  Rank 0's rows of a causal pair tile see their last
                // block fully masked; their maximum is finite by then (block 0 is
                // never fully masked), so that block's exponentials are all 0.
                float corr = 1.f;
                if (m_run == -INFINITY) m_run = block_max() * sl2;
                float l_blk = exp_block(m_run == -INFINITY ? 0.f : -m_run);
                if (__any_sync(0xffffffffu, !(l_blk < 0x1p60f))) {
                    const float m_new = fmaxf(m_run, block_max() * sl2);
                    if (m_new > m_run) {
                        corr = fast_exp2(m_run - m_new);
                        m_run = m_new;
                    }
                    tmem_wait_st();
                    l_blk = exp_block(m_run == -INFINITY ? 0.f : -m_run);
                    // O moves only when the maximum does, so its rescale is checked
                    // here, off the common path.
                    if (j > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t ov[32];
                            tmem_ld32(tO + c * 32, ov);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * corr);
                            tmem_st32(tO + c * 32, ov);
                        }
                    }
                }
                l_run = l_run * corr + l_blk;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_remote(p_full);
            }
            if (!ok) break;

            ok = wait_pair_warp(bar(kBarOFull + t), o_waits & 1, p.wait_ns, ab);
            if (!ok) break;
            ++o_waits;
            tc_fence_after();
            const float inv_l = 1.f / l_run;
            const bool row_ok = row < p.N;
            __nv_bfloat16 *orow = p.o + ((size_t)(w.b * p.Hq + w.h) * p.N + (row_ok ? row : 0)) * p.d_store;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(tO + c * 32, ov);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
                if (row_ok) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int col = c * 32 + g * 8;
                        if (col < p.d_store)
                            *reinterpret_cast<uint4 *>(orow + col) =
                                make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
                    }
                }
            }
            if (row_ok && p.lse)
                p.lse[(size_t)(w.b * p.Hq + w.h) * p.N + row] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_remote(o_empty);
        }
    }

    // Teardown: both CTAs leave together (no remote arrival or copy may target
    // a CTA that has exited), then free TMEM together.
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
    if (threadIdx.x == 0 && p.order != kNaiveHeadFirst) {
        __threadfence();
        const unsigned int done = atomicAdd(&g_fwd_pair_work[p.sched_slot][kPairWorkDone], 1u);
        if (done == gridDim.x - 1) {
            atomicExch(&g_fwd_pair_work[p.sched_slot][0], 0u);
            atomicExch(&g_fwd_pair_work[p.sched_slot][1], 0u);
            atomicExch(&g_fwd_pair_work[p.sched_slot][kPairWorkDone], 0u);
        }
    }
}

}  // namespace fwd2

int fwd_pair_units_per_head(int N) { return (N + fwd2::kUnitRowsPair - 1) / fwd2::kUnitRowsPair; }

int fwd_pair_launch(const FwdLaunch &a, cudaStream_t stream) {
    using namespace fwd2;
    if (a.d != D) return ATTN_ERR_UNSUPPORTED;  // the pair kernel is built for d = 128
    CUtensorMap mq, mk, mv;
    const uint64_t dq = uint64_t(a.d);
    if (!encode_bf16_3d(&mq, a.q, dq, uint64_t(a.N), uint64_t(a.B) * a.Hq, 64, kTileM) ||
        !encode_bf16_3d(&mk, a.k, dq, uint64_t(a.N), uint64_t(a.B) * a.Hkv, 64, kBlockN / 2) ||
        !encode_bf16_3d(&mv, a.v, dq, uint64_t(a.N), uint64_t(a.B) * a.Hkv, 64, kBlockN))
        return note_cuda_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (pair forward)");
    Params p;
    p.o = reinterpret_cast<__nv_bfloat16 *>(a.o);
    p.lse = a.lse;
    p.B = a.B;
    p.N = a.N;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.d_store = a.d;
    p.causal = a.causal ? 1 : 0;
    p.order = a.order;
    p.nb = fwd_pair_units_per_head(a.N);
    p.total_units = (long long)a.B * a.Hq * p.nb;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.wait_ns = a.wait_ns;
    p.sched_slot = int(g_fwd_pair_launch_seq.fetch_add(1) % kPairSchedSlots);
    p.die_of_sm = nullptr;
    if (a.order == kDieSplitHeadFirst) {
        const int rc = die_map_device(&p.die_of_sm);
        if (rc < 0) return rc;
    }
    // Causal GQA head-first stays ACC by ACC at every size here (this ablation
    // was measured that way); the one-CTA launch reduces small entries to
    // block-first (effective_order).
    const bool grouped = grouped_causal_order(a.order, p.G, p.causal);
    auto kernel = grouped ? fwd_pair_kernel<true> : fwd_pair_kernel<false>;

    // Per device and instantiation: the attributes, and how many pairs can be
    // resident at once (the persistent grid's size).
    static int max_pairs[2][kMaxDevices] = {};
    static std::mutex mu;
    const int dev = slot_for_device();
    int pairs_resident = (dev >= 0) ? max_pairs[grouped][dev] : 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (pairs_resident <= 0) {
        std::lock_guard<std::mutex> lock(mu);
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncGetAttributes(fwd_pair_kernel)");
        if (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads)
            return note_cuda_error(cudaErrorInvalidConfiguration,
                                   "fwd_pair_kernel register count differs from the setmaxnreg split");
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncSetAttribute(fwd_pair_kernel)");
        cfg.gridDim = dim3(2 * unsigned(a.num_sms / 2));
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaOccupancyMaxActiveClusters(fwd_pair_kernel)");
        if (n <= 0) return note_cuda_error(cudaErrorInvalidConfiguration, "no CTA pair of fwd_pair_kernel fits");
        pairs_resident = n;
        if (dev >= 0) max_pairs[grouped][dev] = n;
    }
    long long pairs = p.total_units;
    if (a.order != kNaiveHeadFirst && pairs > pairs_resident) pairs = pairs_resident;
    if (2 * pairs > 0x7fffffffLL) return ATTN_ERR_ARG;
    cfg.gridDim = dim3(unsigned(2 * pairs));
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, p);
    return e == cudaSuccess ? 0 : note_cuda_error(e, "fwd_pair_kernel launch");
}

cudaError_t fwd_pair_take_status(int *bits) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_fwd_pair_status, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_fwd_pair_status, &zero, sizeof(int));
}

}  // namespace attn
