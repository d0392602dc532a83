// fwd_kernel.cuh -- FlashAttention-2 style forward (prefill) kernel for sm_103a.
//
// Computes O = softmax(scale * Q K^T) V and lse per query row ("Optimizing
// Attention on GPUs by Exploiting GPU Architectural NUMA Effects", detail
// page, section 4 equation) with FA2's partitioning (Figure 4: each CTA owns
// a block of query rows and streams every K/V block of its head) and an
// online softmax (running max m, running sum l, rescaled O; kernbench2
// "Fused Grouped-Query Attention", short-context section: running
// accumulators (m, l, O)).
//
// Design (one persistent CTA per SM, 12 warps = 3 warpgroups):
//   warp 0      TMA producer: Q tiles, then a ring of K/V blocks (128 keys).
//   warp 1      tcgen05 issuer + TMEM owner: the whole warp runs the issue
//               loop and one elected lane issues each MMA and commit.
//   warps 2-3   idle (they complete the control warpgroup).
//   warps 4-7   softmax / epilogue of MMA tile 0 (query rows 0-127 of the unit)
//   warps 8-11  softmax / epilogue of MMA tile 1 (rows 128-255)
// A warp may only touch TMEM lanes [32 (w % 4), +32), so each warpgroup
// covers the 128 rows of its tile once.  After set-up the control warpgroup
// gives registers back (setmaxnreg) so each softmax thread can hold a whole
// 128-column row of S in registers.
// A unit is 256 query rows of one head: two 128-row MMA tiles share every
// K/V block loaded into shared memory.  TMEM (512 columns): S/P of tile t at
// columns [128 t, 128 t + 128), O of tile t at [256 + D t, 256 + D t + D).
// S = Q K^T is an SS MMA (M=128, N=128, K=16 steps); P (bf16) is written
// over S in TMEM and O += P V is a TS MMA with V read MN-major from shared
// memory.  The issue order QK(t, j+1) after PV(t, j) means the commit that
// announces S(t, j+1) also guarantees PV(t, j) is complete, so the softmax
// warps may rescale O(t) in TMEM right after they see S(t, j+1).  The row's
// reference maximum is exact for its first block and then kept while the
// block's exponentials sum below 2^60 (no overflow is possible there); only
// when that check fails is the block maximum taken, O rescaled and P
// rewritten (the same result up to rounding, since l and O always share the
// reference maximum).
//
// The kernel is one template over the unit mapping, instantiated by two
// translation units: fwd_sm103.cu (the tile orders, and the grouped causal
// GQA mapping) and fwd_splitkv_sm103.cu (each head's keys cut into ranges,
// fp32 partials per range).  The mappings are compile-time variants, so each
// instantiation carries only its own mapping's code; each translation unit
// has its own copy of the work counters and the status word below.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "attn_internal.h"
#include "sm103_ptx.cuh"
#include "tile_order.cuh"

namespace attn {

static __device__ int g_fwd_status;

// Work counters of the persistent forward kernel: for each of kSchedSlots
// launch slots, {next unit to hand out (die 0 in the die-split order), next
// unit of die 1 (die-split order only), CTAs finished, unused}.  CTAs take
// units in the chosen order by atomically incrementing a `next` counter; the
// last CTA of the launch to finish resets the slot to zero.  Successive
// launches rotate over the slots, so launches only share a slot kSchedSlots
// launches apart.
constexpr int kSchedSlots = 64;
constexpr int kWorkDone = 2;
static __device__ unsigned int g_fwd_work[kSchedSlots][4];
// Launch sequence number behind the slot choice: one counter for every
// instantiation of a translation unit, since they share its g_fwd_work.
static std::atomic<unsigned int> g_fwd_launch_seq{0};

namespace fwd {

constexpr int kTileM = 128;    // query rows per MMA tile
constexpr int kBlockN = 128;   // keys per K/V block
constexpr int kNT = 2;         // MMA tiles per unit
constexpr int kThreads = 384;  // 12 warps
// Register split after set-up.  The launch gives 168 registers per thread
// (65536 / 384, rounded down to a multiple of 8): 384 x 168 = 64512 in all.
// The split must not exceed that or setmaxnreg.inc would wait forever; the
// host checks the compiled count before every launch.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 120;  // the warp-wide MMA issue loop spills at 104
constexpr int kSoftmaxRegs = 192;
static_assert(128 * kCtrlRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kTmemCols = 512;

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;              // 128-byte column chunks per row
    static constexpr int kChunkBytes = 128 * 128;       // 128 rows x 128 bytes
    static constexpr int kQBytes = kTileM * D * 2;
    static constexpr int kKVBytes = kBlockN * D * 2;
    static constexpr int kStages = (D == 128) ? 4 : 8;  // K/V ring slots
    static constexpr int kOCol = 2 * kTileM;            // first O column in TMEM
    // barriers: q_full[2] q_empty[2] s_full[2] p_full[2] o_full[2] o_empty[2]
    //           kv_full[S] kv_empty[S] drain
    static constexpr int kBarQFull = 0, kBarQEmpty = 2, kBarSFull = 4, kBarPFull = 6,
                         kBarOFull = 8, kBarOEmpty = 10, kBarKVFull = 12,
                         kBarKVEmpty = 12 + kStages, kBarDrain = 12 + 2 * kStages,
                         kBarUQFull = 13 + 2 * kStages, kBarUQEmpty = 15 + 2 * kStages,
                         kNumBars = 17 + 2 * kStages;
    static constexpr int kDataBytes = kNT * kQBytes + kStages * kKVBytes;
    // data, barriers, TMEM address, abort flag, two-entry unit queue, align slack
    static constexpr int kSmemBytes = kDataBytes + kNumBars * 8 + 32 + 1024;
};

struct Params {
    __nv_bfloat16 *o;
    float *lse;
    int B, N, Hq, Hkv, G, d_store, causal, order, nb;
    long long total_units;
    float scale_log2;
    unsigned long long wait_ns;
    int sched_slot;  // g_fwd_work slot of this launch (persistent orders)
    const int *die_of_sm;  // die of each SM id (die-split order; else null)
};

// Parameters of split launches: key range s is blocks [s * chunk_blocks,
// (s + 1) * chunk_blocks); the outputs are the ranges' partials (o and lse
// are unused).
struct SplitParams : Params {
    float *part_o;    // [splits][B * Hq][N][d_store] fp32: O of each range, normalised by its own l
    float *part_lse;  // [splits][B * Hq][N] fp32: natural-log lse of each range (-inf when empty)
    int splits, chunk_blocks;
};

struct UnitWork {
    int b, h, kvh;
    int row0[kNT];
    int nkv[kNT];  // K/V blocks each tile visits from jb (0: tile lies past N, or nothing in its range)
    int nmax;
};

// Unit mappings, one kernel instantiation each:
//   kMapOrder    the tile order of the launch (unit_to_tile);
//   kMapGrouped  causal GQA in a head-first order (unit_to_tile_grouped_causal);
//   kMapSplit    sub-ACC head-first order over key ranges: an ACC (the query
//                heads of one KV head of one batch entry) runs key range 0 for
//                all its heads and row blocks, then range 1, and so on, so the
//                CTAs running at the same time stream one range of one K/V
//                head.  Inside a range: query head, then row block
//                (descending when causal, longest first).
enum UnitMap : int { kMapOrder = 0, kMapGrouped = 1, kMapSplit = 2 };

// Parameter block of each mapping.
template <int kMap>
struct ParamsOf {
    using type = Params;
};
template <>
struct ParamsOf<kMapSplit> {
    using type = SplitParams;
};

// A unit's work under mapping kMap: s is its key range and jb the range's
// first K/V block; both are the constant 0 except for split launches, so the
// other mappings carry no extra state.
template <int kMap>
struct MappedWork : UnitWork {
    static constexpr int s = 0, jb = 0;
};
template <>
struct MappedWork<kMapSplit> : UnitWork {
    int s, jb;
};

template <int kMap>
__device__ __forceinline__ MappedWork<kMap> unit_work(const typename ParamsOf<kMap>::type &p, long long u) {
    if constexpr (kMap == kMapSplit) {
        MappedWork<kMap> w;
        const int nkv_all = (p.N + kBlockN - 1) / kBlockN;
        w.nmax = 0;
        const long long per_split = (long long)p.G * p.nb;
        const long long upa = per_split * p.splits;  // units per ACC
        const long long a = u / upa;
        const long long w0 = u % upa;
        const int s = int(w0 / per_split);
        const int w1 = int(w0 % per_split);
        const int hg = w1 / p.nb, r = w1 % p.nb;
        w.b = int(a / p.Hkv);
        w.kvh = int(a % p.Hkv);
        w.h = w.kvh * p.G + hg;
        w.s = s;
        w.jb = s * p.chunk_blocks;
        const int m = p.causal ? (p.nb - 1 - r) : r;
        const int je_all = min(nkv_all, w.jb + p.chunk_blocks);
#pragma unroll
        for (int tt = 0; tt < kNT; ++tt) {
            const int r0 = m * kUnitRows + tt * kTileM;
            w.row0[tt] = r0;
            int n = 0;
            if (r0 < p.N) {
                const int je = p.causal ? min(je_all, r0 / kBlockN + 1) : je_all;
                n = max(0, je - w.jb);
            }
            w.nkv[tt] = n;
            w.nmax = max(w.nmax, n);
        }
        return w;
    } else {
        const Tile t = kMap == kMapGrouped ? unit_to_tile_grouped_causal(u, p.Hq, p.G, p.nb)
                                           : unit_to_tile(p.order, u, p.Hq, p.nb, p.causal);
        MappedWork<kMap> w;
        w.b = t.b;
        w.h = t.h;
        w.kvh = t.h / p.G;
        const int nkv_all = (p.N + kBlockN - 1) / kBlockN;
        w.nmax = 0;
#pragma unroll
        for (int tt = 0; tt < kNT; ++tt) {
            const int r0 = t.m * kUnitRows + tt * kTileM;
            w.row0[tt] = r0;
            int n = 0;
            if (r0 < p.N) n = p.causal ? min(nkv_all, r0 / kBlockN + 1) : nkv_all;
            w.nkv[tt] = n;
            w.nmax = max(w.nmax, n);
        }
        return w;
    }
}

// The i-th unit this CTA processes, or -1 when there is none left.  Naive
// head-first: one unit per CTA, its block index.  Otherwise the next unit of
// the order from the launch's work counter, so CTAs running at the same time
// hold consecutive units (one ACC at a time in head-first order) and faster
// CTAs simply take more units.  Die-split: each die has its own counter over
// its own ACCs; a die whose ACCs are all handed out takes the other die's
// remaining units, so no SM idles while work is left.
__device__ __forceinline__ long long fetch_unit(const Params &p, long long i, int my_die) {
    if (p.order == kNaiveHeadFirst) return i == 0 ? (long long)blockIdx.x : -1;
    if (p.order == kDieSplitHeadFirst) {
        for (int s = 0; s < kDies; ++s) {
            const int die = (my_die + s) % kDies;
            const unsigned int k = atomicAdd(&g_fwd_work[p.sched_slot][die], 1u);
            const long long u = die_split_unit(die, (long long)k, p.B, p.Hkv, p.G, p.nb);
            if (u >= 0) return u;
        }
        return -1;
    }
    const unsigned int u = atomicAdd(&g_fwd_work[p.sched_slot][0], 1u);
    return (long long)u < p.total_units ? (long long)u : -1;
}

// Last tile (highest index) that still uses K/V block j.
__device__ __forceinline__ int last_user(const UnitWork &w, int j) {
    int last = -1;
#pragma unroll
    for (int t = 0; t < kNT; ++t)
        if (j < w.nkv[t]) last = t;
    return last;
}

// The kernel, one instantiation per head dimension and unit mapping.  It is
// the kernel template itself, not a body called from thin per-mapping
// kernels: a __global__ wrapper passing its parameters by reference to an
// inlined body ran the d = 128 ordinary launches 4% slower (same registers
// and stack; measured side by side on one GPU).
template <int D, int kMap>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const typename ParamsOf<kMap>::type p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sQ = smem;
    uint8_t *sKV = smem + kNT * C::kQBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kDataBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *unit_q = reinterpret_cast<volatile int *>(tmem_slot + 2);  // 2 entries

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };

    if (threadIdx.x == 0) {
        for (int t = 0; t < kNT; ++t) {
            mbar_init(bar(C::kBarQFull + t), 1);
            mbar_init(bar(C::kBarQEmpty + t), 1);
            mbar_init(bar(C::kBarSFull + t), 1);
            mbar_init(bar(C::kBarPFull + t), 4);   // one arrival per softmax warp
            mbar_init(bar(C::kBarOFull + t), 1);
            mbar_init(bar(C::kBarOEmpty + t), 4);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(C::kBarKVFull + s), 1);
            mbar_init(bar(C::kBarKVEmpty + s), 1);
        }
        mbar_init(bar(C::kBarDrain), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::kBarUQFull + i), 1);
            mbar_init(bar(C::kBarUQEmpty + i), 1 + 8);  // MMA warp + 8 softmax warps
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
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int *status = &g_fwd_status;

    // Each role runs inside the branch that set its register limit, so the
    // compiler allocates each role's code under that role's limit.
    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
      if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            long long fills = 0;          // K/V ring fills issued
            int q_loads[kNT] = {0, 0};    // Q loads issued per tile
            bool ok = true;
            int my_die = 0;
            if (p.die_of_sm) {
                uint32_t smid;
                asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
                if (smid < uint32_t(kDieMapMaxSms)) my_die = p.die_of_sm[smid] & 1;
            }
            for (long long qi = 0; ok; ++qi) {
                // Publish the next unit to the other roles (two-entry queue).
                const long long u = fetch_unit(p, qi, my_die);
                const int qs = int(qi & 1);
                if (qi >= 2 && !mbar_wait_bounded(bar(C::kBarUQEmpty + qs), uint32_t(((qi >> 1) - 1) & 1),
                                                  p.wait_ns, abort_flag, status)) {
                    ok = false;
                    break;
                }
                unit_q[qs] = int(u);
                mbar_arrive(bar(C::kBarUQFull + qs));
                if (u < 0) break;
                const auto w = unit_work<kMap>(p, u);
                for (int t = 0; t < kNT && ok; ++t) {
                    if (w.nkv[t] == 0) continue;
                    if (q_loads[t] > 0)
                        ok = mbar_wait_bounded(bar(C::kBarQEmpty + t), (q_loads[t] - 1) & 1,
                                               p.wait_ns, abort_flag, status);
                    if (!ok) break;
                    const uint32_t qb = bar(C::kBarQFull + t);
                    mbar_arrive_expect_tx(qb, C::kQBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(smem_u32(sQ + t * C::kQBytes + c * C::kChunkBytes), &tmQ, qb,
                                    c * 64, w.row0[t], w.b * p.Hq + w.h);
                    ++q_loads[t];
                }
                for (int j = 0; ok && j < w.nmax; ++j) {
                    for (int kv = 0; kv < 2; ++kv) {
                        const int slot = int(fills % C::kStages);
                        const long long round = fills / C::kStages;
                        if (round > 0) {
                            ok = mbar_wait_bounded(bar(C::kBarKVEmpty + slot), uint32_t((round - 1) & 1),
                                                   p.wait_ns, abort_flag, status);
                            if (!ok) break;
                        }
                        const uint32_t fb = bar(C::kBarKVFull + slot);
                        mbar_arrive_expect_tx(fb, C::kKVBytes);
                        const CUtensorMap *map = kv == 0 ? &tmK : &tmV;
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d(smem_u32(sKV + slot * C::kKVBytes + c * C::kChunkBytes), map,
                                        fb, c * 64, (w.jb + j) * kBlockN, w.b * p.Hkv + w.kvh);
                        ++fills;
                    }
                }
            }
            if (!ok) {
                // Drain: wait (bounded, independent of the caller's limit) for the
                // last fill of every slot and the last Q load of every tile, so no
                // copy is still writing shared memory when the CTA exits.
                const unsigned long long drain_ns = 1000000000ull;
                volatile int no_abort = 0;
                for (int s = 0; s < C::kStages; ++s) {
                    long long last = fills - 1 - ((fills - 1 - s) % C::kStages + C::kStages) % C::kStages;
                    if (fills == 0 || last < 0) continue;
                    if (!mbar_wait_bounded(bar(C::kBarKVFull + int(last % C::kStages)),
                                           uint32_t((last / C::kStages) & 1), drain_ns, &no_abort,
                                           status))
                        atomicOr(status, kStatusDrainTimeout);
                }
                for (int t = 0; t < kNT; ++t)
                    if (q_loads[t] > 0 &&
                        !mbar_wait_bounded(bar(C::kBarQFull + t), (q_loads[t] - 1) & 1, drain_ns,
                                           &no_abort, status))
                        atomicOr(status, kStatusDrainTimeout);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        // The whole warp runs the issuer's loop (its state is warp-uniform);
        // each MMA, commit and arrival goes out from one elected lane.  The
        // earlier form, one lane running the loop alone, ran the kernel about
        // 20% slower at d = 128 (14% at d <= 64) with the same MMAs, waits and
        // commits; a warp-uniform loop lets the compiler treat its state and
        // the MMA operands as uniform across the warp.
        {
            constexpr uint32_t kIdescQK = idesc_bf16_f32(kTileM, kBlockN, 0);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileM, D, 1);
            long long fills = 0;                 // ring position of the next block used
            int q_used[kNT] = {0, 0};            // Q loads consumed per tile
            int p_waits[kNT] = {0, 0};           // P(t) handoffs consumed
            int units_done[kNT] = {0, 0};        // epilogues owed per tile
            bool ok = true;

            auto wait_slot = [&](long long f) {
                return mbar_wait_warp(bar(C::kBarKVFull + int(f % C::kStages)),
                                      uint32_t((f / C::kStages) & 1), p.wait_ns, abort_flag, status);
            };
            // Descriptors of the first Q tile and the first ring slot; every other
            // operand start is base + (byte offset >> 4) in the 14-bit address
            // field (shared-memory offsets stay below 256 KiB, so no carry).
            const uint64_t dQ = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dK = smem_desc_sw128(smem_u32(sKV), 16, 1024);
            const uint64_t dV = smem_desc_sw128(smem_u32(sKV), C::kChunkBytes, 1024);
            auto slot_off = [&](long long f) {
                return uint64_t(int(f % C::kStages) * (C::kKVBytes >> 4));
            };
            // Each group of MMAs goes out from one asm block (descriptors
            // computed first), so the issuing warp needs no issue slots
            // between them while the softmax warps of its sub-partition run.
            auto issue_qk = [&](int t, long long fK) {
                const uint64_t a0 = dQ + uint64_t(t * (C::kQBytes >> 4));
                const uint64_t b0 = dK + slot_off(fK);
                const uint32_t d_tmem = tmem_base + t * kTileM;
#pragma unroll
                for (int g = 0; g < D / 64; ++g) {  // four K=16 steps per 128-byte chunk
                    uint64_t a[4], b[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint64_t off = uint64_t((g * C::kChunkBytes + i * 32) >> 4);
                        a[i] = a0 + off;
                        b[i] = b0 + off;
                    }
                    tc_mma_ss_x4_elect(d_tmem, a, b, kIdescQK, g > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, long long fV, bool acc) {
                const uint64_t b0 = dV + slot_off(fV);
                const uint32_t d_tmem = tmem_base + C::kOCol + t * D;
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
                    tc_mma_ts_x4_elect(d_tmem, a, b, kIdescPV, (acc || g > 0) ? 1u : 0u);
                }
            };

            for (long long qi = 0; ok; ++qi) {
                const int qs = int(qi & 1);
                ok = mbar_wait_warp(bar(C::kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns,
                                       abort_flag, status);
                if (!ok) break;
                const long long u = __shfl_sync(0xffffffffu, int(unit_q[qs]), 0);
                mbar_arrive_elect(bar(C::kBarUQEmpty + qs));
                if (u < 0) break;
                const auto w = unit_work<kMap>(p, u);
                if constexpr (kMap == kMapSplit) {
                    // A causal unit whose rows all lie before its key range has
                    // no block to visit (the producer loads nothing for it).
                    if (w.nmax == 0) continue;
                }
                const long long f0 = fills;  // K_j at f0 + 2j, V_j at f0 + 2j + 1
                // prologue: S(t, 0) = Q(t) K_0^T
                ok = wait_slot(f0);
                for (int t = 0; ok && t < kNT; ++t) {
                    if (w.nkv[t] == 0) continue;
                    ok = mbar_wait_warp(bar(C::kBarQFull + t), q_used[t] & 1, p.wait_ns,
                                           abort_flag, status);
                    if (!ok) break;
                    ++q_used[t];
                    tc_fence_after();
                    issue_qk(t, f0);
                    tc_commit_elect(bar(C::kBarSFull + t));
                }
                for (int j = 0; ok && j < w.nmax; ++j) {
                    const long long fV = f0 + 2 * j + 1, fK = f0 + 2 * j + 2;
                    bool v_ready = false, k_ready = false;
                    for (int t = 0; ok && t < kNT; ++t) {
                        if (j >= w.nkv[t]) continue;
                        ok = mbar_wait_warp(bar(C::kBarPFull + t), p_waits[t] & 1, p.wait_ns,
                                               abort_flag, status);
                        if (!ok) break;
                        ++p_waits[t];
                        if (j == 0 && units_done[t] > 0) {
                            ok = mbar_wait_warp(bar(C::kBarOEmpty + t), (units_done[t] - 1) & 1,
                                                   p.wait_ns, abort_flag, status);
                            if (!ok) break;
                        }
                        if (!v_ready) {
                            ok = wait_slot(fV);
                            if (!ok) break;
                            v_ready = true;
                        }
                        tc_fence_after();
                        issue_pv(t, fV, j > 0);
                        if (t == last_user(w, j)) tc_commit_elect(bar(C::kBarKVEmpty + int(fV % C::kStages)));
                        if (j + 1 < w.nkv[t]) {
                            if (!k_ready) {
                                ok = wait_slot(fK);
                                if (!ok) break;
                                k_ready = true;
                            }
                            issue_qk(t, fK);
                            tc_commit_elect(bar(C::kBarSFull + t));
                        } else {
                            tc_commit_elect(bar(C::kBarOFull + t));   // O(t) final for this unit
                            tc_commit_elect(bar(C::kBarQEmpty + t));  // Q(t) buffer reusable
                            ++units_done[t];
                        }
                    }
                }
                fills = f0 + 2 * (long long)w.nmax;
            }
            // Teardown: make sure every issued MMA has finished before TMEM is freed.
            tc_commit_elect(bar(C::kBarDrain));
            volatile int no_abort = 0;
            if (!mbar_wait_warp(bar(C::kBarDrain), 0, 1000000000ull, &no_abort, status) && lane == 0)
                atomicOr(status, kStatusDrainTimeout);
        }
        __syncwarp();
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
        // ------------------------------------------------- softmax / epilogue
        const int t = (warp - 4) >> 2;      // MMA tile of this warpgroup
        const int quarter = warp & 3;       // TMEM lane quarter of this warp
        const int r = quarter * 32 + lane;  // row inside the tile
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        const uint32_t tS = tmem_base + lane_off + t * kTileM;
        const uint32_t tO = tmem_base + lane_off + C::kOCol + t * D;
        const float sl2 = p.scale_log2;
        int s_waits = 0, o_waits = 0;
        long long kv_base = 0;  // ring position of the current unit's first K/V fill
        // One thread of the warpgroup frees K slots of the ring.  S(t, j)
        // complete means every MMA issued before its commit is complete, QK(t', j)
        // of every tile included, so the last tile to use K_j frees its slot on
        // seeing S(t, j) and the MMA warp needs no commit of its own for it.
        // (V slots keep their commit right after the last PV that reads them:
        // waiting for the next S would free them about eight MMAs later, which
        // measured slower.)
        const bool frees_slots = (quarter == 0);  // warp-uniform; the elected lane arrives
        bool ok = true;

        for (long long qi = 0; ok; ++qi) {
            const int qs = int(qi & 1);
            ok = mbar_wait_warp(bar(C::kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns, abort_flag,
                                status);
            if (!ok) break;
            const long long u = unit_q[qs];
            __syncwarp();
            mbar_arrive_elect(bar(C::kBarUQEmpty + qs));
            if (u < 0) break;
            const auto w = unit_work<kMap>(p, u);
            const long long f0 = kv_base;  // K_j at ring position f0 + 2j
            kv_base += 2 * (long long)w.nmax;
            const int nkv = w.nkv[t];
            if (nkv == 0) continue;
            const int row = w.row0[t] + r;
            float m_run = -INFINITY, l_run = 0.f;

            for (int j = 0; j < nkv; ++j) {
                ok = mbar_wait_warp(bar(C::kBarSFull + t), s_waits & 1, p.wait_ns, abort_flag,
                                    status);
                if (!ok) break;
                ++s_waits;
                if (frees_slots && t == last_user(w, j))
                    mbar_arrive_elect(bar(C::kBarKVEmpty + int((f0 + 2 * j) % C::kStages)));
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

                const int kv0 = (w.jb + j) * kBlockN;
                const bool ragged = kv0 + kBlockN > p.N;
                const bool diag = p.causal && (kv0 + kBlockN - 1 > w.row0[t]);
                if (ragged || diag) {
                    int lim = p.N - kv0;
                    if (p.causal) lim = min(lim, row + 1 - kv0);
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                // Row maximum of the block: four independent chains of three-input maxima.
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
                // P = 2^(s*scale*log2e - m) in bf16, written over S in TMEM; returns
                // the block's row sum (four independent pairs of partial sums).
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
                // The reference maximum m_run is exact for a row's first block and
                // is otherwise kept: exponentials against it cannot overflow while
                // the block's sum stays below 2^60 (bf16 and fp32 share the
                // exponent range), so the block maximum is only needed when that
                // check fails.  Then the warp takes the exact maximum, rescales and
                // writes P again (lanes whose reference did not move store the
                // same values once more).
                float corr = 1.f;
                if (m_run == -INFINITY) m_run = block_max() * sl2;  // stays -inf if all masked
                float l_blk = exp_block(m_run == -INFINITY ? 0.f : -m_run);
                if (__any_sync(0xffffffffu, !(l_blk < 0x1p60f))) {
                    const float m_new = fmaxf(m_run, block_max() * sl2);
                    if (m_new > m_run) {
                        corr = fast_exp2(m_run - m_new);
                        m_run = m_new;
                    }
                    tmem_wait_st();
                    l_blk = exp_block(m_run == -INFINITY ? 0.f : -m_run);
                    // Rescale this row of O when its reference maximum moved (never
                    // on the first block: PV(t, 0) overwrites O).  The maximum only
                    // moves here, so the check stays off the common path, where a
                    // second warp vote and branch cost about 60 clocks per block.
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
                mbar_arrive_elect(bar(C::kBarPFull + t));
            }
            if (!ok) break;

            // Epilogue: O / l -> bf16, lse = (m + log2 l) * ln 2; split launches
            // write the range's O / l in fp32 and its lse instead (a row with no
            // key in the range has l = 0: its lse is -inf and the merge skips it).
            ok = mbar_wait_warp(bar(C::kBarOFull + t), o_waits & 1, p.wait_ns, abort_flag, status);
            if (!ok) break;
            ++o_waits;
            tc_fence_after();
            if constexpr (kMap == kMapSplit) {
                const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
                const bool row_ok = row < p.N;
                const size_t prow =
                    ((size_t)w.s * p.B * p.Hq + (size_t)(w.b * p.Hq + w.h)) * p.N + (row_ok ? row : 0);
                float *orow = p.part_o + prow * p.d_store;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(tO + c * 32, ov);
                    tmem_wait_ld();
                    if (row_ok) {
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            const int col = c * 32 + g * 4;
                            if (col < p.d_store)
                                *reinterpret_cast<float4 *>(orow + col) = make_float4(
                                    __uint_as_float(ov[4 * g]) * inv_l, __uint_as_float(ov[4 * g + 1]) * inv_l,
                                    __uint_as_float(ov[4 * g + 2]) * inv_l, __uint_as_float(ov[4 * g + 3]) * inv_l);
                        }
                    }
                }
                if (row_ok)
                    p.part_lse[prow] = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
            } else {
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
                        pk[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l,
                                            __uint_as_float(ov[2 * i + 1]) * inv_l);
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
            }
            tc_fence_before();
            __syncwarp();
            mbar_arrive_elect(bar(C::kBarOEmpty + t));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
    if (threadIdx.x == 0 && p.order != kNaiveHeadFirst) {
        // Every CTA has fetched its last unit before it gets here, so the last
        // CTA to arrive may reset the launch's counters for the next user.
        __threadfence();
        const unsigned int done = atomicAdd(&g_fwd_work[p.sched_slot][kWorkDone], 1u);
        if (done == gridDim.x - 1) {
            atomicExch(&g_fwd_work[p.sched_slot][0], 0u);
            atomicExch(&g_fwd_work[p.sched_slot][1], 0u);
            atomicExch(&g_fwd_work[p.sched_slot][kWorkDone], 0u);
        }
    }
}

}  // namespace fwd
}  // namespace attn
