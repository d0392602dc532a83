// fwd_splitkv_sm103.cu -- forward attention with the key range of every head
// split into sub-ranges ("sub-ACC" split), then a log-sum-exp merge.
//
// "Optimizing Attention on GPUs by Exploiting GPU Architectural NUMA
// Effects" (related-work page, on the Attention Compute Cluster when one
// head's K/V outgrows an L2 slice) suggests splitting an ACC's keys so that
// the CTAs running together stream a piece of K/V that fits in L2.  Here the
// units of an ACC run key range 0 for all its heads and row blocks, then key
// range 1, and so on; each unit writes the fp32 partial (O_s normalised by
// its own l_s, lse_s) of its rows over its range, and a merge kernel combines
// the ranges of every row as the decode merge does (kernbench2 "Fused
// Grouped-Query Attention", Case 4: the (m, l, O) reduction):
//     L = max_s lse_s,  w_s = exp(lse_s - L),  O = sum_s w_s O_s / sum_s w_s,
//     lse = L + log(sum_s w_s).
// The kernel is the forward kernel of fwd_sm103.cu (same roles, TMEM plan,
// softmax and bounded waits) with the unit mapping, the K/V block offset and
// the epilogue changed; it lives in its own translation unit so that the
// forward kernel's code is untouched.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "../../include/attn.h"
#include "attn_internal.h"
#include "sm103_ptx.cuh"
#include "tile_order.cuh"

namespace attn {

static __device__ int g_fwd_split_status;

// Work counters of the persistent split-KV kernel, as in the forward kernel:
// per launch slot {next unit, unused, CTAs finished, unused}; the last CTA of
// a launch resets its slot.  Own slots, so the kernels never share one.
constexpr int kSchedSlots = 64;
constexpr int kWorkDone = 2;
static __device__ unsigned int g_fwd_split_work[kSchedSlots][4];
static std::atomic<unsigned int> g_fwd_split_launch_seq{0};

namespace fwd3 {

constexpr int kTileM = 128;    // query rows per MMA tile
constexpr int kBlockN = 128;   // keys per K/V block
constexpr int kNT = 2;         // MMA tiles per unit
constexpr int kThreads = 384;  // 12 warps
// Register split after set-up.  The launch gives 168 registers per thread
// (65536 / 384, rounded down to a multiple of 8): 384 x 168 = 64512 in all.
// The split must not exceed that or setmaxnreg.inc would wait forever; the
// host checks the compiled count before every launch.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 104;
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
    float *part_o;    // [splits][B * Hq][N][d_store] fp32: O of each key range, normalised by its own l
    float *part_lse;  // [splits][B * Hq][N] fp32: natural-log lse of each key range (-inf when empty)
    int B, N, Hq, Hkv, G, d_store, causal, nb;
    int splits, chunk_blocks;  // key range s = blocks [s * chunk_blocks, (s + 1) * chunk_blocks)
    long long total_units;
    float scale_log2;
    unsigned long long wait_ns;
    int sched_slot;
};

struct UnitWork {
    int b, h, kvh, s;
    int jb;        // first K/V block of the unit's key range
    int row0[kNT];
    int nkv[kNT];  // K/V blocks each tile visits from jb (0: nothing to attend in the range)
    int nmax;
};

// Sub-ACC head-first order: an ACC (the query heads of one KV head of one
// batch entry) runs key range 0 for all its heads and row blocks, then key
// range 1, and so on, so CTAs running at the same time stream one range of
// one K/V head.  Inside a range: query head, then row block (descending when
// causal, longest first).
__device__ __forceinline__ UnitWork unit_work(const Params &p, long long u) {
    const long long per_split = (long long)p.G * p.nb;
    const long long upa = per_split * p.splits;  // units per ACC
    const long long a = u / upa;
    const long long w0 = u % upa;
    const int s = int(w0 / per_split);
    const int w1 = int(w0 % per_split);
    const int hg = w1 / p.nb, r = w1 % p.nb;
    UnitWork w;
    w.b = int(a / p.Hkv);
    w.kvh = int(a % p.Hkv);
    w.h = w.kvh * p.G + hg;
    w.s = s;
    const int m = p.causal ? (p.nb - 1 - r) : r;
    const int nkv_all = (p.N + kBlockN - 1) / kBlockN;
    w.jb = s * p.chunk_blocks;
    const int je_all = min(nkv_all, w.jb + p.chunk_blocks);
    w.nmax = 0;
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
}

// The next unit from the launch's work counter, or -1 when none is left.
__device__ __forceinline__ long long fetch_unit(const Params &p) {
    const unsigned int u = atomicAdd(&g_fwd_split_work[p.sched_slot][0], 1u);
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_split_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const Params p) {
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
            mbar_init(bar(C::kBarUQEmpty + i), 1 + 8);  // MMA thread + 8 softmax warps
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

    int *status = &g_fwd_split_status;

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
            for (long long qi = 0; ok; ++qi) {
                // Publish the next unit to the other roles (two-entry queue).
                const long long u = fetch_unit(p);
                const int qs = int(qi & 1);
                if (qi >= 2 && !mbar_wait_bounded(bar(C::kBarUQEmpty + qs), uint32_t(((qi >> 1) - 1) & 1),
                                                  p.wait_ns, abort_flag, status)) {
                    ok = false;
                    break;
                }
                unit_q[qs] = int(u);
                mbar_arrive(bar(C::kBarUQFull + qs));
                if (u < 0) break;
                const UnitWork w = unit_work(p, u);
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
        if (lane == 0) {
            constexpr uint32_t kIdescQK = idesc_bf16_f32(kTileM, kBlockN, 0);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileM, D, 1);
            long long fills = 0;                 // ring position of the next block used
            int q_used[kNT] = {0, 0};            // Q loads consumed per tile
            int p_waits[kNT] = {0, 0};           // P(t) handoffs consumed
            int units_done[kNT] = {0, 0};        // epilogues owed per tile
            bool ok = true;

            auto wait_slot = [&](long long f) {
                return mbar_wait_bounded(bar(C::kBarKVFull + int(f % C::kStages)),
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
            // computed first), so the issuing thread needs no issue slots
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
                    tc_mma_ss_x4(d_tmem, a, b, kIdescQK, g > 0 ? 1u : 0u);
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
                    tc_mma_ts_x4(d_tmem, a, b, kIdescPV, (acc || g > 0) ? 1u : 0u);
                }
            };

            for (long long qi = 0; ok; ++qi) {
                const int qs = int(qi & 1);
                ok = mbar_wait_bounded(bar(C::kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns,
                                       abort_flag, status);
                if (!ok) break;
                const long long u = unit_q[qs];
                mbar_arrive(bar(C::kBarUQEmpty + qs));
                if (u < 0) break;
                const UnitWork w = unit_work(p, u);
                // A causal unit whose rows all lie before its key range has no
                // block to visit (the producer loads nothing for it).
                if (w.nmax == 0) continue;
                const long long f0 = fills;  // K_j at f0 + 2j, V_j at f0 + 2j + 1
                // prologue: S(t, 0) = Q(t) K_0^T
                ok = wait_slot(f0);
                for (int t = 0; ok && t < kNT; ++t) {
                    if (w.nkv[t] == 0) continue;
                    ok = mbar_wait_bounded(bar(C::kBarQFull + t), q_used[t] & 1, p.wait_ns,
                                           abort_flag, status);
                    if (!ok) break;
                    ++q_used[t];
                    tc_fence_after();
                    issue_qk(t, f0);
                    tc_commit(bar(C::kBarSFull + t));
                }
                for (int j = 0; ok && j < w.nmax; ++j) {
                    const long long fV = f0 + 2 * j + 1, fK = f0 + 2 * j + 2;
                    bool v_ready = false, k_ready = false;
                    for (int t = 0; ok && t < kNT; ++t) {
                        if (j >= w.nkv[t]) continue;
                        ok = mbar_wait_bounded(bar(C::kBarPFull + t), p_waits[t] & 1, p.wait_ns,
                                               abort_flag, status);
                        if (!ok) break;
                        ++p_waits[t];
                        if (j == 0 && units_done[t] > 0) {
                            ok = mbar_wait_bounded(bar(C::kBarOEmpty + t), (units_done[t] - 1) & 1,
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
                        if (t == last_user(w, j)) tc_commit(bar(C::kBarKVEmpty + int(fV % C::kStages)));
                        if (j + 1 < w.nkv[t]) {
                            if (!k_ready) {
                                ok = wait_slot(fK);
                                if (!ok) break;
                                k_ready = true;
                            }
                            issue_qk(t, fK);
                            tc_commit(bar(C::kBarSFull + t));
                        } else {
                            tc_commit(bar(C::kBarOFull + t));   // O(t) final for this unit
                            tc_commit(bar(C::kBarQEmpty + t));  // Q(t) buffer reusable
                            ++units_done[t];
                        }
                    }
                }
                fills = f0 + 2 * (long long)w.nmax;
            }
            // Teardown: make sure every issued MMA has finished before TMEM is freed.
            tc_commit(bar(C::kBarDrain));
            volatile int no_abort = 0;
            if (!mbar_wait_bounded(bar(C::kBarDrain), 0, 1000000000ull, &no_abort, status))
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
        // seeing S(t, j) and the MMA thread needs no commit of its own for it.
        // (V slots keep their commit right after the last PV that reads them:
        // waiting for the next S would free them about eight MMAs later, which
        // measured slower.)
        const bool frees_slots = (quarter == 0 && lane == 0);
        bool ok = true;

        for (long long qi = 0; ok; ++qi) {
            const int qs = int(qi & 1);
            ok = mbar_wait_warp(bar(C::kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns, abort_flag,
                                status);
            if (!ok) break;
            const long long u = unit_q[qs];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarUQEmpty + qs));
            if (u < 0) break;
            const UnitWork w = unit_work(p, u);
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
                    mbar_arrive(bar(C::kBarKVEmpty + int((f0 + 2 * j) % C::kStages)));
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
                }
                l_run = l_run * corr + l_blk;
                // Rescale this row of O when its reference maximum moved (never on
                // the first block: PV(t, 0) overwrites O).
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
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarPFull + t));
            }
            if (!ok) break;

            // Epilogue: this key range's O / l in fp32 and its lse = (m + log2 l) * ln 2
            // (a row with no key in the range has l = 0: its lse is -inf and the
            // merge skips it).
            ok = mbar_wait_warp(bar(C::kBarOFull + t), o_waits & 1, p.wait_ns, abort_flag, status);
            if (!ok) break;
            ++o_waits;
            tc_fence_after();
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
            const bool row_ok = row < p.N;
            const size_t prow = ((size_t)w.s * p.B * p.Hq + (size_t)(w.b * p.Hq + w.h)) * p.N + (row_ok ? row : 0);
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
                            *reinterpret_cast<float4 *>(orow + col) =
                                make_float4(__uint_as_float(ov[4 * g]) * inv_l, __uint_as_float(ov[4 * g + 1]) * inv_l,
                                            __uint_as_float(ov[4 * g + 2]) * inv_l,
                                            __uint_as_float(ov[4 * g + 3]) * inv_l);
                    }
                }
            }
            if (row_ok)
                p.part_lse[prow] = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarOEmpty + t));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
    if (threadIdx.x == 0) {
        // Every CTA has fetched its last unit before it gets here, so the last
        // CTA to arrive may reset the launch's counters for the next user.
        __threadfence();
        const unsigned int done = atomicAdd(&g_fwd_split_work[p.sched_slot][kWorkDone], 1u);
        if (done == gridDim.x - 1) {
            atomicExch(&g_fwd_split_work[p.sched_slot][0], 0u);
            atomicExch(&g_fwd_split_work[p.sched_slot][kWorkDone], 0u);
        }
    }
}


// One warp per query row: combine the row's key ranges.  A causal row i
// attends range s only if it starts at or before i (s * C <= i); otherwise
// that range's partial is not read.  Lane l holds columns [4l, 4l + 4).
__global__ void __launch_bounds__(256)
    split_merge_kernel(const float *part_o, const float *part_lse, __nv_bfloat16 *o, float *lse, long long rows,
                       int N, int d, int splits, int chunk_keys, int causal) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int i = int(row % N);  // position of the row in its sequence
    const int ns = causal ? min(splits, i / chunk_keys + 1) : splits;
    const size_t stride = (size_t)rows;  // rows per split
    float L = -INFINITY;
    for (int s = 0; s < ns; ++s) L = fmaxf(L, part_lse[s * stride + row]);
    const int c0 = lane * 4;
    const bool active = c0 < d;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float ls = part_lse[s * stride + row];
        if (ls == -INFINITY) continue;
        const float w = __expf(ls - L);
        wsum += w;
        if (active) {
            const float4 v = *reinterpret_cast<const float4 *>(part_o + (s * stride + row) * d + c0);
            acc[0] += w * v.x;
            acc[1] += w * v.y;
            acc[2] += w * v.z;
            acc[3] += w * v.w;
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    if (active) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t *>(&lo);
        pk.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(o + row * d + c0) = pk;
    }
    if (lane == 0 && lse) lse[row] = wsum > 0.f ? L + __logf(wsum) : -INFINITY;
}

template <int D>
int launch(const FwdSplitLaunch &a, cudaStream_t stream) {
    using C = Cfg<D>;
    CUtensorMap mq, mk, mv;
    const uint64_t dq = uint64_t(a.d);
    if (!encode_bf16_3d(&mq, a.q, dq, uint64_t(a.N), uint64_t(a.B) * a.Hq, 64, kTileM) ||
        !encode_bf16_3d(&mk, a.k, dq, uint64_t(a.N), uint64_t(a.B) * a.Hkv, 64, kBlockN) ||
        !encode_bf16_3d(&mv, a.v, dq, uint64_t(a.N), uint64_t(a.B) * a.Hkv, 64, kBlockN))
        return note_cuda_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (split-KV forward)");
    Params p;
    p.part_o = a.part_o;
    p.part_lse = a.part_lse;
    p.B = a.B;
    p.N = a.N;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.d_store = a.d;
    p.causal = a.causal ? 1 : 0;
    p.nb = unit_blocks(a.N);
    p.splits = a.splits;
    p.chunk_blocks = a.chunk_keys / kBlockN;
    p.total_units = (long long)a.B * a.Hq * p.nb * a.splits;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.wait_ns = a.wait_ns;
    p.sched_slot = int(g_fwd_split_launch_seq.fetch_add(1) % kSchedSlots);
    auto kernel = fwd_split_kernel<D>;
    static bool attr_set[kMaxDevices] = {};
    const int dev = slot_for_device();
    if (dev < 0 || !attr_set[dev]) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncGetAttributes(fwd_split_kernel)");
        if (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads)
            return note_cuda_error(cudaErrorInvalidConfiguration,
                                   "fwd_split_kernel register count differs from the setmaxnreg split");
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncSetAttribute(fwd_split_kernel)");
        if (dev >= 0) attr_set[dev] = true;
    }
    long long grid = p.total_units;
    if (grid > a.num_sms) grid = a.num_sms;
    kernel<<<dim3(unsigned(grid)), dim3(kThreads), C::kSmemBytes, stream>>>(mq, mk, mv, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return note_cuda_error(e, "fwd_split_kernel launch");
    const long long rows = (long long)a.B * a.Hq * a.N;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return ATTN_ERR_ARG;
    split_merge_kernel<<<dim3(unsigned(blocks)), dim3(256), 0, stream>>>(
        a.part_o, a.part_lse, reinterpret_cast<__nv_bfloat16 *>(a.o), a.lse, rows, a.N, a.d, a.splits, a.chunk_keys,
        a.causal ? 1 : 0);
    e = cudaGetLastError();
    return e == cudaSuccess ? 0 : note_cuda_error(e, "split_merge_kernel launch");
}

}  // namespace fwd3

int fwd_split_launch(const FwdSplitLaunch &a, cudaStream_t stream) {
    if (a.d <= 64) return fwd3::launch<64>(a, stream);
    return fwd3::launch<128>(a, stream);
}

cudaError_t fwd_split_take_status(int *bits) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_fwd_split_status, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_fwd_split_status, &zero, sizeof(int));
}

}  // namespace attn
