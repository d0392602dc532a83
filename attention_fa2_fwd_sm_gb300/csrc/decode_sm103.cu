// decode_sm103.cu -- split-KV grouped-query decode (one query row per query
// head) and the log-sum-exp merge of the per-split partial states.
//
// kernbench2 "Fused Grouped-Query Attention": a decode step processes a
// single query position against the whole KV history, so its time is the
// time to stream the KV cache from HBM; each KV head is shared by a group of
// G query heads; the KV sequence is split and the running softmax states
// (m, l, O) of the pieces are reduced (section "Inference with Long-Context
// Length", Case 4).  Here the pieces are CTAs of one GPU and the reduction is
// a second kernel.
//
// Decode CTA = (split s, KV head g, batch b); 4 consumer warps + 1 TMA warp.
// The chunk of keys [lo, hi) of the split streams through a ring of 64-key
// stages (K and V tiles, 128-byte swizzled, loaded by TMA).  Each consumer
// warp takes 16 keys of a stage and computes, for the G <= 16 query heads of
// the group at once, S = Q K^T and O += P V with m16n8k16 bf16 MMAs (query
// heads on the M dimension), keeping its own online-softmax state.  At the
// end the four warp states are combined through shared memory into the
// split's partial (O_s normalised, lse_s), or into O directly when there is a
// single split.
//
// Ragged multi-user batches (attn_decode_varlen): one chunk size for the whole
// batch, chosen on the device from the total number of cached keys, cuts every
// sequence into chunks; a plan kernel writes the resulting work list (batch
// entry, key range) and each decode CTA takes one item of it, so a long
// sequence is spread over many CTAs however short the others are.  The
// reduction then has two levels, as in the kernbench2 decode family's
// multi-user "two-level reduce-to-root" (short-context section): the warps of
// a CTA are combined in shared memory, and one merge per (user, query head)
// reduces that user's chunks.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {

static __device__ int g_decode_status;

// Built-in scratch for attn_decode_noalloc: the split partials of callers
// that cannot hand the library a workspace.  A fixed-size array that is part
// of the library image, so every GPU that loads the library holds it until
// the process exits.  Host code must not use the symbol itself as a pointer
// (on the host it names a stand-in, not device memory); decode_noalloc_scratch
// looks up the real device address.
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[kDecodeNoAllocScratchBytes];

namespace dec {

constexpr int kKeysPerStage = 64;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxGroup = 16;
constexpr int kChunkGranule = 64;

// K/V ring depth.  Three 32 KiB stages at d = 128 let two CTAs share an SM;
// a grid of at most one CTA per SM (short batches, latency-bound) takes six,
// twice the bytes in flight per CTA.
template <int D>
constexpr int kBaseStages = (D == 128) ? 3 : 6;
template <int D>
constexpr int kDeepStages = 6;

template <int D, int S = kBaseStages<D>>
struct Cfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kChunkBytes = kKeysPerStage * 128;      // 64 keys x 128 bytes
    static constexpr int kTileBytes = kKeysPerStage * D * 2;     // one K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = S;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kCombineBytes = kConsumerWarps * (kMaxGroup * D + 2 * kMaxGroup) * 4;
    static constexpr int kDataBytes = kRingBytes > kCombineBytes ? kRingBytes : kCombineBytes;
    static constexpr int kNumBars = 2 * kStages;
    static constexpr int kSmemBytes = kDataBytes + kNumBars * 8 + 16 + 1024;
};

struct Params {
    const __nv_bfloat16 *q;
    const int *seqlens;
    __nv_bfloat16 *o;
    float *ws_o, *ws_lse;
    const int *plan;  // work list of the varlen path (null: split grid)
    int B, Hq, Hkv, G, max_seqlen, num_splits;
    float scale_log2;
    unsigned long long wait_ns;
};

// Varlen plan layout (ints): [0] item count, [1] chunk size C, [2, 2 + B)
// first item of each batch entry, [2 + B, 2 + 2B) its item count, then the
// items as (b, lo, hi) triples.
__host__ __device__ inline int plan_items_offset(int B) { return 2 + 2 * B; }

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Byte address of the 16-byte unit `u` (elements 8u..8u+7) of key row `k` of a
// 64-key tile stored as D/64 chunks of 128-byte rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_unit_addr(uint32_t tile, int k, int u) {
    return tile + (u >> 3) * (kKeysPerStage * 128) + k * 128 + (((u & 7) ^ (k & 7)) << 4);
}

// Zero the bf16 halves of a V fragment register whose keys lie at or beyond
// `n_valid` (keys k_lo and k_lo + 1 live in the low and high halves).
__device__ __forceinline__ uint32_t mask_pair(uint32_t r, int k_lo, int n_valid) {
    if (k_lo >= n_valid) r &= 0xffff0000u;
    if (k_lo + 1 >= n_valid) r &= 0x0000ffffu;
    return r;
}

template <int D, int S>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const Params p) {
    using C = Cfg<D, S>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kDataBytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + C::kNumBars);
    int *status = &g_decode_status;

    // Varlen grid: (KV head, work item), so the KV heads of one sequence are
    // launched together as in the split grid (split, KV head, batch).
    const int split = p.plan ? blockIdx.y : blockIdx.x;
    const int g = p.plan ? blockIdx.x : blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // In work-list mode the plan kernel ahead of this grid may still be
    // running (programmatic launch): wait for its list.
    griddep_wait();
    int b, lo, hi;
    if (p.plan) {
        // Varlen: this CTA is work item `split` of the plan (the grid is an
        // upper bound on the item count; CTAs past it have nothing to do).
        if (split >= p.plan[0]) return;
        const int *it = p.plan + plan_items_offset(p.B) + 3 * split;
        b = it[0];
        lo = it[1];
        hi = it[2];
    } else {
        b = blockIdx.z;
        int seqlen = p.seqlens[b];
        seqlen = seqlen < 0 ? 0 : (seqlen > p.max_seqlen ? p.max_seqlen : seqlen);
        int per = (seqlen + p.num_splits - 1) / p.num_splits;
        const int chunk = (per + kChunkGranule - 1) / kChunkGranule * kChunkGranule;
        lo = min(split * chunk, seqlen);
        hi = min(lo + chunk, seqlen);
    }
    const int ntiles = (hi - lo + kKeysPerStage - 1) / kKeysPerStage;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(bars + s), 1);                          // full
            mbar_init(smem_u32(bars + C::kStages + s), kConsumerWarps);  // empty
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // Per-warp online-softmax state for rows (query heads) r = lane/4 and r + 8.
    float m_st[2] = {-INFINITY, -INFINITY};
    float l_st[2] = {0.f, 0.f};
    float acc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;

    int issued = 0;  // tiles whose copies were issued (producer lane only)
    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            for (int i = 0; i < ntiles; ++i) {
                const int s = i % C::kStages;
                const int round = i / C::kStages;
                if (round > 0 && !mbar_wait_bounded(smem_u32(bars + C::kStages + s), (round - 1) & 1,
                                                    p.wait_ns, abort_flag, status))
                    break;
                const uint32_t fb = smem_u32(bars + s);
                mbar_arrive_expect_tx(fb, C::kStageBytes);
                const uint32_t kt = smem_u32(smem + s * C::kStageBytes);
                const int key0 = lo + i * kKeysPerStage;
                const int plane = b * p.Hkv + g;
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(kt + c * C::kChunkBytes, &tmK, fb, c * 64, key0, plane);
                    tma_load_3d(kt + C::kTileBytes + c * C::kChunkBytes, &tmV, fb, c * 64, key0, plane);
                }
                issued = i + 1;
            }
        }
    } else {
        // ------------------------------------------------------------ consumer
        const int gq = lane >> 2, tq = lane & 3;
        // Q fragments (A operand, rows = query heads of the group, k = head dim).
        uint32_t qa[D / 16][4];
        const int h0 = g * p.G;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = gq + ((i & 1) ? 8 : 0);
                const int col = ks * 16 + tq * 2 + ((i & 2) ? 8 : 0);
                uint32_t v = 0;
                if (row < p.G)
                    v = *reinterpret_cast<const uint32_t *>(p.q + ((size_t)(b * p.Hq + h0 + row)) * D + col);
                qa[ks][i] = v;
            }
        }
        const float sl2 = p.scale_log2;
        for (int i = 0; i < ntiles; ++i) {
            const int s = i % C::kStages;
            if (!mbar_wait_warp(smem_u32(bars + s), (i / C::kStages) & 1, p.wait_ns, abort_flag, status))
                break;
            const int kw = lo + i * kKeysPerStage + warp * 16;  // first key of this warp
            const int n_valid = min(16, hi - kw);
            if (n_valid > 0) {
                const uint32_t kt = smem_u32(smem + s * C::kStageBytes);
                const uint32_t vt = kt + C::kTileBytes;
                float sc[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[h][e] = 0.f;
                {
                    const int sub = lane >> 3, rr = lane & 7;
                    const int key = warp * 16 + ((sub & 2) ? 8 : 0) + rr;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(tile_unit_addr(kt, key, 2 * ks + (sub & 1)), b0, b1, b2, b3);
                        mma_bf16_16816(sc[0], qa[ks], b0, b1);
                        mma_bf16_16816(sc[1], qa[ks], b2, b3);
                    }
                }
                // scores in log2 units, masked past the chunk end
                float x[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int kl = h * 8 + tq * 2 + (e & 1);
                        x[h][e] = kl < n_valid ? sc[h][e] * sl2 : -INFINITY;
                    }
                uint32_t pa[4];
                float corr[2];
#pragma unroll
                for (int rsel = 0; rsel < 2; ++rsel) {  // rows gq (e = 0,1) and gq + 8 (e = 2,3)
                    float mx = fmaxf(fmaxf(x[0][2 * rsel], x[0][2 * rsel + 1]),
                                     fmaxf(x[1][2 * rsel], x[1][2 * rsel + 1]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float m_new = fmaxf(m_st[rsel], mx);
                    corr[rsel] = m_new == -INFINITY ? 1.f : fast_exp2(m_st[rsel] - m_new);  // 0 when the old max is -inf
                    m_st[rsel] = m_new;
                    const float nm = m_new == -INFINITY ? 0.f : -m_new;
                    const float p00 = fast_exp2(x[0][2 * rsel] + nm), p01 = fast_exp2(x[0][2 * rsel + 1] + nm);
                    const float p10 = fast_exp2(x[1][2 * rsel] + nm), p11 = fast_exp2(x[1][2 * rsel + 1] + nm);
                    l_st[rsel] = l_st[rsel] * corr[rsel] + (p00 + p01 + p10 + p11);
                    pa[rsel] = pack_bf16x2(p00, p01);      // a0 (row gq) / a1 (row gq+8), keys 2tq..
                    pa[2 + rsel] = pack_bf16x2(p10, p11);  // a2 / a3, keys 8+2tq..
                }
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    acc[n][0] *= corr[0];
                    acc[n][1] *= corr[0];
                    acc[n][2] *= corr[1];
                    acc[n][3] *= corr[1];
                }
                {
                    const int sub = lane >> 3, rr = lane & 7;
                    const int key = warp * 16 + ((sub & 1) ? 8 : 0) + rr;
#pragma unroll
                    for (int nt = 0; nt < D / 16; ++nt) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(tile_unit_addr(vt, key, 2 * nt + (sub >> 1)), b0, b1, b2, b3);
                        if (n_valid < 16) {
                            b0 = mask_pair(b0, 2 * tq, n_valid);
                            b1 = mask_pair(b1, 8 + 2 * tq, n_valid);
                            b2 = mask_pair(b2, 2 * tq, n_valid);
                            b3 = mask_pair(b3, 8 + 2 * tq, n_valid);
                        }
                        mma_bf16_16816(acc[2 * nt], pa, b0, b1);
                        mma_bf16_16816(acc[2 * nt + 1], pa, b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(bars + C::kStages + s));
        }
    }

    // ------------------------------------------------ combine the four warps
    griddep_launch_dependents();  // the merge grid may be scheduled now
    __syncthreads();
    if (*abort_flag) {
        // A wait ran out somewhere.  Before the CTA exits, wait (bounded, with
        // a fixed limit) for the copies of the last fill of every ring slot so
        // that none is still writing shared memory; outputs stay unwritten.
        if (warp == kConsumerWarps && lane == 0) {
            volatile int no_abort = 0;
            for (int i = max(0, issued - C::kStages); i < issued; ++i)
                if (!mbar_wait_bounded(smem_u32(bars + i % C::kStages), (i / C::kStages) & 1,
                                       1000000000ull, &no_abort, status))
                    atomicOr(status, kStatusDrainTimeout);
        }
        return;
    }
    // Every issued tile was consumed: the ring can be reused for the combine.
    float *cw = reinterpret_cast<float *>(smem);  // [warp][16][D] O, then [warp][16] m, [warp][16] l
    float *cm = cw + kConsumerWarps * kMaxGroup * D;
    float *cl = cm + kConsumerWarps * kMaxGroup;
    if (warp < kConsumerWarps) {
        const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
        for (int rsel = 0; rsel < 2; ++rsel) {
            float l = l_st[rsel];
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            l_st[rsel] = l;
        }
        float *ow = cw + warp * kMaxGroup * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            const int col = n * 8 + tq * 2;
            ow[gq * D + col] = acc[n][0];
            ow[gq * D + col + 1] = acc[n][1];
            ow[(gq + 8) * D + col] = acc[n][2];
            ow[(gq + 8) * D + col + 1] = acc[n][3];
        }
        if (tq == 0) {
            cm[warp * kMaxGroup + gq] = m_st[0];
            cm[warp * kMaxGroup + gq + 8] = m_st[1];
            cl[warp * kMaxGroup + gq] = l_st[0];
            cl[warp * kMaxGroup + gq + 8] = l_st[1];
        }
    }
    __syncthreads();
    const int G = p.G;
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int row = idx / D, col = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cm[w * kMaxGroup + row]);
        float wsum = 0.f, osum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float f = fast_exp2(cm[w * kMaxGroup + row] - M);
                wsum += f * cl[w * kMaxGroup + row];
                osum += f * cw[(w * kMaxGroup + row) * D + col];
            }
        }
        const float o = wsum > 0.f ? osum / wsum : 0.f;
        const int h = g * G + row;
        if (p.plan) {
            const size_t pi = (size_t)split * p.Hq + h;
            p.ws_o[pi * D + col] = o;
            if (col == 0) p.ws_lse[pi] = wsum > 0.f ? (M + __log2f(wsum)) * 0.69314718055994531f : -INFINITY;
        } else if (p.num_splits == 1) {
            p.o[(size_t)(b * p.Hq + h) * D + col] = __float2bfloat16_rn(o);
        } else {
            const size_t pi = (size_t)(b * p.Hq + h) * p.num_splits + split;
            p.ws_o[pi * D + col] = o;
            if (col == 0) p.ws_lse[pi] = wsum > 0.f ? (M + __log2f(wsum)) * 0.69314718055994531f : -INFINITY;
        }
    }
}

// Merge: L = max_s lse_s, w_s = exp(lse_s - L), O = sum_s w_s O_s / sum_s w_s.
// The block stages the lse values in shared memory (one load per thread) and
// issues the partial outputs eight splits at a time, so the merge costs a few
// memory round trips instead of one per split; the sums run over s in order.
template <int D>
__global__ void __launch_bounds__(D) merge_kernel(const float *ws_o, const float *ws_lse,
                                                  __nv_bfloat16 *o, int num_splits) {
    __shared__ float lse_sh[kDecodeMaxSplits];
    __shared__ float max_sh[D / 32];
    griddep_wait();  // launched behind the decode grid, which writes the partials
    const int bh = blockIdx.x, col = threadIdx.x;
    const float *lse = ws_lse + (size_t)bh * num_splits;
    const float *po = ws_o + (size_t)bh * num_splits * D;
    float L = -INFINITY;
    for (int s = col; s < num_splits; s += D) {
        const float v = lse[s];
        lse_sh[s] = v;
        L = fmaxf(L, v);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L = fmaxf(L, __shfl_xor_sync(0xffffffffu, L, off));
    if ((col & 31) == 0) max_sh[col >> 5] = L;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < D / 32; ++w) L = fmaxf(L, max_sh[w]);
    float wsum = 0.f, acc = 0.f;
    if (L != -INFINITY) {
        int s = 0;
        for (; s + 8 <= num_splits; s += 8) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = po[(size_t)(s + i) * D + col];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float w = __expf(lse_sh[s + i] - L);
                wsum += w;
                acc += w * v[i];
            }
        }
        for (; s < num_splits; ++s) {
            const float w = __expf(lse_sh[s] - L);
            wsum += w;
            acc += w * po[(size_t)s * D + col];
        }
    }
    o[(size_t)bh * D + col] = __float2bfloat16_rn(wsum > 0.f ? acc / wsum : 0.f);
}

// Varlen plan, one CTA: total keys T = sum_b min(max(seqlens[b], 0), max_seqlen);
// chunk C = max(min_chunk, ceil(T * Hkv / target) rounded up to 64); sequence
// b gets n_b = ceil(len_b / C) items [c C, min(c C + C, len_b)), numbered
// consecutively by b.  The item count is at most ceil(target / Hkv) + B.
__global__ void __launch_bounds__(256) varlen_plan_kernel(const int *seqlens, int B, int max_seqlen, int Hkv,
                                                          long long target, int min_chunk, int *plan) {
    __shared__ long long warp_part[8];
    __shared__ int chunk_s;
    griddep_launch_dependents();  // the decode grid may be scheduled; it waits for this one
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int per = (B + 255) / 256;  // consecutive sequences per thread
    const int b0 = min(t * per, B), b1 = min(b0 + per, B);
    auto len_of = [&](int b) {
        const int n = seqlens[b];
        return n < 0 ? 0 : (n > max_seqlen ? max_seqlen : n);
    };
    // Inclusive block scan of one value per thread (warp shuffles, then the
    // eight warp totals); returns the thread's exclusive prefix and the total.
    auto block_scan = [&](long long v, long long &total) {
        long long x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        __syncthreads();
        if (lane == 31) warp_part[w] = x;
        __syncthreads();
        long long before = 0;
        total = 0;
        for (int i = 0; i < 8; ++i) {
            if (i < w) before += warp_part[i];
            total += warp_part[i];
        }
        return before + x - v;
    };
    long long keys = 0;
    for (int b = b0; b < b1; ++b) keys += len_of(b);
    long long T = 0;
    block_scan(keys, T);
    if (t == 0) {
        long long c = (T * Hkv + target - 1) / target;
        c = (c + kChunkGranule - 1) / kChunkGranule * kChunkGranule;
        if (c < min_chunk) c = min_chunk;
        chunk_s = int(c < 0x40000000LL ? c : 0x40000000LL);
        plan[1] = chunk_s;
    }
    __syncthreads();
    const int C = chunk_s;
    long long mine = 0;  // items of this thread's sequences
    for (int b = b0; b < b1; ++b) mine += (len_of(b) + C - 1) / C;
    long long count = 0;
    int first = int(block_scan(mine, count));
    if (t == 0) plan[0] = int(count);
    int *items = plan + plan_items_offset(B);
    for (int b = b0; b < b1; ++b) {
        const int len = len_of(b);
        const int n = (len + C - 1) / C;
        plan[2 + b] = first;
        plan[2 + B + b] = n;
        for (int c = 0; c < n; ++c) {
            int *it = items + 3 * (first + c);
            it[0] = b;
            it[1] = c * C;
            it[2] = min(c * C + C, len);
        }
        first += n;
    }
}

// Varlen merge: for (b, h), the n_b partials of b's items.  n_b = 0 gives O = 0.
template <int D>
__global__ void __launch_bounds__(D) merge_varlen_kernel(const int *plan, int B, int Hq, const float *ws_o,
                                                         const float *ws_lse, __nv_bfloat16 *o) {
    griddep_wait();  // launched behind the decode grid, which writes the partials
    const int bh = blockIdx.x, col = threadIdx.x;
    const int b = bh / Hq, h = bh % Hq;
    const int f = plan[2 + b], n = plan[2 + B + b];
    float L = -INFINITY;
    for (int s = f; s < f + n; ++s) L = fmaxf(L, ws_lse[(size_t)s * Hq + h]);
    float wsum = 0.f, acc = 0.f;
    if (L != -INFINITY) {
        for (int s = f; s < f + n; ++s) {
            const float w = __expf(ws_lse[(size_t)s * Hq + h] - L);
            wsum += w;
            acc += w * ws_o[((size_t)s * Hq + h) * D + col];
        }
    }
    o[(size_t)bh * D + col] = __float2bfloat16_rn(wsum > 0.f ? acc / wsum : 0.f);
}

// Launch `kernel` allowing it to start before the grid ahead of it on the
// stream has finished (it must griddep_wait() before reading that grid's
// output).
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int D, int S>
int launch(const DecodeLaunch &a, cudaStream_t stream) {
    using C = Cfg<D, S>;
    CUtensorMap mk, mv;
    if (!encode_bf16_3d(&mk, a.kcache, D, uint64_t(a.max_seqlen), uint64_t(a.B) * a.Hkv, 64,
                        kKeysPerStage) ||
        !encode_bf16_3d(&mv, a.vcache, D, uint64_t(a.max_seqlen), uint64_t(a.B) * a.Hkv, 64,
                        kKeysPerStage))
        return note_cuda_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (decode)");
    Params p;
    p.q = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    p.seqlens = a.seqlens;
    p.o = reinterpret_cast<__nv_bfloat16 *>(a.o);
    p.ws_o = a.ws_o;
    p.ws_lse = a.ws_lse;
    p.plan = a.plan;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.max_seqlen = a.max_seqlen;
    p.num_splits = a.num_splits;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.wait_ns = a.wait_ns;
    static bool attr_set[kMaxDevices] = {};  // per instantiation and device
    const int dev = slot_for_device();
    if (dev < 0 || !attr_set[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(
            decode_kernel<D, S>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncSetAttribute(decode_kernel)");
        if (dev >= 0) attr_set[dev] = true;
    }
    // The kernels after the first are launched with programmatic stream
    // serialization: each may be scheduled while the one ahead drains and
    // waits (griddep_wait) for it before touching its output.
    if (a.plan) {
        varlen_plan_kernel<<<1, 256, 0, stream>>>(a.seqlens, a.B, a.max_seqlen, a.Hkv, a.varlen_target,
                                                  a.varlen_min_chunk, a.plan);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return note_cuda_error(e, "varlen_plan_kernel launch");
        e = launch_programmatic(decode_kernel<D, S>, dim3(a.Hkv, a.varlen_max_items, 1), dim3(kThreads),
                                C::kSmemBytes, stream, mk, mv, p);
        if (e != cudaSuccess) return note_cuda_error(e, "decode_kernel launch (varlen)");
        e = launch_programmatic(merge_varlen_kernel<D>, dim3(a.B * a.Hq), dim3(D), 0, stream,
                                (const int *)a.plan, a.B, a.Hq, (const float *)a.ws_o, (const float *)a.ws_lse, p.o);
        return e == cudaSuccess ? 0 : note_cuda_error(e, "merge_varlen_kernel launch");
    }
    decode_kernel<D, S><<<dim3(a.num_splits, a.Hkv, a.B), dim3(kThreads), C::kSmemBytes, stream>>>(mk, mv, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return note_cuda_error(e, "decode_kernel launch");
    if (a.num_splits > 1) {
        e = launch_programmatic(merge_kernel<D>, dim3(a.B * a.Hq), dim3(D), 0, stream, (const float *)a.ws_o,
                                (const float *)a.ws_lse, p.o, a.num_splits);
        if (e != cudaSuccess) return note_cuda_error(e, "merge_kernel launch");
    }
    return 0;
}

}  // namespace dec

int decode_launch(const DecodeLaunch &a, cudaStream_t stream) {
    // The split grid of at most one CTA per SM runs the deep ring; the varlen
    // grid (an upper bound on its work items) keeps the base ring.
    const bool deep = !a.plan && a.num_sms > 0 && (long long)a.num_splits * a.Hkv * a.B <= a.num_sms;
    if (a.d == 64) return dec::launch<64, dec::kBaseStages<64>>(a, stream);
    return deep ? dec::launch<128, dec::kDeepStages<128>>(a, stream)
                : dec::launch<128, dec::kBaseStages<128>>(a, stream);
}

cudaError_t decode_noalloc_scratch(void **ptr) {
    // One lookup per device, made with that device current; later calls reuse it.
    static void *addr[kMaxDevices] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

cudaError_t decode_take_status(int *bits) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_decode_status, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(int));
}

}  // namespace attn
