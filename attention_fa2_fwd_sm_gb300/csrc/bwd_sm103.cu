// bwd_sm103.cu -- FlashAttention-2 style backward pass for sm_103a.
//
// Gradients of O = softmax(scale * Q K^T) V ("Optimizing Attention on GPUs by
// Exploiting GPU Architectural NUMA Effects", detail page, section 4
// equation; the same pages measure an FA2 backward pass, section 5 "backward
// pass") for an output gradient dO, by the chain rule:
//   P = exp(scale * Q K^T - lse)      (lse saved by the forward pass)
//   dV = P^T dO,   dP = dO V^T,   Delta = rowsum(dO * O)
//   dS = P * (dP - Delta),   dQ = scale * dS K,   dK = scale * dS^T Q
// with the causal mask and grouped-query heads as in the forward pass (the
// gradient of a KV head sums over the query heads that read it).
//
// Three kernels, in stream order:
//   bwd_pre_kernel   Delta and lse * log2(e) per query row, into a padded
//                    fp32 workspace (+inf / 0 past the last row, which makes
//                    padded query rows drop out of every product).
//   dkdv_kernel<D>   one unit = 128 keys of one KV head; K and V stay in shared
//                    memory while the query blocks of every query head of the
//                    group stream through a TMA ring (with their lse and Delta):
//                    S^T = K Q^T and dP^T = V dO^T (SS MMAs into TMEM), P^T
//                    and dS^T in bf16 written back over them, then dV += P^T dO
//                    and dK += dS^T Q (TS MMAs, dO and Q read MN-major).
//   dq_kernel<D>     one unit = 256 query rows of one query head (two 128-row
//                    tiles sharing every K/V block); Q and dO stay in shared
//                    memory while K/V blocks stream: S = Q K^T, then dP =
//                    dO V^T in the same TMEM buffer, dS in bf16 over it,
//                    dQ += dS K (TS MMA); the two tiles alternate on the
//                    tensor core.
// Splitting dQ into its own pass recomputes S and dP (seven products instead of
// five) but needs no atomic accumulation: every output element is written
// once, by one CTA, and the result does not depend on the schedule.
//
// Query-head split of the dK/dV pass (non-causal GQA with few units).  A dK/dV unit
// streams every query head of its KV head, so GQA has G times fewer, G
// times longer units than MHA of the same work; GQA 64/8 at 8K keys has
// 512, 3.4 waves on 152 SMs, and the last wave runs a third full.  With a
// workspace large enough, the pass then runs as if each KV head were s
// "virtual" KV heads of G / s query heads (the orders, windows and host maps
// unchanged, over B * Hkv * s pairs), each unit writing fp32 partial dK and
// dV of its query heads; dkdv_reduce_kernel sums the s partials in a fixed
// order.  The result is deterministic and the same for every tile order.
//
// Both main kernels are persistent (one CTA per SM) and take units from an
// atomic counter in the chosen order.  Head-first keeps the CTAs that run at
// the same time on one Attention Compute Cluster, so the operand they all
// stream (the group's Q/dO in dkdv, the head's K/V in dq) is read from HBM
// about once and then served by L2 (detail page, section 2 Q2).
// Roles (384 threads): warp 0 TMA producer, warp 1 tcgen05 issuer and TMEM
// owner, warps 2-3 idle, warps 4-11 elementwise / epilogue.  Warp w owns TMEM
// lanes [32 (w % 4), +32), one row of the tile per thread; the two warps of a
// lane quarter split the row's 128 columns (and, in the epilogue, the D
// output columns) between them.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "attn_internal.h"
#include "sm103_ptx.cuh"
#include "dkdv_order.cuh"
#include "tile_order.cuh"

namespace attn {

static __device__ int g_bwd_status;

// Work counters (as in the forward kernel): per launch slot and kernel
// {next unit, CTAs finished}; the last CTA of a launch resets its pair.
constexpr int kBwdSchedSlots = 64;
static __device__ unsigned int g_bwd_work[kBwdSchedSlots][2][2];
// Launch sequence number behind the slot choice: one counter for both head
// dimensions, since their launches share g_bwd_work.
static std::atomic<unsigned int> g_bwd_launch_seq{0};

namespace bwd {

// (d0, d1) = (a0 - b0, a1 - b1) and (a0 * b0, a1 * b1) as paired fp32 operations.
__device__ __forceinline__ void fsub2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "sub.rn.f32x2 d, a, b;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void fmul2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

constexpr int kRows = 128;     // rows per tile (keys in dkdv, queries in dq)
constexpr int kThreads = 384;  // 12 warps: 4 control, 8 elementwise
constexpr int kEwWarps = 8;    // two per TMEM lane quarter, each on half of the columns
constexpr int kTmemCols = 512;
// Register split after set-up (as in the forward kernel): the launch gives
// 168 registers per thread (384 x 168 = 64512); the control warpgroup drops
// to kCtrl (the issue loops' state) and the two elementwise warpgroups rise
// to kEw.  The host refuses a build whose launch register count differs.
// d = 128: 136 / 184.  d <= 64: 120 / 192, which cuts the elementwise warps'
// spills from about 100 to 4 bytes in dK/dV and ran the backward 2.4% faster
// at d = 64 and d = 56 (at d = 128 it measured 0.5% slower); the d <= 64 dQ
// kernel's control warpgroup takes 112 (its spills 24 / 76 -> 8 / 8 bytes,
// +1.4% at d = 64).
constexpr int kLaunchRegs = 168;
template <int D, bool kDq = false>
struct BwdRegs {
    static constexpr int kCtrl = D <= 64 ? (kDq ? 112 : 120) : 136;
    static constexpr int kEw = D <= 64 ? 192 : 184;
    static_assert(128 * kCtrl + 256 * kEw <= kThreads * kLaunchRegs, "register split");
};

struct Params {
    __nv_bfloat16 *out0, *out1;  // dkdv: dK, dV; dq: dQ (out1 unused)
    const float *nlse2;          // [B*Hq, npad]  -lse * log2(e), -inf past N
    const float *delta;          // [B*Hq, npad]  rowsum(dO * O), 0 past N
    int B, N, npad, Hq, Hkv, G, d_store, causal, order, nblk;
    int kv_window;  // dkdv head-first: (batch, KV head) pairs interleaved per window
    // dkdv query-head split: Hkv and G above are the virtual KV heads (Hkv *
    // kv_split) and their query heads (G / kv_split); K and V come from real
    // KV head g / kv_split of hkv_real, and the partials go to part.
    int kv_split, hkv_real;
    float *part;  // [2][B * Hkv][N][d_store] fp32: dK (scaled), then dV
    long long total_units;
    float scale, scale_log2;
    unsigned long long wait_ns;
    int sched_slot;
};

// ------------------------------------------------------------------ pre-pass

// Delta = sum_c dO[c] * O[c] (fp32) and -lse * log2(e) (negated, so the
// exponent argument is one FMA) per padded query row; rows at or past N get
// -inf and 0.  Eight lanes share a row, each reading 16-byte pieces of O and
// dO (a row of d bf16 is d / 8 pieces: 7, 8 or 16), so a warp covers four
// rows at a time.  (One warp per row with 4-byte loads ran at under half of
// the HBM bandwidth.)
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o,
                                                      const __nv_bfloat16 *__restrict__ dout,
                                                      const float *__restrict__ lse, float *nlse2,
                                                      float *delta, int N, int npad, int d,
                                                      long long rows) {
    const int lane = threadIdx.x & 31;
    const int l8 = lane & 7;        // lane within the row's group of eight
    const int pieces = d / 8;       // 16-byte pieces per row
    const long long groups = (rows + 3) / 4;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long gi = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); gi < groups;
         gi += warps) {
        const long long r = gi * 4 + (lane >> 3);
        const bool valid = r < rows;
        const long long bh = valid ? r / npad : 0;
        const int n = valid ? int(r % npad) : 0;
        const bool live = valid && n < N;
        float acc = 0.f;
        if (live) {
            const size_t base = ((size_t)bh * N + n) * d;
            for (int c = l8; c < pieces; c += 8) {
                const uint4 a = *reinterpret_cast<const uint4 *>(o + base + (size_t)c * 8);
                const uint4 g = *reinterpret_cast<const uint4 *>(dout + base + (size_t)c * 8);
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&aw[k]));
                    const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&gw[k]));
                    acc = fmaf(af.x, gf.x, acc);
                    acc = fmaf(af.y, gf.y, acc);
                }
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if (valid && l8 == 0) {
            nlse2[r] = live ? -(lse[(size_t)bh * N + n] * 1.4426950408889634f) : -INFINITY;
            delta[r] = live ? acc : 0.f;
        }
    }
}

// ------------------------------------------------------------------ schedule

// dkdv unit -> (b, kv head g, key block j): dkdv_unit_to_tile (the
// scheduler header), with the launch's window.
using KvUnit = KvTile;
__device__ __forceinline__ KvUnit kv_unit(const Params &p, long long u) {
    return dkdv_unit_to_tile(p.order, u, p.B, p.Hkv, p.nblk, p.kv_window);
}

// The i-th unit of this CTA (naive head-first: the CTA's own index), or -1.
__device__ __forceinline__ long long fetch_unit(const Params &p, int kernel, long long i) {
    if (p.order == kNaiveHeadFirst) return i == 0 ? (long long)blockIdx.x : -1;
    const unsigned int u = atomicAdd(&g_bwd_work[p.sched_slot][kernel][0], 1u);
    return (long long)u < p.total_units ? (long long)u : -1;
}

__device__ __forceinline__ void finish_schedule(const Params &p, int kernel) {
    if (threadIdx.x == 0 && p.order != kNaiveHeadFirst) {
        __threadfence();
        const unsigned int done = atomicAdd(&g_bwd_work[p.sched_slot][kernel][1], 1u);
        if (done == gridDim.x - 1) {
            atomicExch(&g_bwd_work[p.sched_slot][kernel][0], 0u);
            atomicExch(&g_bwd_work[p.sched_slot][kernel][1], 0u);
        }
    }
}

// Store half `half` of the columns of one row of a TMEM accumulator (D fp32
// columns at `t_row`) to global memory as bf16, multiplied by `mul`; columns
// at or past d_store are clipped.
template <int D>
__device__ __forceinline__ void store_half_row(uint32_t t_row, int half, __nv_bfloat16 *dst, bool row_ok,
                                               int d_store, float mul) {
#pragma unroll
    for (int cc = 0; cc < D / 64; ++cc) {
        const int c = half * (D / 64) + cc;  // 32-column chunk
        uint32_t v[32];
        tmem_ld32(t_row + c * 32, v);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
        if (row_ok) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int col = c * 32 + g * 8;
                if (col < d_store)
                    *reinterpret_cast<uint4 *>(dst + col) =
                        make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
            }
        }
    }
}

// D (+)= A B^T over the head dimension (K-major A and B in 128-byte-swizzled
// 64-column chunks), issued in groups of four MMAs from one asm block by
// the warp's elected lane (the caller is the whole MMA warp).
template <int D, int kChunkBytes>
__device__ __forceinline__ void ss_product(uint32_t d_tmem, uint64_t a0, uint64_t b0, uint32_t idesc) {
#pragma unroll
    for (int g = 0; g < D / 64; ++g) {
        uint64_t a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t off = uint64_t((g * kChunkBytes + i * 32) >> 4);
            a[i] = a0 + off;
            b[i] = b0 + off;
        }
        tc_mma_ss_x4_elect(d_tmem, a, b, idesc, g > 0 ? 1u : 0u);
    }
}

// D (+)= A B with A (bf16) in TMEM from column a_tmem and B read MN-major,
// K = 16 NK rows; the first MMA accumulates iff `acc`.
template <int NK>
__device__ __forceinline__ void ts_product(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0, uint32_t idesc, bool acc) {
#pragma unroll
    for (int g = 0; g < NK / 4; ++g) {
        uint32_t a[4];
        uint64_t b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int kk = g * 4 + i;
            a[i] = a_tmem + kk * 8;
            b[i] = b0 + uint64_t((kk * 16 * 128) >> 4);
        }
        tc_mma_ts_x4_elect(d_tmem, a, b, idesc, (acc || g > 0) ? 1u : 0u);
    }
}

// A 1-D bulk copy global -> shared memory completing on an mbarrier (both
// addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}


// store_half_row in fp32 (the split dK/dV pass's partials).
template <int D>
__device__ __forceinline__ void store_half_row_f32(uint32_t t_row, int half, float *dst, bool row_ok, int d_store,
                                                   float mul) {
#pragma unroll
    for (int cc = 0; cc < D / 64; ++cc) {
        const int c = half * (D / 64) + cc;  // 32-column chunk
        uint32_t v[32];
        tmem_ld32(t_row + c * 32, v);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const int col = c * 32 + g * 4;
                if (col < d_store)
                    *reinterpret_cast<float4 *>(dst + col) =
                        make_float4(__uint_as_float(v[4 * g]) * mul, __uint_as_float(v[4 * g + 1]) * mul,
                                    __uint_as_float(v[4 * g + 2]) * mul, __uint_as_float(v[4 * g + 3]) * mul);
            }
        }
    }
}

// dK and dV from the split pass's partials: for each real KV head, the sum of
// its kv_split virtual heads' fp32 partials in order g = 0, 1, ..., rounded
// to bf16.  Virtual head g of real KV head kvh is plane (b Hkv + kvh)
// kv_split + g; the dV partials follow all the dK partials.  One thread per
// 4 consecutive elements of a key row (d_store is 56, 64 or 128).
__global__ void dkdv_reduce_kernel(const float *part, __nv_bfloat16 *dk, __nv_bfloat16 *dv, int bh_real, int N,
                                   int d_store, int kv_split) {
    const int per_row = d_store / 4;
    const long long rows = (long long)bh_real * N;
    const long long n = rows * per_row;
    const size_t plane = (size_t)rows * kv_split * d_store;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / per_row;  // (b * Hkv + kvh) * N + key
        const int col = int(i % per_row) * 4;
        const long long bh = row / N, key = row % N;
        float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sv = sk;
        for (int g = 0; g < kv_split; ++g) {
            const size_t at = ((size_t)(bh * kv_split + g) * N + key) * d_store + col;
            const float4 a = *reinterpret_cast<const float4 *>(part + at);
            const float4 b = *reinterpret_cast<const float4 *>(part + plane + at);
            sk.x += a.x; sk.y += a.y; sk.z += a.z; sk.w += a.w;
            sv.x += b.x; sv.y += b.y; sv.z += b.z; sv.w += b.w;
        }
        const size_t o = (size_t)row * d_store + col;
        *reinterpret_cast<uint2 *>(dk + o) = make_uint2(pack_bf16x2(sk.x, sk.y), pack_bf16x2(sk.z, sk.w));
        *reinterpret_cast<uint2 *>(dv + o) = make_uint2(pack_bf16x2(sv.x, sv.y), pack_bf16x2(sv.z, sv.w));
    }
}

// ------------------------------------------------------------------- dK, dV

template <int D>
struct KvCfg {
    static constexpr int kChunks = D / 64;             // 128-byte column chunks of a row
    static constexpr int kChunkBytes = kRows * 128;    // one chunk of 128 rows
    static constexpr int kTileBytes = kRows * D * 2;   // one 128 x D bf16 tile
    static constexpr int kStages = (D == 128) ? 2 : 5; // Q/dO ring (d <= 64: 5 measured 1% above 3)
    static constexpr int kStageBytes = 2 * kTileBytes + 1024;  // Q, dO, -lse2, Delta
    // barriers: kv_full kv_empty st_full[S] st_empty[S] s_full[2] p_full[2]
    //           acc_full acc_empty uq_full[2] uq_empty[2] drain
    static constexpr int kBarKVFull = 0, kBarKVEmpty = 1, kBarStFull = 2, kBarStEmpty = 2 + kStages,
                         kBarSFull = 2 + 2 * kStages, kBarPFull = 4 + 2 * kStages,
                         kBarAccFull = 6 + 2 * kStages, kBarAccEmpty = 7 + 2 * kStages,
                         kBarUQFull = 8 + 2 * kStages, kBarUQEmpty = 10 + 2 * kStages,
                         kBarDrain = 12 + 2 * kStages, kNumBars = 13 + 2 * kStages;
    static constexpr int kDataBytes = 2 * kTileBytes + kStages * kStageBytes;
    static constexpr int kSmemBytes = kDataBytes + kNumBars * 8 + 32 + 1024;
    // TMEM: half-buffer h (query rows [64 h, 64 h + 64) of a block) holds S^T
    // at [128 h, +64) and dP^T at [128 h + 64, +64); dV and dK follow.
    static constexpr int kColHalf = 128, kColDV = 256, kColDK = 256 + D;
};

// Query blocks per query head that key block j meets (causal: i >= j).
__device__ __forceinline__ int kv_first_i(const Params &p, int j) { return p.causal ? j : 0; }

// kPart: the split form, writing fp32 partials of virtual KV heads (see the
// file's header); a separate instantiation, so the plain one is unchanged.
template <int D, bool kPart>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const Params p) {
    using C = KvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sK = smem;
    uint8_t *sV = smem + C::kTileBytes;
    uint8_t *sStage = smem + 2 * C::kTileBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kDataBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *unit_q = reinterpret_cast<volatile int *>(tmem_slot + 2);  // 2 entries

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };
    auto stage_q = [&](int s) { return sStage + s * C::kStageBytes; };
    auto stage_do = [&](int s) { return sStage + s * C::kStageBytes + C::kTileBytes; };
    auto stage_l = [&](int s) {
        return reinterpret_cast<const float *>(sStage + s * C::kStageBytes + 2 * C::kTileBytes);
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(C::kBarKVFull), 1);
        mbar_init(bar(C::kBarKVEmpty), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(C::kBarStFull + s), 1);
            mbar_init(bar(C::kBarStEmpty + s), 1 + kEwWarps);  // MMA commit + elementwise warps
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar(C::kBarSFull + h), 1);
            mbar_init(bar(C::kBarPFull + h), kEwWarps / 2);  // the half's warpgroup
        }
        mbar_init(bar(C::kBarAccFull), 1);
        mbar_init(bar(C::kBarAccEmpty), kEwWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::kBarUQFull + i), 1);
            mbar_init(bar(C::kBarUQEmpty + i), 1 + kEwWarps);  // MMA warp + elementwise warps
        }
        mbar_init(bar(C::kBarDrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmDO);
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
    int *status = &g_bwd_status;

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BwdRegs<D>::kCtrl));
      if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            long long fills = 0;  // ring fills issued
            int kv_loads = 0;
            bool ok = true;
            for (long long qi = 0; ok; ++qi) {
                const long long u = fetch_unit(p, 0, qi);
                const int qs = int(qi & 1);
                if (qi >= 2 && !mbar_wait_bounded(bar(C::kBarUQEmpty + qs), uint32_t(((qi >> 1) - 1) & 1),
                                                  p.wait_ns, abort_flag, status)) {
                    ok = false;
                    break;
                }
                unit_q[qs] = int(u);
                mbar_arrive(bar(C::kBarUQFull + qs));
                if (u < 0) break;
                const KvUnit w = kv_unit(p, u);
                if (kv_loads > 0 && !mbar_wait_bounded(bar(C::kBarKVEmpty), uint32_t((kv_loads - 1) & 1),
                                                       p.wait_ns, abort_flag, status)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(C::kBarKVFull), 2 * C::kTileBytes);
                const int kv_plane = kPart ? w.b * p.hkv_real + w.g / p.kv_split : w.b * p.Hkv + w.g;
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(smem_u32(sK + c * C::kChunkBytes), &tmK, bar(C::kBarKVFull), c * 64,
                                w.j * kRows, kv_plane);
                    tma_load_3d(smem_u32(sV + c * C::kChunkBytes), &tmV, bar(C::kBarKVFull), c * 64,
                                w.j * kRows, kv_plane);
                }
                ++kv_loads;
                const int i0 = kv_first_i(p, w.j);
                const int ni = p.nblk - i0;
                const int iters = p.G * ni;
                for (int t = 0; t < iters; ++t) {
                    const int h = w.g * p.G + t / ni;
                    const int i = i0 + t % ni;
                    const int slot = int(fills % C::kStages);
                    const long long round = fills / C::kStages;
                    if (round > 0 && !mbar_wait_bounded(bar(C::kBarStEmpty + slot), uint32_t((round - 1) & 1),
                                                        p.wait_ns, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar(C::kBarStFull + slot);
                    mbar_arrive_expect_tx(fb, 2 * C::kTileBytes + 1024);
                    const int bh = w.b * p.Hq + h;
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_3d(smem_u32(stage_q(slot) + c * C::kChunkBytes), &tmQ, fb, c * 64, i * kRows,
                                    bh);
                        tma_load_3d(smem_u32(stage_do(slot) + c * C::kChunkBytes), &tmDO, fb, c * 64,
                                    i * kRows, bh);
                    }
                    const size_t row0 = (size_t)bh * p.npad + (size_t)i * kRows;
                    bulk_load(smem_u32(stage_l(slot)), p.nlse2 + row0, kRows * 4, fb);
                    bulk_load(smem_u32(stage_l(slot) + kRows), p.delta + row0, kRows * 4, fb);
                    ++fills;
                }
            }
            if (!ok) {
                // Drain: wait (bounded, independent of the caller's limit) for the
                // last fill of every slot and the last K/V load, so no copy is
                // still writing shared memory when the CTA exits.
                const unsigned long long drain_ns = 1000000000ull;
                volatile int no_abort = 0;
                for (int s = 0; s < C::kStages; ++s) {
                    if (fills <= s) continue;
                    const long long last = fills - 1 - ((fills - 1 - s) % C::kStages);
                    if (!mbar_wait_bounded(bar(C::kBarStFull + s), uint32_t((last / C::kStages) & 1), drain_ns,
                                           &no_abort, status))
                        atomicOr(status, kStatusDrainTimeout);
                }
                if (kv_loads > 0 && !mbar_wait_bounded(bar(C::kBarKVFull), uint32_t((kv_loads - 1) & 1),
                                                       drain_ns, &no_abort, status))
                    atomicOr(status, kStatusDrainTimeout);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // Per 128-row query block (one ring stage) and half h (its query rows
        // [64 h, 64 h + 64)): S^T_h = K Q_h^T and dP^T_h = V dO_h^T into
        // half-buffer h, then, once warpgroup h has written P^T_h and dS^T_h,
        // dV += P^T_h dO_h and dK += dS^T_h Q_h.  Issue order per stage t:
        //   dVdK(0, t), S(0, t+1), dVdK(1, t), S(1, t+1)
        // so the tensor core works on one half while warpgroup h computes the
        // other, and the commit announcing S(h, t+1) also covers dVdK(h, t).
        // The whole warp runs the issue loop (its state is warp-uniform); each
        // MMA, commit and arrival goes out from one elected lane.
        {
            constexpr uint32_t kIdescS = idesc_bf16_f32(kRows, 64, 0);  // N = 64 query rows
            constexpr uint32_t kIdescAcc = idesc_bf16_f32(kRows, D, 1);  // B read MN-major
            const uint64_t dK0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t dV0 = smem_desc_sw128(smem_u32(sV), 16, 1024);
            long long fills = 0;
            int kv_used = 0, units_done = 0;
            int p_waits[2] = {0, 0};
            bool ok = true;
            auto wait_stage = [&](long long f) {
                return mbar_wait_warp(bar(C::kBarStFull + int(f % C::kStages)), uint32_t((f / C::kStages) & 1),
                                         p.wait_ns, abort_flag, status);
            };
            // S^T_h and dP^T_h of the stage at ring position f.
            auto issue_s = [&](int h, long long f) {
                const int slot = int(f % C::kStages);
                const uint32_t hrow = uint32_t(h * 64 * 128);  // byte offset of row 64 h in a chunk
                const uint64_t dQk = smem_desc_sw128(smem_u32(stage_q(slot)) + hrow, 16, 1024);
                const uint64_t dOk = smem_desc_sw128(smem_u32(stage_do(slot)) + hrow, 16, 1024);
                const uint32_t tS = tmem_base + h * C::kColHalf;
                ss_product<D, C::kChunkBytes>(tS, dK0, dQk, kIdescS);
                ss_product<D, C::kChunkBytes>(tS + 64, dV0, dOk, kIdescS);
                tc_commit_elect(bar(C::kBarSFull + h));
            };
            for (long long qi = 0; ok; ++qi) {
                const int qs = int(qi & 1);
                ok = mbar_wait_warp(bar(C::kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns, abort_flag,
                                       status);
                if (!ok) break;
                const long long u = __shfl_sync(0xffffffffu, int(unit_q[qs]), 0);
                mbar_arrive_elect(bar(C::kBarUQEmpty + qs));
                if (u < 0) break;
                const KvUnit w = kv_unit(p, u);
                const int iters = p.G * (p.nblk - kv_first_i(p, w.j));
                ok = mbar_wait_warp(bar(C::kBarKVFull), uint32_t(kv_used & 1), p.wait_ns, abort_flag, status);
                if (ok) ok = wait_stage(fills);
                if (!ok) break;
                ++kv_used;
                tc_fence_after();
                issue_s(0, fills);
                issue_s(1, fills);
                for (int t = 0; ok && t < iters; ++t) {
                    const int slot = int(fills % C::kStages);
                    const bool has_next = t + 1 < iters;
                    for (int h = 0; h < 2; ++h) {
                        ok = mbar_wait_warp(bar(C::kBarPFull + h), uint32_t(p_waits[h] & 1), p.wait_ns,
                                               abort_flag, status);
                        if (!ok) break;
                        ++p_waits[h];
                        if (t == 0 && h == 0 && units_done > 0) {
                            ok = mbar_wait_warp(bar(C::kBarAccEmpty), uint32_t((units_done - 1) & 1), p.wait_ns,
                                                   abort_flag, status);
                            if (!ok) break;
                        }
                        tc_fence_after();
                        const uint32_t hrow = uint32_t(h * 64 * 128);
                        const uint64_t dOmn = smem_desc_sw128(smem_u32(stage_do(slot)) + hrow, C::kChunkBytes, 1024);
                        const uint64_t dQmn = smem_desc_sw128(smem_u32(stage_q(slot)) + hrow, C::kChunkBytes, 1024);
                        const uint32_t tH = tmem_base + h * C::kColHalf;
                        const bool first = (t == 0 && h == 0);
                        ts_product<4>(tmem_base + C::kColDV, tH, dOmn, kIdescAcc, !first);  // K = 64 query rows
                        ts_product<4>(tmem_base + C::kColDK, tH + 64, dQmn, kIdescAcc, !first);
                        if (h == 1) tc_commit_elect(bar(C::kBarStEmpty + slot));
                        if (has_next) {
                            if (h == 0) {
                                ok = wait_stage(fills + 1);
                                if (!ok) break;
                                tc_fence_after();
                            }
                            issue_s(h, fills + 1);
                        }
                    }
                    if (!ok) break;
                    ++fills;
                    if (!has_next) {
                        tc_commit_elect(bar(C::kBarAccFull));
                        tc_commit_elect(bar(C::kBarKVEmpty));
                        ++units_done;
                    }
                }
            }
            tc_commit_elect(bar(C::kBarDrain));
            volatile int no_abort = 0;
            if (!mbar_wait_warp(bar(C::kBarDrain), 0, 1000000000ull, &no_abort, status) && lane == 0)
                atomicOr(status, kStatusDrainTimeout);
        }
        __syncwarp();
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(BwdRegs<D>::kEw));
        // ---------------------------------------------------------------- elementwise / epilogue
        // Warpgroup h = (w - 4) / 4 owns half-buffer h: query rows [64 h, +64)
        // of every block; warp w reads TMEM lanes [32 (w % 4), +32), one key
        // row per thread.
        const int quarter = warp & 3;
        const int half = (warp - 4) >> 2;
        const int r = quarter * 32 + lane;  // key row inside the block
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        const uint32_t tH = tmem_base + lane_off + half * C::kColHalf;  // S^T_h; dP^T_h at +64
        const float sl2 = p.scale_log2;
        long long fills = 0;
        int s_waits = 0, acc_waits = 0;
        bool ok = true;
        for (long long qi = 0; ok; ++qi) {
            const int qs = int(qi & 1);
            ok = mbar_wait_warp(bar(C::kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns, abort_flag, status);
            if (!ok) break;
            const long long u = unit_q[qs];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarUQEmpty + qs));
            if (u < 0) break;
            const KvUnit w = kv_unit(p, u);
            const int i0 = kv_first_i(p, w.j);
            const int ni = p.nblk - i0;
            const int iters = p.G * ni;
            for (int t = 0; t < iters; ++t) {
                const int i = i0 + t % ni;
                const int slot = int(fills % C::kStages);
                ok = mbar_wait_warp(bar(C::kBarSFull + half), uint32_t(s_waits & 1), p.wait_ns, abort_flag, status);
                // The stage's lse / Delta rows: wait on the stage's own fill barrier
                // (already complete, since the MMA warp waited on it first).
                if (ok)
                    ok = mbar_wait_warp(bar(C::kBarStFull + slot), uint32_t((fills / C::kStages) & 1), p.wait_ns,
                                        abort_flag, status);
                if (!ok) break;
                ++s_waits;
                tc_fence_after();
                uint32_t sv[2][32], dv[2][32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    tmem_ld32(tH + c * 32, sv[c]);
                    tmem_ld32(tH + 64 + c * 32, dv[c]);
                }
                const float4 *l4 = reinterpret_cast<const float4 *>(stage_l(slot)) + half * 16;
                const float4 *d4 = reinterpret_cast<const float4 *>(stage_l(slot) + kRows) + half * 16;
                const bool diag = p.causal && i == w.j;  // query rows before this key are masked
                tmem_wait_ld();
                // P^T = 2^(S^T * scale * log2 e - lse2) and dS^T = P^T (dP^T - Delta),
                // written as bf16 over the half's columns.  The causal mask
                // (query rows before this key) applies only on the diagonal
                // block, so that block has its own copy of the loop.
                auto elementwise = [&](auto masked) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int q0 = half * 64 + c * 32;  // first query row of the chunk
                        uint32_t pk[16], dk[16];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float4 L = l4[c * 8 + e];   // -lse2
                            const float4 Dl = d4[c * 8 + e];  // Delta
                            const float nl[4] = {L.x, L.y, L.z, L.w};
                            const float dl[4] = {Dl.x, Dl.y, Dl.z, Dl.w};
                            float pr[4], ds[4];
#pragma unroll
                            for (int k = 0; k < 4; k += 2) {
                                float x0, x1;
                                ffma2(x0, x1, __uint_as_float(sv[c][4 * e + k]), __uint_as_float(sv[c][4 * e + k + 1]),
                                      sl2, sl2, nl[k], nl[k + 1]);
                                pr[k] = fast_exp2(x0);
                                pr[k + 1] = fast_exp2(x1);
                            }
                            if constexpr (decltype(masked)::value) {
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    if (q0 + 4 * e + k < r) pr[k] = 0.f;
                            }
#pragma unroll
                            for (int k = 0; k < 4; k += 2) {
                                float t0, t1;
                                fsub2(t0, t1, __uint_as_float(dv[c][4 * e + k]), __uint_as_float(dv[c][4 * e + k + 1]),
                                      dl[k], dl[k + 1]);
                                fmul2(ds[k], ds[k + 1], pr[k], pr[k + 1], t0, t1);
                            }
                            pk[2 * e] = pack_bf16x2(pr[0], pr[1]);
                            pk[2 * e + 1] = pack_bf16x2(pr[2], pr[3]);
                            dk[2 * e] = pack_bf16x2(ds[0], ds[1]);
                            dk[2 * e + 1] = pack_bf16x2(ds[2], ds[3]);
                        }
                        // bf16 pairs over the half's own fp32 columns, all read above
                        tmem_st16(tH + c * 16, pk);
                        tmem_st16(tH + 64 + c * 16, dk);
                    }
                };
                if (diag)
                    elementwise(std::true_type{});
                else
                    elementwise(std::false_type{});
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(C::kBarPFull + half));
                    mbar_arrive(bar(C::kBarStEmpty + slot));
                }
                ++fills;
            }
            if (!ok) break;
            // Epilogue: dV and scale * dK of this thread's key row -> bf16; the
            // two warpgroups store one half of the columns each.
            ok = mbar_wait_warp(bar(C::kBarAccFull), uint32_t(acc_waits & 1), p.wait_ns, abort_flag, status);
            if (!ok) break;
            ++acc_waits;
            tc_fence_after();
            const int key = w.j * kRows + r;
            const bool row_ok = key < p.N;
            const size_t off = ((size_t)(w.b * p.Hkv + w.g) * p.N + (row_ok ? key : 0)) * p.d_store;
            if constexpr (kPart) {
                const size_t plane = (size_t)p.B * p.Hkv * p.N * p.d_store;  // one of dK, dV
                store_half_row_f32<D>(tmem_base + lane_off + C::kColDK, half, p.part + off, row_ok, p.d_store,
                                      p.scale);
                store_half_row_f32<D>(tmem_base + lane_off + C::kColDV, half, p.part + plane + off, row_ok,
                                      p.d_store, 1.f);
            } else {
                store_half_row<D>(tmem_base + lane_off + C::kColDV, half, p.out1 + off, row_ok, p.d_store, 1.f);
                store_half_row<D>(tmem_base + lane_off + C::kColDK, half, p.out0 + off, row_ok, p.d_store,
                                  p.scale);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarAccEmpty));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
    finish_schedule(p, 0);
}

// ---------------------------------------------------------------------- dQ
//
// One unit is 256 query rows of one query head: two 128-row tiles that share
// every K/V block (as in the forward kernel) and alternate on the tensor core.
// TMEM per tile t: one 128-column fp32 buffer X(t) at 128 t that holds S,
// then dP (dS in bf16 is written over its first 64 columns), and the dQ(t)
// accumulator at 256 + D t.  Per K/V block j and tile t:
//   S(t, j) = Q_t K_j^T -> X(t);  warpgroup t keeps P = exp(S - lse) (fp32)
//   in registers; dP(t, j) = dO_t V_j^T -> X(t); warpgroup t writes
//   dS = P (dP - Delta) as bf16; dQ(t) += dS K_j.
// Issue order per block: dP(0, j), dP(1, j), dQ(0, j), S(0, j + 1), dQ(1, j),
// S(1, j + 1), so one tile's elementwise phase overlaps the other tile's MMAs.

template <int D>
struct QCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kChunkBytes = kRows * 128;
    static constexpr int kTileBytes = kRows * D * 2;
    // K/V ring of single tiles.  K tiles and V tiles have rings of their own:
    // V_j is free once both dP products of block j are done, early in the
    // block, while K_j is read by the block's last dQ product; sharing one
    // round-robin ring put V_j+1 into K_j's slot and the MMA warp waited for
    // it at the start of every block.
    static constexpr int kKSlots = (D == 128) ? 2 : 4;
    static constexpr int kVSlots = (D == 128) ? 1 : 2;
    static constexpr int kStages = kKSlots + kVSlots;
    // barriers: q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_full[2]
    //           dp_full[2] ds_full[2] acc_full[2] acc_empty[2] uq_full[2] uq_empty[2] drain
    static constexpr int kBarQFull = 0, kBarQEmpty = 2, kBarKVFull = 4, kBarKVEmpty = 4 + kStages,
                         kBarSFull = 4 + 2 * kStages, kBarPFull = 6 + 2 * kStages, kBarDPFull = 8 + 2 * kStages,
                         kBarDSFull = 10 + 2 * kStages, kBarAccFull = 12 + 2 * kStages,
                         kBarAccEmpty = 14 + 2 * kStages, kBarUQFull = 16 + 2 * kStages,
                         kBarUQEmpty = 18 + 2 * kStages, kBarDrain = 20 + 2 * kStages, kNumBars = 21 + 2 * kStages;
    // shared memory: Q_0, Q_1, dO_0, dO_1, then the ring
    static constexpr int kDataBytes = 4 * kTileBytes + kStages * kTileBytes;
    static constexpr int kSmemBytes = kDataBytes + kNumBars * 8 + 32 + 1024;
    static constexpr int kColDQ = 256;
};

// Fill f of the dQ pass's K/V stream: K_j at f = 2 j, V_j at f = 2 j + 1 (j
// counts blocks over the CTA's units); its ring slot and how many earlier
// fills used that slot (the mbarrier phase count).
template <int D>
__device__ __forceinline__ int dq_slot(long long f) {
    using C = QCfg<D>;
    const long long j = f >> 1;
    return (f & 1) ? C::kKSlots + int(j % C::kVSlots) : int(j % C::kKSlots);
}
template <int D>
__device__ __forceinline__ long long dq_use(long long f) {
    using C = QCfg<D>;
    const long long j = f >> 1;
    return (f & 1) ? j / C::kVSlots : j / C::kKSlots;
}

// dq unit -> (b, h, m): m is a 256-row block; tile t covers rows m 256 + 128 t.
struct QUnit2 {
    int b, h, m;
    int row0[2];
    int nkv[2];  // 128-key blocks tile t visits (0: tile past N)
    int nmax;
};
__device__ __forceinline__ QUnit2 q_unit2(const Params &p, long long u) {
    QUnit2 w;
    const int nq = (p.N + 2 * kRows - 1) / (2 * kRows);  // 256-row blocks per head
    int r;
    if (p.order == kBlockFirst) {
        w.h = int(u % p.Hq);
        const long long bm = u / p.Hq;
        r = int(bm % nq);
        w.b = int(bm / nq);
    } else if (p.order == kHeadFirst && p.causal && p.G > 1) {
        // as the forward's head-first order: a causal GQA ACC's units run
        // longest first across its query heads (block rank, then head)
        const long long upa = (long long)p.G * nq;
        const long long a = u / upa;  // ACC = b * Hkv + KV head
        const int wi = int(u % upa);
        r = wi / p.G;
        w.h = int(a % p.Hkv) * p.G + wi % p.G;
        w.b = int(a / p.Hkv);
    } else {
        r = int(u % nq);
        const long long bh = u / nq;
        w.h = int(bh % p.Hq);
        w.b = int(bh / p.Hq);
    }
    w.m = p.causal ? (nq - 1 - r) : r;
    w.nmax = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int r0 = w.m * 2 * kRows + t * kRows;
        w.row0[t] = r0;
        int n = 0;
        if (r0 < p.N) n = p.causal ? min(p.nblk, r0 / kRows + 1) : p.nblk;
        w.nkv[t] = n;
        w.nmax = max(w.nmax, n);
    }
    return w;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const Params p) {
    using C = QCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sQ = smem;                         // two tiles
    uint8_t *sDO = smem + 2 * C::kTileBytes;    // two tiles
    uint8_t *sKV = smem + 4 * C::kTileBytes;    // ring
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kDataBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *unit_q = reinterpret_cast<volatile int *>(tmem_slot + 2);  // 2 entries

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(C::kBarQFull + t), 1);
            mbar_init(bar(C::kBarQEmpty + t), 1);
            mbar_init(bar(C::kBarSFull + t), 1);
            mbar_init(bar(C::kBarPFull + t), 4);
            mbar_init(bar(C::kBarDPFull + t), 1);
            mbar_init(bar(C::kBarDSFull + t), 4);
            mbar_init(bar(C::kBarAccFull + t), 1);
            mbar_init(bar(C::kBarAccEmpty + t), 4);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(C::kBarKVFull + s), 1);
            mbar_init(bar(C::kBarKVEmpty + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::kBarUQFull + i), 1);
            mbar_init(bar(C::kBarUQEmpty + i), 1 + kEwWarps);
        }
        mbar_init(bar(C::kBarDrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmDO);
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
    int *status = &g_bwd_status;

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BwdRegs<D, true>::kCtrl));
      if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            long long fills = 0;
            int q_loads[2] = {0, 0};
            bool ok = true;
            long long last_use[C::kStages];  // use count of each slot's latest fill (-1: none)
            for (int s = 0; s < C::kStages; ++s) last_use[s] = -1;
            auto emit = [&](const CUtensorMap *map, int blk, int plane) {
                const int slot = dq_slot<D>(fills);
                const long long round = dq_use<D>(fills);
                if (round > 0 && !mbar_wait_bounded(bar(C::kBarKVEmpty + slot), uint32_t((round - 1) & 1),
                                                    p.wait_ns, abort_flag, status))
                    return false;
                const uint32_t fb = bar(C::kBarKVFull + slot);
                mbar_arrive_expect_tx(fb, C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(smem_u32(sKV + slot * C::kTileBytes + c * C::kChunkBytes), map, fb, c * 64,
                                blk * kRows, plane);
                last_use[slot] = round;
                ++fills;
                return true;
            };
            for (long long qi = 0; ok; ++qi) {
                const long long u = fetch_unit(p, 1, qi);
                const int qs = int(qi & 1);
                if (qi >= 2 && !mbar_wait_bounded(bar(C::kBarUQEmpty + qs), uint32_t(((qi >> 1) - 1) & 1),
                                                  p.wait_ns, abort_flag, status)) {
                    ok = false;
                    break;
                }
                unit_q[qs] = int(u);
                mbar_arrive(bar(C::kBarUQFull + qs));
                if (u < 0) break;
                const QUnit2 w = q_unit2(p, u);
                const int bh = w.b * p.Hq + w.h;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (w.nkv[t] == 0) continue;
                    if (q_loads[t] > 0)
                        ok = mbar_wait_bounded(bar(C::kBarQEmpty + t), uint32_t((q_loads[t] - 1) & 1), p.wait_ns,
                                               abort_flag, status);
                    if (!ok) break;
                    const uint32_t qb = bar(C::kBarQFull + t);
                    mbar_arrive_expect_tx(qb, 2 * C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_3d(smem_u32(sQ + t * C::kTileBytes + c * C::kChunkBytes), &tmQ, qb, c * 64,
                                    w.row0[t], bh);
                        tma_load_3d(smem_u32(sDO + t * C::kTileBytes + c * C::kChunkBytes), &tmDO, qb, c * 64,
                                    w.row0[t], bh);
                    }
                    ++q_loads[t];
                }
                const int plane = w.b * p.Hkv + w.h / p.G;
                for (int j = 0; ok && j < w.nmax; ++j) {
                    ok = emit(&tmK, j, plane);
                    if (ok) ok = emit(&tmV, j, plane);
                }
            }
            if (!ok) {
                const unsigned long long drain_ns = 1000000000ull;
                volatile int no_abort = 0;
                for (int s = 0; s < C::kStages; ++s) {
                    if (last_use[s] < 0) continue;
                    if (!mbar_wait_bounded(bar(C::kBarKVFull + s), uint32_t(last_use[s] & 1), drain_ns, &no_abort,
                                           status))
                        atomicOr(status, kStatusDrainTimeout);
                }
                for (int t = 0; t < 2; ++t)
                    if (q_loads[t] > 0 && !mbar_wait_bounded(bar(C::kBarQFull + t), uint32_t((q_loads[t] - 1) & 1),
                                                             drain_ns, &no_abort, status))
                        atomicOr(status, kStatusDrainTimeout);
            }
        }
      } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // The whole warp runs the issue loop (its state is warp-uniform); each
        // MMA, commit and arrival goes out from one elected lane.
        {
            constexpr uint32_t kIdescS = idesc_bf16_f32(kRows, kRows, 0);
            constexpr uint32_t kIdescAcc = idesc_bf16_f32(kRows, D, 1);
            long long fills = 0;
            int q_used[2] = {0, 0}, p_waits[2] = {0, 0}, ds_waits[2] = {0, 0}, units_done[2] = {0, 0};
            bool ok = true;
            auto slot_of = [&](long long f) { return dq_slot<D>(f); };
            auto wait_fill = [&](long long f) {
                return mbar_wait_warp(bar(C::kBarKVFull + slot_of(f)), uint32_t(dq_use<D>(f) & 1), p.wait_ns,
                                         abort_flag, status);
            };
            auto kmaj = [&](long long f) { return smem_desc_sw128(smem_u32(sKV + slot_of(f) * C::kTileBytes), 16, 1024); };
            auto issue_s = [&](int t, long long fK) {  // S(t) = Q_t K^T -> X(t)
                ss_product<D, C::kChunkBytes>(tmem_base + kRows * t,
                                              smem_desc_sw128(smem_u32(sQ + t * C::kTileBytes), 16, 1024), kmaj(fK),
                                              kIdescS);
                tc_commit_elect(bar(C::kBarSFull + t));
            };
            for (long long qi = 0; ok; ++qi) {
                const int qs = int(qi & 1);
                ok = mbar_wait_warp(bar(C::kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns, abort_flag,
                                       status);
                if (!ok) break;
                const long long u = __shfl_sync(0xffffffffu, int(unit_q[qs]), 0);
                mbar_arrive_elect(bar(C::kBarUQEmpty + qs));
                if (u < 0) break;
                const QUnit2 w = q_unit2(p, u);
                const long long f0 = fills;  // K_j at f0 + 2 j, V_j at f0 + 2 j + 1
                ok = wait_fill(f0);
                for (int t = 0; ok && t < 2; ++t) {
                    if (w.nkv[t] == 0) continue;
                    ok = mbar_wait_warp(bar(C::kBarQFull + t), uint32_t(q_used[t] & 1), p.wait_ns, abort_flag,
                                           status);
                    if (!ok) break;
                    ++q_used[t];
                    tc_fence_after();
                    issue_s(t, f0);
                }
                for (int j = 0; ok && j < w.nmax; ++j) {
                    const long long fK = f0 + 2 * j, fV = fK + 1;
                    // dP(t, j) once warpgroup t holds P (X(t) is free again)
                    ok = wait_fill(fV);
                    for (int t = 0; ok && t < 2; ++t) {
                        if (j >= w.nkv[t]) continue;
                        ok = mbar_wait_warp(bar(C::kBarPFull + t), uint32_t(p_waits[t] & 1), p.wait_ns, abort_flag,
                                               status);
                        if (!ok) break;
                        ++p_waits[t];
                        tc_fence_after();
                        ss_product<D, C::kChunkBytes>(tmem_base + kRows * t,
                                                      smem_desc_sw128(smem_u32(sDO + t * C::kTileBytes), 16, 1024),
                                                      kmaj(fV), kIdescS);
                        tc_commit_elect(bar(C::kBarDPFull + t));
                    }
                    if (!ok) break;
                    tc_commit_elect(bar(C::kBarKVEmpty + slot_of(fV)));  // V_j consumed
                    // dQ(t, j) once warpgroup t wrote dS, then S(t, j + 1)
                    bool k_next = false;
                    for (int t = 0; ok && t < 2; ++t) {
                        if (j >= w.nkv[t]) continue;
                        ok = mbar_wait_warp(bar(C::kBarDSFull + t), uint32_t(ds_waits[t] & 1), p.wait_ns,
                                               abort_flag, status);
                        if (!ok) break;
                        ++ds_waits[t];
                        if (j == 0 && units_done[t] > 0) {
                            ok = mbar_wait_warp(bar(C::kBarAccEmpty + t), uint32_t((units_done[t] - 1) & 1),
                                                   p.wait_ns, abort_flag, status);
                            if (!ok) break;
                        }
                        tc_fence_after();
                        const uint64_t kmn = smem_desc_sw128(smem_u32(sKV + slot_of(fK) * C::kTileBytes), C::kChunkBytes,
                                                             1024);
                        ts_product<8>(tmem_base + C::kColDQ + D * t, tmem_base + kRows * t, kmn, kIdescAcc, j > 0);
                        if (j + 1 < w.nkv[t]) {
                            if (!k_next) {
                                ok = wait_fill(fK + 2);
                                if (!ok) break;
                                k_next = true;
                                tc_fence_after();
                            }
                            issue_s(t, fK + 2);
                        } else {
                            tc_commit_elect(bar(C::kBarAccFull + t));  // dQ(t) final for this unit
                            tc_commit_elect(bar(C::kBarQEmpty + t));   // Q_t, dO_t reusable
                            ++units_done[t];
                        }
                    }
                    if (!ok) break;
                    tc_commit_elect(bar(C::kBarKVEmpty + slot_of(fK)));  // K_j consumed
                }
                fills = f0 + 2 * (long long)w.nmax;
            }
            tc_commit_elect(bar(C::kBarDrain));
            volatile int no_abort = 0;
            if (!mbar_wait_warp(bar(C::kBarDrain), 0, 1000000000ull, &no_abort, status) && lane == 0)
                atomicOr(status, kStatusDrainTimeout);
        }
        __syncwarp();
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(BwdRegs<D, true>::kEw));
        // ---------------------------------------------------------------- elementwise / epilogue
        // Warpgroup t = (w - 4) / 4 owns tile t; warp w reads TMEM lanes
        // [32 (w % 4), +32), one query row per thread.
        const int t = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        const uint32_t tX = tmem_base + lane_off + kRows * t;
        const float sl2 = p.scale_log2;
        int s_waits = 0, dp_waits = 0, acc_waits = 0;
        bool ok = true;
        for (long long qi = 0; ok; ++qi) {
            const int qs = int(qi & 1);
            ok = mbar_wait_warp(bar(C::kBarUQFull + qs), uint32_t((qi >> 1) & 1), p.wait_ns, abort_flag, status);
            if (!ok) break;
            const long long u = unit_q[qs];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarUQEmpty + qs));
            if (u < 0) break;
            const QUnit2 w = q_unit2(p, u);
            const int nkv = w.nkv[t];
            if (nkv == 0) continue;
            const int row = w.row0[t] + r;
            const size_t prow = (size_t)(w.b * p.Hq + w.h) * p.npad + row;  // row < npad always
            const float neg_l = p.nlse2[prow];                               // -inf past N
            const float del = p.delta[prow];
            for (int j = 0; j < nkv; ++j) {
                // P = exp(S - lse), kept in registers
                ok = mbar_wait_warp(bar(C::kBarSFull + t), uint32_t(s_waits & 1), p.wait_ns, abort_flag, status);
                if (!ok) break;
                ++s_waits;
                tc_fence_after();
                float pr[kRows];
                {
                    uint32_t sv[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(tX + c * 32, sv[c]);
                    tmem_wait_ld();
                    const int kv0 = j * kRows;
                    int lim = kRows;  // block columns c >= lim are masked (past N or after the row)
                    if (kv0 + kRows > p.N) lim = p.N - kv0;
                    if (p.causal && j == w.row0[t] / kRows) lim = min(lim, r + 1);
                    // Only the last block and the diagonal one mask columns; the
                    // others take the loop without the per-column selects.
                    auto exps = [&](auto masked) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                float x0, x1;
                                ffma2(x0, x1, __uint_as_float(sv[c][2 * e]), __uint_as_float(sv[c][2 * e + 1]), sl2,
                                      sl2, neg_l, neg_l);
                                const int k = c * 32 + 2 * e;
                                if constexpr (decltype(masked)::value) {
                                    pr[k] = k < lim ? fast_exp2(x0) : 0.f;
                                    pr[k + 1] = k + 1 < lim ? fast_exp2(x1) : 0.f;
                                } else {
                                    pr[k] = fast_exp2(x0);
                                    pr[k + 1] = fast_exp2(x1);
                                }
                            }
                    };
                    if (__any_sync(0xffffffffu, lim < kRows))
                        exps(std::true_type{});
                    else
                        exps(std::false_type{});
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarPFull + t));
                // dS = P (dP - Delta) -> bf16 over the first 64 columns of X(t)
                ok = mbar_wait_warp(bar(C::kBarDPFull + t), uint32_t(dp_waits & 1), p.wait_ns, abort_flag, status);
                if (!ok) break;
                ++dp_waits;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t dv[32];
                    tmem_ld32(tX + c * 32, dv);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float t0, t1, d0, d1;
                        fsub2(t0, t1, __uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1]), del, del);
                        fmul2(d0, d1, pr[c * 32 + 2 * e], pr[c * 32 + 2 * e + 1], t0, t1);
                        pk[e] = pack_bf16x2(d0, d1);
                    }
                    tmem_st16(tX + c * 16, pk);  // over columns already read
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarDSFull + t));
            }
            if (!ok) break;
            ok = mbar_wait_warp(bar(C::kBarAccFull + t), uint32_t(acc_waits & 1), p.wait_ns, abort_flag, status);
            if (!ok) break;
            ++acc_waits;
            tc_fence_after();
            const bool row_ok = row < p.N;
            const size_t off = ((size_t)(w.b * p.Hq + w.h) * p.N + (row_ok ? row : 0)) * p.d_store;
            store_half_row<D>(tmem_base + lane_off + C::kColDQ + D * t, 0, p.out0 + off, row_ok, p.d_store, p.scale);
            store_half_row<D>(tmem_base + lane_off + C::kColDQ + D * t, 1, p.out0 + off, row_ok, p.d_store, p.scale);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarAccEmpty + t));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
    finish_schedule(p, 1);
}

template <int D>
int launch(const BwdLaunch &a, cudaStream_t stream) {
    using CA = KvCfg<D>;
    using CB = QCfg<D>;
    const int nblk = (a.N + kRows - 1) / kRows;
    const int npad = nblk * kRows;
    const long long rows = (long long)a.B * a.Hq * npad;
    float *nlse2 = a.workspace;
    float *delta = a.workspace + rows;

    // Pre-pass: Delta and lse * log2(e).
    {
        long long blocks = (rows + 31) / 32;  // 8 warps of 4 rows
        const long long cap = (long long)a.num_sms * 16;
        if (blocks > cap) blocks = cap;
        bwd_pre_kernel<<<unsigned(blocks), 256, 0, stream>>>(
            reinterpret_cast<const __nv_bfloat16 *>(a.o), reinterpret_cast<const __nv_bfloat16 *>(a.dout), a.lse,
            nlse2, delta, a.N, npad, a.d, rows);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return note_cuda_error(e, "bwd_pre_kernel launch");
    }

    CUtensorMap mq, mdo, mk, mv;
    const uint64_t dd = uint64_t(a.d);
    if (!encode_bf16_3d(&mq, a.q, dd, uint64_t(a.N), uint64_t(a.B) * a.Hq, 64, kRows) ||
        !encode_bf16_3d(&mdo, a.dout, dd, uint64_t(a.N), uint64_t(a.B) * a.Hq, 64, kRows) ||
        !encode_bf16_3d(&mk, a.k, dd, uint64_t(a.N), uint64_t(a.B) * a.Hkv, 64, kRows) ||
        !encode_bf16_3d(&mv, a.v, dd, uint64_t(a.N), uint64_t(a.B) * a.Hkv, 64, kRows))
        return note_cuda_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (backward)");

    static bool attr_set[kMaxDevices] = {};  // per instantiation and device
    const int dev = slot_for_device();
    if (dev < 0 || !attr_set[dev]) {
        // The setmaxnreg split assumes the launch register count; refuse a
        // build that differs (its setmaxnreg.inc could never complete).
        cudaFuncAttributes fa, fs, fb;
        cudaError_t e = cudaFuncGetAttributes(&fa, dkdv_kernel<D, false>);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fs, dkdv_kernel<D, true>);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fb, dq_kernel<D>);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncGetAttributes(backward kernels)");
        if (fa.numRegs != kLaunchRegs || fs.numRegs != kLaunchRegs || fb.numRegs != kLaunchRegs ||
            fa.maxThreadsPerBlock < kThreads || fs.maxThreadsPerBlock < kThreads || fb.maxThreadsPerBlock < kThreads)
            return note_cuda_error(cudaErrorInvalidConfiguration,
                                   "backward kernel register count differs from the setmaxnreg split");
        e = cudaFuncSetAttribute(dkdv_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 CA::kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(dkdv_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     CA::kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, CB::kSmemBytes);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncSetAttribute(backward kernels)");
        if (dev >= 0) attr_set[dev] = true;
    }
    Params p;
    p.nlse2 = nlse2;
    p.delta = delta;
    p.B = a.B;
    p.N = a.N;
    p.npad = npad;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.d_store = a.d;
    p.causal = a.causal ? 1 : 0;
    p.order = a.order;
    p.nblk = nblk;
    // Causal dK/dV units differ in length, and with few key blocks per KV
    // head a pair's longest block is a large part of an SM's share of the
    // work, so causal head-first runs windows of pairs longest first.  A
    // list-scheduling simulation of the persistent CTAs (152 SMs, unit time =
    // query blocks + 1) gives GQA 64/8 causal 8K 0.78 -> 0.94 of perfect
    // balance and 16K 0.93 -> 0.98; long sequences keep one pair per window.
    p.kv_split = 1;
    p.hkv_real = a.Hkv;
    p.part = nullptr;
    p.scale = a.scale;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.wait_ns = a.wait_ns;
    p.sched_slot = int(g_bwd_launch_seq.fetch_add(1) % kBwdSchedSlots);

    // dK, dV (split: over B * Hkv * kv_split virtual KV heads of G / kv_split
    // query heads each, then the partials' sum)
    const bool split = a.kv_split > 1 && a.part;
    if (split) {
        p.Hkv = a.Hkv * a.kv_split;
        p.G = (a.Hq / a.Hkv) / a.kv_split;
        p.kv_split = a.kv_split;
        p.part = a.part;
    }
    p.kv_window = dkdv_window(a.order, a.causal, a.B, p.Hkv, nblk, a.num_sms);
    p.out0 = reinterpret_cast<__nv_bfloat16 *>(a.dk);
    p.out1 = reinterpret_cast<__nv_bfloat16 *>(a.dv);
    p.total_units = (long long)a.B * p.Hkv * nblk;
    long long grid = p.total_units;
    if (a.order != kNaiveHeadFirst && grid > a.num_sms) grid = a.num_sms;
    if (grid > 0x7fffffffLL) return -2;
    if (split)
        dkdv_kernel<D, true><<<unsigned(grid), kThreads, CA::kSmemBytes, stream>>>(mq, mdo, mk, mv, p);
    else
        dkdv_kernel<D, false><<<unsigned(grid), kThreads, CA::kSmemBytes, stream>>>(mq, mdo, mk, mv, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return note_cuda_error(e, "dkdv_kernel launch");
    if (split) {
        const long long n = (long long)a.B * a.Hkv * a.N * (a.d / 4);
        long long blocks = (n + 255) / 256;
        const long long cap = (long long)a.num_sms * 16;
        if (blocks > cap) blocks = cap;
        dkdv_reduce_kernel<<<unsigned(blocks), 256, 0, stream>>>(a.part, reinterpret_cast<__nv_bfloat16 *>(a.dk),
                                                                reinterpret_cast<__nv_bfloat16 *>(a.dv),
                                                                a.B * a.Hkv, a.N, a.d, a.kv_split);
        e = cudaGetLastError();
        if (e != cudaSuccess) return note_cuda_error(e, "dkdv_reduce_kernel launch");
        p.Hkv = a.Hkv;  // the dQ pass uses the real heads
        p.G = a.Hq / a.Hkv;
    }

    // dQ.  Its units are the forward's (256 query rows), and causal GQA
    // head-first over an entry whose K/V all fit in L2 together takes the
    // block-first sequence, as the forward does (effective_order).
    const int nq = (a.N + 2 * kRows - 1) / (2 * kRows);
    p.order = effective_order(a.order, a.Hq, p.G, nq, p.causal);
    p.out0 = reinterpret_cast<__nv_bfloat16 *>(a.dq);
    p.out1 = nullptr;
    p.total_units = (long long)a.B * a.Hq * nq;  // 256-row units
    grid = p.total_units;
    if (a.order != kNaiveHeadFirst && grid > a.num_sms) grid = a.num_sms;
    if (grid > 0x7fffffffLL) return -2;
    dq_kernel<D><<<unsigned(grid), kThreads, CB::kSmemBytes, stream>>>(mq, mdo, mk, mv, p);
    e = cudaGetLastError();
    return e == cudaSuccess ? 0 : note_cuda_error(e, "dq_kernel launch");
}

}  // namespace bwd

// The dK/dV pass's query-head split for a problem: the smallest s dividing
// G = Hq / Hkv that gives at least kSplitUnits units (six waves on 152 SMs),
// else G; 1 when the problem already has that many units, and 1 when causal:
// there the head-first windows already balance the unequal units, and the
// split measured 2% slower (GQA 64/8 causal 8K), its partials and their sum
// costing more than the tail it shortens.
int bwd_kv_split(int B, int Hq, int Hkv, int N, int causal) {
    constexpr long long kSplitUnits = 6 * 152;
    if (causal) return 1;
    const int G = Hq / Hkv;
    const long long units = (long long)B * Hkv * ((N + bwd::kRows - 1) / bwd::kRows);
    if (units >= kSplitUnits) return 1;
    for (int s = 2; s < G; ++s)
        if (G % s == 0 && units * s >= kSplitUnits) return s;
    return G;
}

size_t bwd_part_bytes(int B, int Hkv, int N, int d, int kv_split) {
    if (kv_split <= 1) return 0;
    return 2 * (size_t)B * Hkv * kv_split * (size_t)N * d * sizeof(float);
}

int bwd_launch(const BwdLaunch &a, cudaStream_t stream) {
    if (a.d <= 64) return bwd::launch<64>(a, stream);
    return bwd::launch<128>(a, stream);
}

cudaError_t bwd_take_status(int *bits) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_bwd_status, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(int));
}

}  // namespace attn
