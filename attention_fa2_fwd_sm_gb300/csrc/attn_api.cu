// attn_api.cu -- the extern "C" boundary of libattn.so: argument validation
// (entirely on the host, before any CUDA call), dispatch to the kernels,
// device status reporting and the host-side view of the scheduler.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.h"
#include "dkdv_order.cuh"
#include "tile_order.cuh"

namespace attn {

namespace {

std::atomic<long long> g_wait_ns{10LL * 1000 * 1000 * 1000};  // 10 s

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int current_num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    static int cached[kMaxDevices] = {0};
    if (dev >= 0 && dev < kMaxDevices && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return -1;
    if (dev >= 0 && dev < kMaxDevices) cached[dev] = n;
    return n;
}

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxSplits = kDecodeMaxSplits;
constexpr int kDecodeMaxGroup = 16;

}  // namespace

namespace {
thread_local char g_last_error[256] = "";
}

int note_cuda_error(cudaError_t e, const char *where) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), int(e));
    return ATTN_ERR_CUDA;
}

bool encode_bf16_3d(CUtensorMap *map, const void *base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                    uint32_t box0, uint32_t box1) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {dim0, dim1, dim2};
    const cuuint64_t strides[2] = {dim0 * 2, dim0 * dim1 * 2};
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int fwd_run(const FwdLaunch &a, cudaStream_t stream) {
    // The library's choice: the one-CTA kernel (every head dimension).
    if (a.scheme == kSchemePair) return fwd_pair_launch(a, stream);
    return fwd_launch(a, stream);
}

}  // namespace attn

using namespace attn;

extern "C" {

int attn_version(void) { return 100; }

const char *attn_last_error(void) { return g_last_error; }

const char *attn_strerror(int code) {
    switch (code) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_ARG: return "invalid argument (null/misaligned pointer, bad size, Hq % Hkv, scale)";
        case ATTN_ERR_UNSUPPORTED: return "unsupported head dimension or group size";
        case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case ATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
        case ATTN_ERR_TIMEOUT: return "a bounded device wait ran out";
        default: return "unknown status code";
    }
}

long long attn_set_wait_timeout_ns(long long ns) {
    if (ns < 0) ns = 0;
    return g_wait_ns.exchange(ns);
}

long long attn_fwd_units(int B, int Hq, int N) {
    if (B <= 0 || Hq <= 0 || N <= 0) return 0;
    return (long long)B * Hq * unit_blocks(N);
}

int attn_tile_map(int tile_order, int B, int Hq, int Hkv, int N, int causal, long long unit, int *b, int *h,
                  int *m) {
    if (!b || !h || !m || B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || Hq % Hkv) return ATTN_ERR_ARG;
    if (tile_order < kHeadFirst || tile_order > kNaiveHeadFirst) return ATTN_ERR_ARG;
    const long long total = attn_fwd_units(B, Hq, N);
    if (unit < 0 || unit >= total) return ATTN_ERR_ARG;
    const Tile t = unit_to_tile(tile_order, unit, Hq, Hq / Hkv, unit_blocks(N), causal ? 1 : 0);
    *b = t.b;
    *h = t.h;
    *m = t.m;
    return ATTN_OK;
}

int attn_tile_map_die_split(int B, int Hq, int Hkv, int N, int causal, int die, long long k, int *b,
                            int *h, int *m) {
    if (!b || !h || !m || B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || Hq % Hkv) return ATTN_ERR_ARG;
    if (die < 0 || die >= kDies) return ATTN_ERR_ARG;
    const int nb = unit_blocks(N);
    const long long u = die_split_unit(die, k, B, Hkv, Hq / Hkv, nb);
    if (u < 0) return ATTN_ERR_ARG;
    const Tile t = unit_to_tile(kDieSplitHeadFirst, u, Hq, Hq / Hkv, nb, causal ? 1 : 0);  // head-first ids
    *b = t.b;
    *h = t.h;
    *m = t.m;
    return ATTN_OK;
}

int attn_bwd_tile_map(int tile_order, int B, int Hkv, int N, int causal, int num_sms, long long unit, int *b,
                      int *g, int *j) {
    if (!b || !g || !j || B <= 0 || Hkv <= 0 || N <= 0 || num_sms <= 0) return ATTN_ERR_ARG;
    if (tile_order < kHeadFirst || tile_order > kNaiveHeadFirst) return ATTN_ERR_ARG;
    if ((long long)B * Hkv >= (1LL << 31)) return ATTN_ERR_ARG;
    const int nblk = (N + kKeyBlock - 1) / kKeyBlock;
    if (unit < 0 || unit >= (long long)B * Hkv * nblk) return ATTN_ERR_ARG;
    const KvTile t = dkdv_unit_to_tile(tile_order, unit, B, Hkv, nblk,
                                       dkdv_window(tile_order, causal ? 1 : 0, B, Hkv, nblk, num_sms));
    *b = t.b;
    *g = t.g;
    *j = t.j;
    return ATTN_OK;
}

int attn_die_map(int *die_of_sm, int capacity, float *stats) {
    if (capacity < 0 || (capacity > 0 && !die_of_sm)) return ATTN_ERR_ARG;
    return die_map_query(die_of_sm, capacity, stats);
}

// tile_order of the forward entry points: an order in the low byte, at most
// one tile-scheme flag above it.
static int order_of(int tile_order) { return tile_order & 0xff; }
static int scheme_of(int tile_order) {
    const int f = tile_order & ~0xff;
    if (f == 0) return kSchemeAuto;
    if (f == ATTN_FWD_SINGLE_CTA) return kSchemeSingle;
    if (f == ATTN_FWD_CTA_PAIR) return kSchemePair;
    return -1;
}

static int validate_fwd_sizes(int B, int Hq, int Hkv, int N, int d, float scale, int tile_order) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0) return ATTN_ERR_ARG;
    if (Hq % Hkv) return ATTN_ERR_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_ARG;
    const int order = order_of(tile_order), scheme = scheme_of(tile_order);
    if (order < kHeadFirst || order > kDieSplitHeadFirst || scheme < 0) return ATTN_ERR_ARG;
    if (d != 56 && d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (scheme == kSchemePair && d != 128) return ATTN_ERR_UNSUPPORTED;
    // tensor-map limits: each dimension < 2^32, strides < 2^40 bytes
    if ((long long)B * Hq >= (1LL << 31) || (long long)N * d * 2 >= (1LL << 39)) return ATTN_ERR_ARG;
    // The persistent forward and backward kernels take work units (at most
    // B * Hq * ceil(N / 128) of them) from 32-bit counters.
    if ((long long)B * Hq * ((N + 127) / 128) >= (1LL << 31)) return ATTN_ERR_ARG;
    return ATTN_OK;
}

static int validate_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                        int Hq, int Hkv, int N, int d, float scale, int tile_order) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_ARG;
    return validate_fwd_sizes(B, Hq, Hkv, N, d, scale, tile_order);
}

static FwdLaunch fwd_problem(int B, int Hq, int Hkv, int N, int d, float scale, int causal, int tile_order,
                             int sms) {
    FwdLaunch a;
    a.q = a.k = a.v = nullptr;
    a.o = nullptr;
    a.lse = nullptr;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.order = order_of(tile_order);
    a.scheme = scheme_of(tile_order);
    a.wait_ns = (unsigned long long)g_wait_ns.load();
    a.num_sms = sms;
    return a;
}

int attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                int Hkv, int N, int d, float scale, int causal, int tile_order,
                attn_stream_t stream) {
    int rc = validate_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, tile_order);
    if (rc != ATTN_OK) return rc;
    const int sms = current_num_sms();
    if (sms <= 0) return note_cuda_error(cudaErrorNoDevice, "device query");
    FwdLaunch a = fwd_problem(B, Hq, Hkv, N, d, scale, causal, tile_order, sms);
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    return fwd_run(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int kv_heads_per_chunk) {
    if (validate_fwd_sizes(B, Hq, Hkv, N, d, 1.f, kHeadFirst) != ATTN_OK) return 0;
    if (kv_heads_per_chunk > Hkv) return 0;
    const int gc = kv_heads_per_chunk > 0 ? kv_heads_per_chunk : host_default_chunk(Hq, Hkv, N);
    return 2 * host_chunk_layout(Hq, Hkv, N, d, gc).slot_bytes;
}

int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv,
                  int N, int d, float scale, int causal, int tile_order, int kv_heads_per_chunk,
                  void *workspace, size_t workspace_bytes, attn_stream_t stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_ARG;
    int rc = validate_fwd_sizes(B, Hq, Hkv, N, d, scale, tile_order);
    if (rc != ATTN_OK) return rc;
    if (kv_heads_per_chunk > Hkv) return ATTN_ERR_ARG;
    const int gc = kv_heads_per_chunk > 0 ? kv_heads_per_chunk : host_default_chunk(Hq, Hkv, N);
    const size_t need = 2 * host_chunk_layout(Hq, Hkv, N, d, gc).slot_bytes;
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    const int sms = current_num_sms();
    if (sms <= 0) return note_cuda_error(cudaErrorNoDevice, "device query");
    FwdHostLaunch a;
    a.fwd = fwd_problem(B, Hq, Hkv, N, d, scale, causal, tile_order, sms);
    a.q_host = q;
    a.k_host = k;
    a.v_host = v;
    a.o_host = o;
    a.lse_host = lse;
    a.kv_heads_per_chunk = gc;
    a.workspace = workspace;
    return fwd_host_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_host_trace(int enable) { return fwd_host_trace(enable); }

long long attn_fwd_host_trace_read(float *ms, long long capacity) {
    if (capacity < 0 || (capacity > 0 && !ms)) return ATTN_ERR_ARG;
    const long long n = fwd_host_trace_read(ms, capacity);
    return n == -1 ? ATTN_ERR_ARG : n;
}

// Split-KV forward: the key range of each head in `splits` pieces of
// `chunk_keys` keys (a multiple of the 128-key block); kv_splits <= 0 picks
// the fewest pieces whose K and V of one KV head fit in 32 MiB.
constexpr int kMaxKvSplits = 64;
static bool splitkv_plan(int N, int d, int kv_splits, int *splits, int *chunk_keys) {
    if (kv_splits > kMaxKvSplits) return false;
    int s = kv_splits;
    if (s <= 0) {
        const long long budget_keys = (32LL << 20) / (4LL * d);  // K + V bf16 of one head per key: 4 d bytes
        s = int((N + budget_keys - 1) / budget_keys);
        if (s < 1) s = 1;
        if (s > kMaxKvSplits) s = kMaxKvSplits;
    }
    long long chunk = (N + s - 1) / s;
    chunk = (chunk + 127) / 128 * 128;
    *chunk_keys = int(chunk);
    *splits = int((N + chunk - 1) / chunk);
    return true;
}

static void splitkv_layout(int B, int Hq, int N, int d, int splits, size_t *o_bytes, size_t *lse_bytes) {
    const size_t rows = (size_t)B * Hq * N;
    *o_bytes = (rows * splits * d * sizeof(float) + 255) / 256 * 256;
    *lse_bytes = rows * splits * sizeof(float);
}

size_t attn_fwd_splitkv_workspace_bytes(int B, int Hq, int N, int d, int kv_splits) {
    if (B <= 0 || Hq <= 0 || N <= 0 || (d != 56 && d != 64 && d != 128)) return 0;
    int splits = 0, chunk = 0;
    if (!splitkv_plan(N, d, kv_splits, &splits, &chunk)) return 0;
    size_t a = 0, b = 0;
    splitkv_layout(B, Hq, N, d, splits, &a, &b);
    return a + b;
}

int attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv,
                     int N, int d, float scale, int causal, int kv_splits, void *workspace, size_t workspace_bytes,
                     attn_stream_t stream) {
    int rc = validate_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, kHeadFirst);
    if (rc != ATTN_OK) return rc;
    int splits = 0, chunk = 0;
    if (!splitkv_plan(N, d, kv_splits, &splits, &chunk)) return ATTN_ERR_ARG;
    if ((long long)B * Hq * unit_blocks(N) * splits >= (1LL << 31)) return ATTN_ERR_ARG;
    size_t o_bytes = 0, lse_bytes = 0;
    splitkv_layout(B, Hq, N, d, splits, &o_bytes, &lse_bytes);
    if (!workspace || !aligned16(workspace) || workspace_bytes < o_bytes + lse_bytes) return ATTN_ERR_WORKSPACE;
    const int sms = current_num_sms();
    if (sms <= 0) return note_cuda_error(cudaErrorNoDevice, "device query");
    FwdSplitLaunch a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.splits = splits;
    a.chunk_keys = chunk;
    a.part_o = static_cast<float *>(workspace);
    a.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + o_bytes);
    a.wait_ns = (unsigned long long)g_wait_ns.load();
    a.num_sms = sms;
    return fwd_split_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
             int Hkv, int N, int d, float scale, int causal, attn_stream_t stream) {
    return attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, ATTN_ORDER_HEAD_FIRST,
                       stream);
}

size_t attn_bwd_workspace_bytes(int B, int Hq, int N) {
    if (B <= 0 || Hq <= 0 || N <= 0) return 0;
    return (size_t)B * Hq * (size_t)((N + 127) / 128) * 128 * 2 * sizeof(float);
}

size_t attn_bwd_workspace_bytes_ex(int B, int Hq, int Hkv, int N, int d, int causal) {
    if (validate_fwd_sizes(B, Hq, Hkv, N, d, 1.f, kHeadFirst) != ATTN_OK) return 0;
    const size_t base = attn_bwd_workspace_bytes(B, Hq, N);
    const size_t part = bwd_part_bytes(B, Hkv, N, d, bwd_kv_split(B, Hq, Hkv, N, causal));
    return part ? (base + 255) / 256 * 256 + part : base;
}

int attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse,
             void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N, int d, float scale, int causal,
             int tile_order, void *workspace, size_t workspace_bytes, attn_stream_t stream) {
    int rc = validate_fwd(q, k, v, dq, nullptr, B, Hq, Hkv, N, d, scale, kHeadFirst);
    if (rc != ATTN_OK) return rc;
    if (!aligned16(o) || !aligned16(dout) || !aligned16(dk) || !aligned16(dv)) return ATTN_ERR_ARG;
    if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_ARG;
    if (tile_order < kHeadFirst || tile_order > kNaiveHeadFirst) return ATTN_ERR_ARG;
    const size_t need = (size_t)B * Hq * (size_t)((N + 127) / 128) * 128 * 2 * sizeof(float);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    // The dK/dV pass's query-head split, when the workspace also holds its partials.
    const int kv_split = bwd_kv_split(B, Hq, Hkv, N, causal);
    const size_t part_at = (need + 255) / 256 * 256;
    const size_t part_bytes = bwd_part_bytes(B, Hkv, N, d, kv_split);
    const int sms = current_num_sms();
    if (sms <= 0) return note_cuda_error(cudaErrorNoDevice, "device query");
    BwdLaunch a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.order = tile_order;
    a.workspace = static_cast<float *>(workspace);
    if (part_bytes > 0 && workspace_bytes >= part_at + part_bytes) {
        a.kv_split = kv_split;
        a.part = reinterpret_cast<float *>(static_cast<char *>(workspace) + part_at);
    }
    a.wait_ns = (unsigned long long)g_wait_ns.load();
    a.num_sms = sms;
    return bwd_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t attn_decode_workspace_bytes(int B, int Hq, int d, int num_splits) {
    if (B <= 0 || Hq <= 0 || d <= 0 || num_splits <= 1) return 0;
    const size_t parts = (size_t)B * Hq * num_splits;
    size_t o_bytes = parts * d * sizeof(float);
    o_bytes = (o_bytes + 255) / 256 * 256;
    return o_bytes + parts * sizeof(float);
}

// Split count: aim at about 5/3 CTAs per SM in all (the decode kernel keeps
// two CTAs resident per SM, and a grid just over one wave leaves a tail wave
// on a few SMs), never below 512 keys per split, at most kMaxSplits.  Chosen
// from a sweep of split counts over batch {1, 8, 32} x keys {8K, 32K, 128K}
// (H_Q = 64, H_KV = 8, d = 128), where it lands within a few percent of the
// best split count in every configuration.
static int splits_for(int B, int Hkv, int max_seqlen, int sms) {
    const long long ctas = (long long)B * Hkv;
    const long long target = (5LL * sms) / 3;
    long long s = (target + ctas / 2) / ctas;  // round to nearest
    const long long by_len = max_seqlen / 512;
    if (s > by_len) s = by_len;
    if (s > kMaxSplits) s = kMaxSplits;
    if (s < 1) s = 1;
    // Long caches: double the splits while each keeps at least 4096 keys and
    // the grid stays within four CTAs per SM (about 1.7 waves of two resident
    // CTAs per SM); the split sweep measured that 1-3% faster.
    while (2 * s <= kMaxSplits && max_seqlen / (2 * s) >= 4096 && ctas * 2 * s <= 4LL * sms) s *= 2;
    return int(s);
}

int attn_decode_num_splits(int B, int Hq, int Hkv, int max_seqlen) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || max_seqlen < 0 || Hq % Hkv) return ATTN_ERR_ARG;
    const int sms = current_num_sms();
    if (sms <= 0) return ATTN_ERR_CUDA;
    return splits_for(B, Hkv, max_seqlen, sms);
}

// Varlen decode: work-list capacity and the chunk rule (see attn.h).
constexpr int kVarlenMinChunk = 512;
static long long varlen_target(int sms) {
    const long long t = (5LL * sms) / 3;
    return t > 0 ? t : 1;
}
static long long varlen_max_items(int B, int Hkv, int sms) {
    const long long t = varlen_target(sms);
    return (t + Hkv - 1) / Hkv + B;
}
static void varlen_layout(int B, int Hq, int d, long long items, size_t *plan_bytes, size_t *o_bytes,
                          size_t *lse_bytes) {
    *plan_bytes = ((size_t)(2 + 2LL * B + 3 * items) * sizeof(int) + 255) / 256 * 256;
    *o_bytes = ((size_t)items * Hq * d * sizeof(float) + 255) / 256 * 256;
    *lse_bytes = (size_t)items * Hq * sizeof(float);
}

size_t attn_decode_varlen_workspace_bytes(int B, int Hq, int Hkv, int d) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv) return 0;
    const int sms = current_num_sms();
    if (sms <= 0) return 0;
    size_t a, b, c;
    varlen_layout(B, Hq, d, varlen_max_items(B, Hkv, sms), &a, &b, &c);
    return a + b + c;
}

int attn_decode_varlen(const void *q, const void *kcache, const void *vcache, const int *seqlens, void *o,
                       int B, int Hq, int Hkv, int d, float scale, int max_seqlen, void *workspace,
                       size_t workspace_bytes, attn_stream_t stream) {
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) || !seqlens ||
        (reinterpret_cast<uintptr_t>(seqlens) & 3u))
        return ATTN_ERR_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || max_seqlen <= 0 || Hq % Hkv) return ATTN_ERR_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (Hq / Hkv > kDecodeMaxGroup) return ATTN_ERR_UNSUPPORTED;
    if (B > (1 << 20) || Hkv > 65535 || (long long)max_seqlen * d * 2 >= (1LL << 39)) return ATTN_ERR_ARG;
    // the plan's T * Hkv stays below 2^62; the merge grid has B * Hq blocks
    if ((double)B * (double)max_seqlen * (double)Hkv >= 4.0e18 || (long long)B * Hq > 0x7fffffffLL)
        return ATTN_ERR_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u)) return ATTN_ERR_WORKSPACE;
    const int sms = current_num_sms();
    if (sms <= 0) return note_cuda_error(cudaErrorNoDevice, "device query");
    const long long items = varlen_max_items(B, Hkv, sms);
    if (items > 65535) return ATTN_ERR_ARG;  // grid.y limit of the decode launch
    size_t plan_bytes, o_bytes, lse_bytes;
    varlen_layout(B, Hq, d, items, &plan_bytes, &o_bytes, &lse_bytes);
    if (workspace_bytes < plan_bytes + o_bytes + lse_bytes) return ATTN_ERR_WORKSPACE;
    DecodeLaunch a;
    a.q = q;
    a.kcache = kcache;
    a.vcache = vcache;
    a.seqlens = seqlens;
    a.o = o;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.max_seqlen = max_seqlen;
    a.num_splits = 0;
    a.scale = scale;
    char *ws = static_cast<char *>(workspace);
    a.plan = reinterpret_cast<int *>(ws);
    a.ws_o = reinterpret_cast<float *>(ws + plan_bytes);
    a.ws_lse = reinterpret_cast<float *>(ws + plan_bytes + o_bytes);
    a.varlen_max_items = int(items);
    a.varlen_target = varlen_target(sms);
    a.varlen_min_chunk = kVarlenMinChunk;
    a.wait_ns = (unsigned long long)g_wait_ns.load();
    a.num_sms = sms;
    return decode_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

int attn_decode(const void *q, const void *kcache, const void *vcache, const int *seqlens, void *o,
                int B, int Hq, int Hkv, int d, float scale, int num_splits, int max_seqlen,
                void *workspace, size_t workspace_bytes, attn_stream_t stream) {
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) || !seqlens ||
        (reinterpret_cast<uintptr_t>(seqlens) & 3u))
        return ATTN_ERR_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || max_seqlen <= 0 || Hq % Hkv) return ATTN_ERR_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_ARG;
    if (num_splits > kMaxSplits) return ATTN_ERR_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (Hq / Hkv > kDecodeMaxGroup) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535 || Hkv > 65535 || (long long)max_seqlen * d * 2 >= (1LL << 39)) return ATTN_ERR_ARG;
    if (num_splits <= 0) {
        const int sms = current_num_sms();
        if (sms <= 0) return ATTN_ERR_CUDA;
        num_splits = splits_for(B, Hkv, max_seqlen, sms);
    }
    const size_t need = attn_decode_workspace_bytes(B, Hq, d, num_splits);
    if (need > 0 && (!workspace || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 15u)))
        return ATTN_ERR_WORKSPACE;
    DecodeLaunch a;
    a.q = q;
    a.kcache = kcache;
    a.vcache = vcache;
    a.seqlens = seqlens;
    a.o = o;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.max_seqlen = max_seqlen;
    a.num_splits = num_splits;
    a.scale = scale;
    const size_t parts = (size_t)B * Hq * num_splits;
    size_t o_bytes = (parts * d * sizeof(float) + 255) / 256 * 256;
    a.ws_o = need ? reinterpret_cast<float *>(workspace) : nullptr;
    a.ws_lse = need ? reinterpret_cast<float *>(reinterpret_cast<char *>(workspace) + o_bytes) : nullptr;
    a.wait_ns = (unsigned long long)g_wait_ns.load();
    a.num_sms = current_num_sms();  // 0 if unknown: the base ring
    return decode_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

static_assert(ATTN_DECODE_NOALLOC_SCRATCH_BYTES == attn::kDecodeNoAllocScratchBytes,
              "header and library disagree on the built-in scratch size");

int attn_decode_noalloc(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                        void *o, int B, int Hq, int Hkv, int d, float scale, int num_splits,
                        int max_seqlen, attn_stream_t stream) {
    // The argument checks of attn_decode, made here first so that a bad call
    // is refused before the one-time scratch set-up touches CUDA.
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) || !seqlens ||
        (reinterpret_cast<uintptr_t>(seqlens) & 3u))
        return ATTN_ERR_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || max_seqlen <= 0 || Hq % Hkv) return ATTN_ERR_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_ARG;
    if (num_splits > kMaxSplits) return ATTN_ERR_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (Hq / Hkv > kDecodeMaxGroup) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535 || Hkv > 65535 || (long long)max_seqlen * d * 2 >= (1LL << 39)) return ATTN_ERR_ARG;
    const size_t cap = kDecodeNoAllocScratchBytes;
    if (num_splits <= 0) {
        const int sms = current_num_sms();
        if (sms <= 0) return ATTN_ERR_CUDA;
        num_splits = splits_for(B, Hkv, max_seqlen, sms);
        while (num_splits > 1 && attn_decode_workspace_bytes(B, Hq, d, num_splits) > cap) --num_splits;
    } else if (attn_decode_workspace_bytes(B, Hq, d, num_splits) > cap) {
        return ATTN_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    const cudaError_t se = decode_noalloc_scratch(&scratch);
    if (se != cudaSuccess || !scratch) return note_cuda_error(se, "cudaGetSymbolAddress(scratch)");
    return attn_decode(q, kcache, vcache, seqlens, o, B, Hq, Hkv, d, scale, num_splits, max_seqlen,
                       scratch, cap, stream);
}

int attn_device_status(attn_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    int a = 0, b = 0, c = 0, e = 0, f = 0;
    if (fwd_take_status(&a) != cudaSuccess || decode_take_status(&b) != cudaSuccess ||
        bwd_take_status(&c) != cudaSuccess || fwd_pair_take_status(&e) != cudaSuccess ||
        fwd_split_take_status(&f) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return (a | b | c | e | f) ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

}  // extern "C"
