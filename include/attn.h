/*
 * attn.h -- C ABI of libattn.so: fused scaled dot-product attention for
 * NVIDIA GB300 (sm_103a), FlashAttention-2 style, with a head-first
 * persistent tile scheduler and a split-KV grouped-query decode.
 *
 * What is computed (all entry points): for each batch b, query head h and
 * query row i,
 *     s_j = scale * <q_i, k_j>,   P = softmax over the attended keys j,
 *     o_i = sum_j P_j v_j,        lse_i = log(sum_j exp(s_j))  (natural log)
 * -- the equation of "Optimizing Attention on GPUs by Exploiting GPU
 * Architectural NUMA Effects" (detail page, section 4, "Equation physical
 * meaning"), with the caller passing scale (normally 1/sqrt(d)).  Query head
 * h reads KV head h / (Hq / Hkv) (contiguous groups of query heads share one
 * KV head, as in grouped-query attention).
 *
 * Conventions shared by every entry point
 *  - Pointers named q, k, v, o, kcache, vcache, seqlens, lse and workspace
 *    are DEVICE pointers owned by the caller, 16-byte aligned, to contiguous
 *    row-major tensors.  The library never allocates, frees or keeps them.
 *  - Element types: q, k, v, o, kcache, vcache are bf16; lse and the
 *    workspace are fp32; seqlens is int32.  Arithmetic is bf16 x bf16 with
 *    fp32 accumulation; probabilities are rounded to bf16 before the P*V
 *    product; outputs are rounded to bf16 (round to nearest even).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument errors are detected on the host before any
 *    CUDA call and leave all memory untouched.
 *  - Return value: ATTN_OK (0) or one of the negative ATTN_ERR_* codes.
 *    attn_strerror() gives a message for each.
 *  - CUDA graphs: the launches of attn_fwd, attn_fwd_ex, attn_fwd_host,
 *    attn_bwd and the decode entry points can be captured into a CUDA graph
 *    on `stream` and replayed; a replay reads what the buffers hold at replay
 *    time (the ragged decode's seqlens included: it plans on the device).
 *    Make one ordinary call per device first (it sets up per-device state:
 *    kernel attributes, scratch addresses, the die map, the host-copy
 *    streams).  The persistent forward and backward kernels take one of 64
 *    scheduler slots per launch and a captured launch keeps its slot, so
 *    replay it where it cannot overlap 64 other forward or backward launches
 *    (for example, on the stream that issues them).  attn_device_status
 *    synchronises and is not captured.
 *  - Device-side bounded waits: every spin on a barrier inside the kernels
 *    is limited in time.  A wait that runs out sets a device status word and
 *    the kernel returns early (its outputs are then undefined).
 *    attn_device_status() reads and clears that word.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *attn_stream_t;

enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_ARG = -1,         /* null or misaligned pointer, bad size, Hq % Hkv != 0, scale <= 0 */
    ATTN_ERR_UNSUPPORTED = -2, /* head dimension or group size this library does not implement */
    ATTN_ERR_WORKSPACE = -3,   /* workspace missing or smaller than attn_decode_workspace_bytes() */
    ATTN_ERR_CUDA = -4,        /* a CUDA runtime or driver call failed (launch, tensor map, ...) */
    ATTN_ERR_TIMEOUT = -5      /* a bounded device wait ran out (reported by attn_device_status) */
};

/* Orders in which the persistent forward kernel visits its work units (a
 * unit = 256 query rows of one query head of one batch entry).
 *  HEAD_FIRST: all row blocks of one Attention Compute Cluster (the query
 *    heads sharing one KV head) before the next one, so CTAs running at the
 *    same time read the same K/V and reuse it in L2 (detail page, section 2
 *    Q2 and section 3 "before/after" table).  Inside an ACC the row blocks
 *    of one head follow each other; for causal GQA the ACC's units instead
 *    run longest first across its heads (block descending, then head).
 *    Causal GQA on batch entries whose K/V all fit in L2 together (Hkv times
 *    ceil(N / 256) at most 512) runs longest first over all the entry's
 *    heads instead, which is BLOCK_FIRST's sequence: no ACC can then evict
 *    another's K/V.  The backward's dQ pass (same units) follows this order.
 *  BLOCK_FIRST: all heads of one row block before the next row block (the
 *    pages' "Naive Block-first" baseline).
 *  NAIVE_HEAD_FIRST: head-first linear order, but one CTA per unit with the
 *    hardware choosing placement (the pages' "Naive Head-first").
 *  DIE_SPLIT_HEAD_FIRST: the pages' Swizzled Head-first with the GPU's two
 *    dies in place of XCDs (detail page, section 2 Q2 and Figure 10): ACC a
 *    (a = b * Hkv + KV head) belongs to die a % 2, the CTAs on each die walk
 *    their die's ACCs in head-first order, and a die that runs out takes the
 *    other die's remaining units.  Which SM is on which die is measured on the
 *    first die-split launch on each device (see attn_die_map); that first
 *    launch therefore synchronises the device and must not be captured into
 *    a CUDA graph. */
enum attn_tile_order {
    ATTN_ORDER_HEAD_FIRST = 0,
    ATTN_ORDER_BLOCK_FIRST = 1,
    ATTN_ORDER_NAIVE_HEAD_FIRST = 2,
    ATTN_ORDER_DIE_SPLIT_HEAD_FIRST = 3
};

/* Tile schemes of the forward kernel, OR-ed into the tile_order argument of
 * attn_fwd_ex and attn_fwd_host (at most one):
 *  ATTN_FWD_SINGLE_CTA: each SM runs units of 256 query rows (two 128-row
 *    MMA tiles sharing every K/V block it loads).
 *  ATTN_FWD_CTA_PAIR: pairs of SMs (a cluster of two CTAs) run units of 512
 *    query rows with tcgen05 MMAs of the cta_group::2 kind (M = 256): each SM
 *    loads half of every K/V block and one warp issues the MMAs of both.
 *    The pages keep the workgroups that share one head's K/V on one chiplet
 *    (detail page, section 2 Q1-Q2); a pair shares each block through the
 *    MMA itself.  d = 128 only (ATTN_ERR_UNSUPPORTED otherwise).  The units
 *    of the orders above are then 512-row blocks.
 * Without a flag the library picks the scheme.  Results agree across
 * schemes within the forward's tolerance; every order of one scheme gives
 * bit-identical results. */
#define ATTN_FWD_SINGLE_CTA 0x100
#define ATTN_FWD_CTA_PAIR 0x200

/*
 * Forward (prefill) attention.  Detail page, section 4 equation; FA2 tiling of
 * Figure 4 (each CTA owns a block of query rows and streams all of K and V).
 *   q      [B, Hq,  N, d]  bf16
 *   k, v   [B, Hkv, N, d]  bf16
 *   o      [B, Hq,  N, d]  bf16 (written)
 *   lse    [B, Hq,  N]     fp32 (written; may be NULL)
 *   d in {56, 64, 128}; d = 56 is computed as 64 with zero columns, which
 *   gives the same result as explicit zero padding (scale stays as passed).
 *   causal != 0 keeps key j for query i iff j <= i.
 *   B, Hq, Hkv, N >= 1; Hq % Hkv == 0; scale > 0 and finite;
 *   B * Hq * ceil(N / 128) < 2^31 (work units are handed out from 32-bit
 *   counters; no call whose tensors fit in device memory comes near it).
 * Uses the HEAD_FIRST order.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int Hq, int Hkv, int N, int d, float scale, int causal,
             attn_stream_t stream);

/* attn_fwd with an explicit tile order (enum attn_tile_order).  All orders
 * give bit-identical results; only the schedule differs. */
int attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                int tile_order, attn_stream_t stream);

/*
 * attn_fwd_ex on HOST-resident tensors, for callers whose q, k, v live in host
 * memory: the copies to the device, the forward kernels and the copies of o
 * and lse back are overlapped.  The problem is cut into chunks of
 * kv_heads_per_chunk KV heads of one batch entry (each with the Hq / Hkv
 * query heads that read them); while chunk c is computed, chunk c+1 is
 * copied in and chunk c-1 copied out.  Results are bit-identical to attn_fwd_ex
 * on device copies of the same tensors.
 *   q, k, v, o, lse  HOST pointers with the layouts of attn_fwd (lse may be
 *                    NULL).  Page-locked (pinned) memory lets the copies
 *                    overlap the kernels; with pageable memory the result
 *                    is the same but the copies do not overlap.
 *   kv_heads_per_chunk  1..Hkv, or <= 0 for the library's choice: the
 *                    fewest KV heads whose chunk holds at least 304 forward
 *                    work units (two waves on 152 SMs; a unit is 256 query
 *                    rows of one query head), at most Hkv.
 *   workspace        DEVICE memory, 16-byte aligned, of at least
 *                    attn_fwd_host_workspace_bytes(B, Hq, Hkv, N, d,
 *                    kv_heads_per_chunk) bytes: two chunk slots of q, k, v,
 *                    o and lse.
 * Ordering: everything starts after the work already enqueued on `stream`,
 * and work enqueued on `stream` after the call starts after the last copy
 * back.  The call returns once the work is enqueued; the host buffers must
 * stay valid, and o / lse unread, until `stream` has been synchronised.
 * Internally the library uses three more streams and a few events per
 * device (created on the first call); calls from several host threads are
 * enqueued one after the other.  Other arguments and errors as attn_fwd_ex;
 * ATTN_ERR_WORKSPACE if the workspace is missing, misaligned or too small.
 */
int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                  int tile_order, int kv_heads_per_chunk, void *workspace,
                  size_t workspace_bytes, attn_stream_t stream);

/* Device workspace bytes attn_fwd_host needs (0 for invalid sizes or a
 * chunk larger than Hkv). */
size_t attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int N, int d,
                                     int kv_heads_per_chunk);

/*
 * Forward attention with each head's keys split into ranges (the "sub-ACC"
 * split).  "Optimizing Attention on GPUs by Exploiting GPU Architectural NUMA
 * Effects" (related-work page) suggests, for long contexts whose per-head K/V
 * outgrows an L2 slice, splitting an Attention Compute Cluster's keys so that
 * the workgroups running together stream a piece that fits.  Here the units
 * of an ACC (the query heads of one KV head) run key range 0 for all their
 * row blocks, then range 1, and so on; each writes fp32 partials (O_s
 * normalised by its own sum, lse_s) to the workspace, and a merge kernel on
 * the same stream combines every row's ranges with the log-sum-exp weights
 * (kernbench2 "Fused Grouped-Query Attention", Case 4's (m, l, O) reduction).
 * Same tensors, layouts, arguments and errors as attn_fwd (head-first order;
 * d in {56, 64, 128}); the result agrees with attn_fwd within the forward's
 * tolerance, not bit for bit (the merge reassociates the sums).
 *   kv_splits   1..64 ranges; each range is ceil(N / kv_splits) keys rounded
 *               up to 128 (so fewer ranges may result), or <= 0 for the
 *               library's choice: the fewest ranges whose K and V of one KV
 *               head fit in 32 MiB (one range up to N = 65536 at d = 128).
 *   workspace   DEVICE memory, 16-byte aligned, of at least
 *               attn_fwd_splitkv_workspace_bytes(B, Hq, N, d, kv_splits)
 *               bytes: ranges x B x Hq x N x (d + 1) floats, rounded;
 *               ATTN_ERR_WORKSPACE if missing or short.
 * Two kernels run on `stream`.
 */
int attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                     int kv_splits, void *workspace, size_t workspace_bytes,
                     attn_stream_t stream);

/* Workspace bytes attn_fwd_splitkv needs (0 for invalid sizes). */
size_t attn_fwd_splitkv_workspace_bytes(int B, int Hq, int N, int d, int kv_splits);

/*
 * Timeline of attn_fwd_host, for measuring how far its copies overlap its
 * kernels (instrumentation; the pages define no such call).
 * attn_fwd_host_trace(1) makes every later attn_fwd_host call on the current
 * device record CUDA timing events: one on `stream` as the call starts and,
 * per chunk, one after its copy-in, one when its compute stream reaches the
 * kernel launch, one after the kernel and one after its copy-out.
 * attn_fwd_host_trace(0) stops recording (the last timeline stays readable).
 * Returns ATTN_OK or ATTN_ERR_CUDA.
 * Tracing adds only event records to the same streams; do not trace a call
 * that is being captured into a CUDA graph.
 *
 * attn_fwd_host_trace_read waits for the last traced call on the current
 * device to finish and writes, for chunk c < capacity, four times in
 * milliseconds from the call's start into ms[4c .. 4c+3]: copy-in done,
 * kernel reached, kernel done, copy-out done.  Chunks are numbered in the
 * call's order (batch entry, then KV-head chunk).  Returns the call's chunk
 * count (which may exceed capacity), ATTN_ERR_ARG if ms is NULL with
 * capacity > 0 or no traced call has been made since tracing was switched
 * on, or ATTN_ERR_CUDA.
 */
int attn_fwd_host_trace(int enable);
long long attn_fwd_host_trace_read(float *ms, long long capacity);

/*
 * Backward pass of attn_fwd: gradients dQ, dK, dV for the output gradient
 * dout.  The pages measure an FA2 backward pass under the same tile orders
 * (detail page, section 5 "backward pass"); the gradient itself is the chain
 * rule of the section-4 equation:
 *   P = exp(scale * q k^T - lse),  dV = P^T dout,  dP = dout v^T,
 *   Delta = rowsum(dout * o),  dS = P * (dP - Delta),
 *   dQ = scale * dS k,  dK = scale * dS^T q,
 * with the causal mask of the forward pass; for grouped-query attention the
 * gradient of a KV head is the sum over the Hq / Hkv query heads that read it.
 *   q, dout, o  [B, Hq,  N, d]  bf16 (o: the forward output)
 *   k, v        [B, Hkv, N, d]  bf16
 *   lse         [B, Hq,  N]     fp32, the forward's log-sum-exp (required)
 *   dq          [B, Hq,  N, d]  bf16 (written)
 *   dk, dv      [B, Hkv, N, d]  bf16 (written)
 *   d in {56, 64, 128} as in attn_fwd; tile_order HEAD_FIRST, BLOCK_FIRST or
 *   NAIVE_HEAD_FIRST (the die-split order is forward-only).
 *   workspace: device memory of at least attn_bwd_workspace_bytes(B, Hq, N)
 *   bytes, 16-byte aligned; it receives -lse * log2(e) and Delta per query row.
 *   With at least attn_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, causal) bytes
 *   the dK/dV pass may split each KV head's query heads into s groups (non-
 *   causal grouped-query problems with fewer than 912 dK/dV units, six waves
 *   on 152 SMs): each group's units write fp32 partial dK and dV into the
 *   workspace and a fourth kernel sums the s partials in a fixed order.  The
 *   split depends only on B, Hq, Hkv, N and causal; its results differ from
 *   the unsplit pass's by fp32 rounding and are, like them, independent of
 *   the tile order.
 * Three kernels run on `stream` (four when the dK/dV pass splits): the Delta
 * pre-pass, the dK/dV pass (units of 128 keys of one KV head) and the dQ pass
 * (units of 256 query rows of one query head); the two main passes are
 * persistent grids that take units in the tile order (the dQ pass in the
 * forward's, as attn_tile_map gives it).  Under HEAD_FIRST a causal dK/dV pass runs windows of the
 * fewest (batch, KV head) pairs whose key blocks cover the SMs three times,
 * longest block first across the window, so that no head's long blocks start
 * at the end of the launch.  Every output element is written once; results
 * do not depend on the order.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
             const float *lse, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N, int d,
             float scale, int causal, int tile_order, void *workspace, size_t workspace_bytes,
             attn_stream_t stream);

/* Workspace bytes attn_bwd needs: 8 * B * Hq * roundup(N, 128) (0 for bad sizes). */
size_t attn_bwd_workspace_bytes(int B, int Hq, int N);

/* Workspace bytes for attn_bwd with the dK/dV query-head split where it
 * applies: attn_bwd_workspace_bytes(B, Hq, N) rounded up to 256, plus
 * 8 * B * Hkv * s * N * d for s > 1 (s as attn_bwd chooses it); equal to
 * attn_bwd_workspace_bytes when the problem is not split; 0 for bad sizes. */
size_t attn_bwd_workspace_bytes_ex(int B, int Hq, int Hkv, int N, int d, int causal);

/*
 * Split-KV grouped-query decode, one query row per (batch, query head).
 * kernbench2 "Fused Grouped-Query Attention": decode step with T_q = 1
 * against the whole KV history; the KV sequence is split and the partial
 * softmax states (m, l, O) are merged (section "Inference with Long-Context
 * Length", Case 4).
 *   q        [B, Hq, d]                bf16
 *   kcache   [B, Hkv, max_seqlen, d]   bf16
 *   vcache   [B, Hkv, max_seqlen, d]   bf16
 *   seqlens  [B]  int32 device array; sequence b attends keys [0, seqlens[b]),
 *            each value must lie in [0, max_seqlen] (not checked on device:
 *            larger values are clamped to max_seqlen).
 *   o        [B, Hq, d]                bf16 (written; zeros for seqlens[b] = 0)
 *   d in {64, 128}; 1 <= Hq / Hkv <= 16.
 *   num_splits <= 0 picks a split count (attn_decode_num_splits); otherwise
 *   1 <= num_splits <= 256.  The key range of sequence b is cut into chunks of
 *   ceil(seqlens[b] / num_splits) keys rounded up to 64; empty chunks are
 *   allowed.  Different split counts agree up to fp32 rounding.
 *   workspace: fp32 scratch of at least attn_decode_workspace_bytes(B, Hq, d,
 *   splits) bytes (may be NULL when that is 0).  Layout: partial outputs
 *   [B, Hq, splits, d] (each normalised by its own sum) followed by partial
 *   log-sum-exps [B, Hq, splits] (-inf for an empty chunk).
 * A second kernel merges the partials when splits > 1.
 */
int attn_decode(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                void *o, int B, int Hq, int Hkv, int d, float scale, int num_splits,
                int max_seqlen, void *workspace, size_t workspace_bytes,
                attn_stream_t stream);

/* Size in bytes of the scratch array built into the library for
 * attn_decode_noalloc. */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES 4194304u

/*
 * attn_decode for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for integration.
 *
 * Who needs it: code that may not call cudaMalloc or own a buffer of its
 * own -- for example a plug-in inside a host framework whose memory pool
 * has reserved the whole device and forbids side allocations, or a
 * latency-critical serving loop where an allocation (and the device-wide
 * synchronisation it can imply) is not acceptable, or a caller whose own
 * interface has no way to pass a workspace through.  Such a caller still
 * passes its inputs and its output; the split partials go to a scratch
 * array of ATTN_DECODE_NOALLOC_SCRATCH_BYTES bytes that is part of the
 * library image.  Every GPU that loads the library holds that array until
 * the process exits.  This entry point allocates nothing and calls no
 * allocating routine.
 *
 * Arguments, layouts and results are those of attn_decode, without the
 * workspace.  num_splits <= 0 takes attn_decode_num_splits' count, lowered
 * until the partials fit in the scratch (1 split needs none).  An explicit
 * num_splits whose partials need more than the scratch holds, i.e.
 * attn_decode_workspace_bytes(B, Hq, d, num_splits) >
 * ATTN_DECODE_NOALLOC_SCRATCH_BYTES, is refused with ATTN_ERR_WORKSPACE
 * before any work is queued; argument errors are reported as by
 * attn_decode.
 *
 * Set-up: the first call on each device looks up the device address of the
 * scratch array (cudaGetSymbolAddress, with that device current) and keeps
 * it for later calls.  Make that first call before capturing any stream.
 * The kept address belongs to the context that was current on that first
 * call (normally the device's primary context, which the runtime API uses):
 * after cudaDeviceReset, or from another driver context made current on the
 * same device, the library's module is loaded anew and the kept address is
 * stale, so do not call this entry point in either situation.
 *
 * Sharing: all calls use the same array, and it keeps whatever the last call
 * wrote.  Each call writes every partial it later reads, so nothing needs
 * clearing between calls.  Calls whose kernels can run at the same time on
 * the GPU (different streams without ordering between them) race on the
 * array and give wrong results: order such calls on one stream or with
 * events.
 */
int attn_decode_noalloc(const void *q, const void *kcache, const void *vcache,
                        const int *seqlens, void *o, int B, int Hq, int Hkv, int d,
                        float scale, int num_splits, int max_seqlen, attn_stream_t stream);

/*
 * Decode for a ragged multi-user batch: the same computation and layouts as
 * attn_decode, with the work balanced over the whole batch instead of a fixed
 * split count per sequence.  kernbench2 "Fused Grouped-Query Attention":
 * the decode family reduces partial outputs per user in two levels
 * ("two-level reduce-to-root", short-context section); here the levels are
 * the warps of a CTA (combined in shared memory) and the chunks of a user
 * (one merge per (user, query head)).
 * Three kernels run on `stream`, with no host synchronisation:
 *   1. a one-CTA plan: T = sum_b min(max(seqlens[b], 0), max_seqlen) keys in
 *      all; chunk C = max(512, ceil(T * Hkv / target) rounded up to 64) with
 *      target = floor(5 * SMs / 3) (at least 1); sequence b is cut into
 *      n_b = ceil(len_b / C) chunks [c C, min(c C + C, len_b)), numbered
 *      consecutively in b;
 *   2. one decode CTA per (chunk, KV head);
 *   3. the merge of each (b, query head) over b's chunks (O = 0 when n_b = 0).
 * workspace: at least attn_decode_varlen_workspace_bytes(B, Hq, Hkv, d)
 * bytes, 16-byte aligned.  Its head holds the plan as int32: [0] chunk
 * count, [1] C, [2, 2 + B) first chunk of each b, [2 + B, 2 + 2B) n_b, then
 * (b, lo, hi) per chunk; the partial states follow.  Arguments and errors as
 * attn_decode (no num_splits); d in {64, 128}, Hq / Hkv <= 16, and
 * ceil(target / Hkv) + B <= 65535.
 */
int attn_decode_varlen(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                       void *o, int B, int Hq, int Hkv, int d, float scale, int max_seqlen,
                       void *workspace, size_t workspace_bytes, attn_stream_t stream);

/* Workspace bytes attn_decode_varlen needs on the current device: room for
 * ceil(target / Hkv) + B chunks (the most the plan can make), with target as
 * above.  0 for bad sizes or when the device cannot be queried. */
size_t attn_decode_varlen_workspace_bytes(int B, int Hq, int Hkv, int d);

/* Bytes of workspace attn_decode needs for this shape and split count
 * (0 when num_splits == 1).  num_splits <= 0 is not resolved here: pass the
 * value returned by attn_decode_num_splits. */
size_t attn_decode_workspace_bytes(int B, int Hq, int d, int num_splits);

/* Split count attn_decode uses when given num_splits <= 0: about 5/3 CTAs
 * per SM of the current device in all (B * Hkv * splits), no split shorter
 * than 512 keys, at most 256 splits; then doubled while every split keeps at
 * least 4096 keys and the grid stays within 4 CTAs per SM.  Returns a value >= 1 (or a negative
 * error code for bad arguments).  Queries the current device's SM count once. */
int attn_decode_num_splits(int B, int Hq, int Hkv, int max_seqlen);

/* Host-side view of the forward scheduler: unit `unit` of the order maps to
 * (*b, *h, *m) where m is the index of a 256-row block.  Pure host code; the
 * same function runs inside the kernel.  Orders 0-2 only (the die-split order
 * has one sequence per die: attn_tile_map_die_split).  Hkv matters for the
 * causal head-first order only.  Returns ATTN_OK or ATTN_ERR_ARG. */
int attn_tile_map(int tile_order, int B, int Hq, int Hkv, int N, int causal, long long unit,
                  int *b, int *h, int *m);

/* The k-th unit (k >= 0) that die `die` (0 or 1) takes from its own ACCs
 * under ATTN_ORDER_DIE_SPLIT_HEAD_FIRST, as (*b, *h, *m).  Pure host code; the
 * same function runs inside the kernel.  Returns ATTN_ERR_ARG when the die has
 * no k-th unit (then its CTAs take the other die's remaining units). */
int attn_tile_map_die_split(int B, int Hq, int Hkv, int N, int causal, int die, long long k,
                            int *b, int *h, int *m);

/* Host-side view of the backward's dK/dV scheduler (attn_bwd): unit `unit`,
 * 0 <= unit < B * Hkv * ceil(N / 128), maps to (*b, *g, *j): batch entry, KV
 * head and 128-key block.  num_sms is the SM count of the launch (the causal
 * HEAD_FIRST window depends on it; attn_bwd uses the current device's).
 * Orders 0-2.  Pure host code; the same function runs inside the kernel.
 * Returns ATTN_OK or ATTN_ERR_ARG. */
int attn_bwd_tile_map(int tile_order, int B, int Hkv, int N, int causal, int num_sms, long long unit,
                      int *b, int *g, int *j);

/* Which die each SM of the current device is on, as the die-split order uses
 * it.  On the first call for a device (or the first die-split launch) a short
 * calibration runs synchronously on the legacy default stream: one thread per
 * SM times dependent L2 loads to 128 probe words (every address is homed in
 * the L2 of one die, and far lines take longer), and the SMs are split into
 * the two groups whose latency patterns agree (two-means on the correlation
 * of the patterns; SM 0's group is die 0).  If the split is not clean (an SM
 * correlates with its own group's mean pattern by less than 0.5 more than
 * with the other group's, or a die would hold under a quarter of the SMs),
 * SM ids are split in halves instead.  The map is kept for the life of the
 * process; call this before any stream capture.
 *   die_of_sm  host array of `capacity` ints, receives 0 or 1 for SM ids
 *              0 .. min(capacity, SMs) - 1 (may be NULL when capacity is 0)
 *   stats      host array of 4 floats (may be NULL): [0] 1 if measured, else
 *              the reason for the halves fallback (0: the split was not
 *              clean, -1: the probe did not reach every SM, -2: more SMs
 *              than 256); [1] the smallest margin of an
 *              SM (own-group minus other-group correlation, at most 2);
 *              [2] / [3] mean near / far latency in SM clocks per dependent
 *              L2 load.
 * Returns the number of SMs, or a negative ATTN_ERR_* code. */
int attn_die_map(int *die_of_sm, int capacity, float *stats);

/* Number of work units (B * Hq * ceil(N / 256)) of the forward pass. */
long long attn_fwd_units(int B, int Hq, int N);

/* Synchronise `stream`, then read and clear the device status word that the
 * bounded waits set.  Returns ATTN_OK, ATTN_ERR_TIMEOUT or ATTN_ERR_CUDA. */
int attn_device_status(attn_stream_t stream);

/* Time limit, in nanoseconds, of every device-side barrier wait in later
 * launches (default 10 s; 0 makes any wait that is not already satisfied run
 * out at once, which tests use to exercise the timeout path).  Returns the
 * previous value. */
long long attn_set_wait_timeout_ns(long long ns);

/* Description of the last failed CUDA call made by this library on the
 * calling thread (the call behind the last ATTN_ERR_CUDA), or "" if none.
 * Thread-local storage; valid until the next failing call on this thread. */
const char *attn_last_error(void);

/* Message for a status code (static storage, never NULL). */
const char *attn_strerror(int code);

/* Library version as 10000*major + 100*minor + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
