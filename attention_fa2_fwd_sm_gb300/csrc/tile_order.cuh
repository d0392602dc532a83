// tile_order.cuh -- work-unit scheduler of the forward kernel (host + device).
//
// A unit is kUnitRows query rows of one query head of one batch entry.  The
// order decides which units run at the same time, and hence which K/V tiles
// the L2 cache can share between concurrently running CTAs.
//
// "Optimizing Attention on GPUs by Exploiting GPU Architectural NUMA
// Effects" (detail page): an Attention Compute Cluster (ACC) is the set of
// workgroups sharing one head's K/V (one KV group for GQA), section 2 Q2;
// head-first runs one ACC's row blocks together, block-first runs every head
// of one row block together (section 3 "before/after" table).  The XCD
// placement half of the pages' swizzle has no counterpart here: the GPU's
// L2 is coherent across its two dies (section 2 Q1), so the head-first order
// alone keeps the ACC's CTAs together in time.
#pragma once

#include <cstdint>

namespace attn {

constexpr int kUnitRows = 256;  // query rows per unit (two 128-row MMA tiles)

enum TileOrder : int { kHeadFirst = 0, kBlockFirst = 1, kNaiveHeadFirst = 2, kDieSplitHeadFirst = 3 };

constexpr int kDies = 2;  // the GPU's two dies

struct Tile {
    int b, h, m;  // batch entry, query head, 256-row block index
};

__host__ __device__ inline int unit_blocks(int N) { return (N + kUnitRows - 1) / kUnitRows; }

// Linear unit id -> tile.  Head-first (and naive head-first): the block index
// runs fastest, then the query head, then the batch entry; because query
// heads of one KV group are contiguous, a group's units are consecutive.
// Block-first: the query head runs fastest.  Causal: blocks are visited in
// descending order so the longest units start first.
__host__ __device__ inline Tile unit_to_tile(int order, long long u, int Hq, int nb, int causal) {
    Tile t;
    int r;
    if (order == kBlockFirst) {
        t.h = int(u % Hq);
        long long bm = u / Hq;
        r = int(bm % nb);
        t.b = int(bm / nb);
    } else {
        r = int(u % nb);
        long long bh = u / nb;
        t.h = int(bh % Hq);
        t.b = int(bh / Hq);
    }
    t.m = causal ? (nb - 1 - r) : r;
    return t;
}

// Head-first (and die-split, whose unit ids are head-first ids) for causal
// attention with G > 1 query heads per KV head: still ACC-major (an ACC's
// G * nb units are consecutive), but inside the ACC the units go longest
// first across its query heads -- block rank, then head -- so that the last
// ACC's long units do not start last.
__host__ __device__ inline Tile unit_to_tile_grouped_causal(long long u, int Hq, int G, int nb) {
    const long long upa = (long long)G * nb;  // units per ACC
    const long long a = u / upa;             // ACC = b * Hkv + KV head
    const int w = int(u % upa);
    const int Hkv = Hq / G;
    Tile t;
    t.h = int(a % Hkv) * G + w % G;
    t.b = int(a / Hkv);
    t.m = nb - 1 - w / G;
    return t;
}

// Whether an order uses the grouped causal mapping above.
__host__ __device__ inline bool grouped_causal_order(int order, int G, int causal) {
    return causal && G > 1 && (order == kHeadFirst || order == kDieSplitHeadFirst);
}

// Causal GQA head-first on batch entries whose K/V all fit in L2 together
// (Hkv * nb <= kWholeEntryBlocks, nb = ceil(N / 256): 8 KV heads of 16K keys,
// 64 MiB of K and V at d = 128, half the L2).  No ACC's K/V can then be
// evicted for another's, which is what head-first guards against, so the
// entry's units go longest first over all its query heads: the block-first
// sequence, which balances the persistent CTAs' unequal causal units better
// than longest first inside each ACC (GQA 64/8 causal, one box: 1517 -> 1560
// TFLOP/s at 8K, 1636 -> 1681 at 16K; at 32K neither order leads on every box).
constexpr long long kWholeEntryBlocks = 512;
__host__ __device__ inline int effective_order(int order, int Hq, int G, int nb, int causal) {
    const bool whole = causal && G > 1 && (long long)(Hq / G) * nb <= kWholeEntryBlocks;
    return order == kHeadFirst && whole ? kBlockFirst : order;
}

// The mapping of any order (host view and tests).
__host__ __device__ inline Tile unit_to_tile(int order, long long u, int Hq, int G, int nb, int causal) {
    const int eo = effective_order(order, Hq, G, nb, causal);
    return grouped_causal_order(eo, G, causal) ? unit_to_tile_grouped_causal(u, Hq, G, nb)
                                               : unit_to_tile(eo, u, Hq, nb, causal);
}

// Die-split head-first: the Attention Compute Clusters (ACC: the query heads
// of one KV head of one batch entry, G * nb consecutive head-first units) are
// dealt to the dies in turn, ACC a to die a % kDies, and each die walks its
// own ACCs in head-first order.  This is the pages' Swizzled Head-first idea
// (every ACC confined to one chiplet, detail page section 2 Q2 and Figure 10)
// with the GPU's dies in place of XCDs.  Returns the head-first unit id of the
// k-th unit of die `die`, or -1 when that die has no k-th unit.  (Unit ids are
// head-first ids, so unit_to_tile maps them.)
__host__ __device__ inline long long die_split_unit(int die, long long k, int B, int Hkv, int G, int nb) {
    const long long upa = (long long)G * nb;  // units per ACC
    const long long n_acc = (long long)B * Hkv;
    if (k < 0 || die < 0 || die >= kDies) return -1;
    const long long a = (k / upa) * kDies + die;  // ACC index
    if (a >= n_acc) return -1;
    return a * upa + (k % upa);
}

// Number of units die `die` owns under die-split head-first.
__host__ __device__ inline long long die_split_units(int die, int B, int Hkv, int G, int nb) {
    const long long n_acc = (long long)B * Hkv;
    const long long accs = n_acc / kDies + (die < n_acc % kDies ? 1 : 0);
    return accs * G * nb;
}

}  // namespace attn
