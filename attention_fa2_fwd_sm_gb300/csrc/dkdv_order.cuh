// dkdv_order.cuh -- work-unit scheduler of the backward's dK/dV pass (host +
// device).  The orders are the forward's (tile_order.cuh) applied to a pass
// whose Attention Compute Cluster is one (batch entry, KV head) pair: its CTAs
// all stream the Q/dO rows of the query heads that read that KV head.
#pragma once

#include "tile_order.cuh"

namespace attn {

// A dK/dV unit is key block j (kKeyBlock keys) of KV head g of batch entry b;
// the CTA streams the Q/dO rows of the G query heads that read that KV head,
// so a (b, g) pair is the pass's ACC.  Under the causal mask key block j is
// read by the N - kKeyBlock j query rows after it: block 0 is the longest.
// Head-first: pairs one after another, j fastest and ascending.  With a window
// W > 1, W consecutive pairs form a window whose units go longest first
// across its pairs (block rank, then pair), so that no pair's long blocks
// start at the end of the launch.  Block-first: the pairs run fastest.  Naive
// head-first: head-first's linear order.
constexpr int kKeyBlock = 128;
constexpr int kKvWindowWaves = 3;

struct KvTile {
    int b, g, j;  // batch entry, KV head, key block
};

__host__ __device__ inline KvTile dkdv_unit_to_tile(int order, long long u, int B, int Hkv, int nblk,
                                                    int window) {
    KvTile t;
    const int nbg = B * Hkv;
    int bg;
    if (order == kBlockFirst) {
        bg = int(u % nbg);
        t.j = int(u / nbg);
    } else if (window > 1) {
        const long long span = (long long)window * nblk;  // units of a full window
        const long long win = u / span;
        const int first = int(win) * window;              // first pair of the window
        const int width = nbg - first < window ? nbg - first : window;  // pairs in this window
        const long long r = u - win * span;
        t.j = int(r / width);
        bg = first + int(r % width);
    } else {
        t.j = int(u % nblk);
        bg = int(u / nblk);
    }
    t.b = bg / Hkv;
    t.g = bg % Hkv;
    return t;
}

// The window of a dK/dV launch: for causal head-first, the fewest pairs whose
// key blocks cover the SMs kKvWindowWaves times (a list-scheduling simulation
// of the persistent CTAs chose the factor); one pair otherwise.
__host__ __device__ inline int dkdv_window(int order, int causal, int B, int Hkv, int nblk, int num_sms) {
    if (order != kHeadFirst || !causal) return 1;
    const long long nbg = (long long)B * Hkv;
    const long long want = ((long long)kKvWindowWaves * num_sms + nblk - 1) / nblk;
    return int(want < 1 ? 1 : (want > nbg ? nbg : want));
}

}  // namespace attn
