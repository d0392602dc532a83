"""Plain definitions of the tile orders (pure integer arithmetic, slow and obvious).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Shares no code with
the CUDA scheduler; the tests compare the two mapping by mapping.

A *unit* is one CTA work item: the ``bm`` query rows ``[m*bm, (m+1)*bm)`` of
query head ``h`` in batch ``b``.  ``nb = ceil(N / bm)`` row blocks per head.

Orders (the pages' names, detail page of "Optimizing Attention on GPUs by
Exploiting GPU Architectural NUMA Effects", section 2 Q2 and section 3
"before/after" table):

* head-first: all row blocks of one Attention Compute Cluster (the query
  heads that share one KV head) before the next one.  With contiguous GQA
  groups, (batch, kv group, head in group, block) order is simply
  (batch, head, block).  For causal attention with several query heads per
  KV head the ACC's units go (block rank, head in group): every head's
  longest unit, then every head's second longest, and so on -- unless the
  batch entry's K/V all fit in L2 together (KV heads x row blocks <= 512,
  ``WHOLE_ENTRY_BLOCKS``), where no ACC can evict another's K/V and the
  entry's units go longest first over all its query heads, which is the
  block-first sequence (a reading: the pages' head-first exists for that
  cache reuse).
* block-first: all heads of one row block before the next row block.
* naive head-first: the head-first linear order, but each unit is its own
  CTA and the hardware decides where it runs.
* die-split head-first: the pages' Swizzled Head-first placement (each ACC
  confined to one chiplet, section 2 Q2 and Figure 10) with the GPU's two dies
  in place of XCDs: ACCs are dealt to the dies in turn and each die takes its
  own ACCs in head-first order (``die_split_sequence``).

For causal attention the blocks of a head are visited last-block-first, so
the longest units start first (the pages give only "ACC before next ACC";
the within-ACC orders are readings).
"""
from __future__ import annotations

HEAD_FIRST = 0
BLOCK_FIRST = 1
NAIVE_HEAD_FIRST = 2
ORDERS = (HEAD_FIRST, BLOCK_FIRST, NAIVE_HEAD_FIRST)


def num_blocks(n: int, bm: int) -> int:
    return -(-n // bm)


WHOLE_ENTRY_BLOCKS = 512  # KV heads x row blocks of an entry whose K/V fit in L2 together


def unit_to_tile(order: int, u: int, batch: int, heads: int, nb: int, causal: bool, group: int = 1,
                 whole_entry: bool = True):
    """Linear unit id -> (b, h, m); ``group`` query heads share one KV head.
    ``whole_entry=False`` keeps causal GQA head-first ACC by ACC at every
    size (the order the die-split placement deals out)."""
    total = batch * heads * nb
    if not 0 <= u < total:
        raise ValueError("unit out of range")
    if (whole_entry and order == HEAD_FIRST and causal and group > 1
            and (heads // group) * nb <= WHOLE_ENTRY_BLOCKS):
        order = BLOCK_FIRST
    if order == HEAD_FIRST and causal and group > 1:
        acc, w = divmod(u, group * nb)       # ACC = (batch entry, KV head)
        r, head_in_group = divmod(w, group)  # block rank, then head
        b, kv_head = divmod(acc, heads // group)
        h = kv_head * group + head_in_group
    elif order in (HEAD_FIRST, NAIVE_HEAD_FIRST):
        bh, r = divmod(u, nb)
        b, h = divmod(bh, heads)
    elif order == BLOCK_FIRST:
        bm_, h = divmod(u, heads)
        b, r = divmod(bm_, nb)
    else:
        raise ValueError("unknown order")
    m = nb - 1 - r if causal else r
    return b, h, m


def swizzled_head_first(wid: int, batch: int, heads: int, blocks_per_head: int, num_xcd: int):
    """The pages' Swizzled Head-first WG-ID remap (detail page, section 7,
    Figure 11 key code), returning (batch, head, block).

    Reading of a garbled line: the page computes the per-batch id as
    ``wid // BATCH`` while taking the batch as ``(wid // (blocks*H)) % BATCH``;
    the two disagree for BATCH > 1 (the map is then not one-to-one).  Here the
    batch is outermost and the per-batch id is ``wid % (H * blocks)``, which
    agrees with the printed code for BATCH = 1.
    """
    if heads % num_xcd:
        raise ValueError("heads must be a multiple of num_xcd (pages give no fallback)")
    per_batch = heads * blocks_per_head
    wid_pb = wid % per_batch
    heads_per_xcd = heads // num_xcd
    chunk = num_xcd * blocks_per_head
    head = (wid_pb % num_xcd) * heads_per_xcd + wid_pb // (num_xcd * blocks_per_head)
    block = (wid_pb % chunk) // num_xcd
    b = (wid // per_batch) % batch
    return b, head, block


def swizzle_chiplet(wgid: int, grid: int, num_xcd: int) -> int:
    """The chiplet swizzle baseline (detail page, section 7, Figure 3)."""
    per_xcd = grid // num_xcd
    return (wgid % num_xcd) * per_xcd + wgid // num_xcd


def die_split_sequence(die: int, batch: int, hq: int, hkv: int, nb: int, causal: bool, dies: int = 2):
    """Units of one die under die-split head-first, in the order that die
    takes them.  The ACCs (batch entry b, KV head g; ACC index a = b*hkv + g)
    are dealt round-robin, ACC a to die a % dies, and each die visits its ACCs
    in increasing a, each ACC in head-first order: the ACC's query heads one
    after the other, every row block of a head before the next head -- or,
    causal with several query heads per KV head, block rank by block rank
    (longest first), the ACC's heads inside each rank."""
    g_size = hq // hkv
    out = []
    for a in range(batch * hkv):
        if a % dies != die:
            continue
        b, kvh = divmod(a, hkv)
        heads = range(kvh * g_size, (kvh + 1) * g_size)
        if causal and g_size > 1:
            for r in range(nb):
                for h in heads:
                    out.append((b, h, nb - 1 - r))
        else:
            for h in heads:
                for r in range(nb):
                    out.append((b, h, nb - 1 - r if causal else r))
    return out


KEY_BLOCK = 128    # keys per dK/dV unit
WINDOW_WAVES = 3   # causal head-first dK/dV windows cover the SMs this many times


def dkdv_window(order: int, causal: bool, batch: int, hkv: int, nblk: int, num_sms: int) -> int:
    """(batch entry, KV head) pairs per window of the dK/dV order: under the
    causal mask and head-first, the fewest pairs whose key blocks together
    number at least WINDOW_WAVES * num_sms (at most every pair); one pair in
    every other case.  The pages define no backward order; this and
    ``dkdv_sequence`` are this library's reading of "head-first" for a pass
    whose ACC is one (batch entry, KV head) pair."""
    if order != HEAD_FIRST or not causal:
        return 1
    need = -(-(WINDOW_WAVES * num_sms) // nblk)
    return max(1, min(batch * hkv, need))


def dkdv_sequence(order: int, batch: int, hkv: int, n: int, causal: bool, num_sms: int):
    """Every dK/dV unit (b, g, j) -- key block j of KV head g of batch entry
    b -- in the order the persistent CTAs take them.

    * block-first: key block by key block, all pairs inside each block;
    * head-first and naive head-first: the pairs in windows of
      ``dkdv_window`` consecutive pairs; inside a window, key block by key
      block in increasing j (under the causal mask key block j is read by the
      N - 128 j query rows after it, so this is longest first), the window's
      pairs inside each block.  A window of one pair is plain head-first:
      every block of a pair before the next pair."""
    nblk = num_blocks(n, KEY_BLOCK)
    pairs = [divmod(p, hkv) for p in range(batch * hkv)]
    out = []
    if order == BLOCK_FIRST:
        for j in range(nblk):
            for b, g in pairs:
                out.append((b, g, j))
        return out
    if order not in (HEAD_FIRST, NAIVE_HEAD_FIRST):
        raise ValueError("unknown order")
    w = dkdv_window(order, causal, batch, hkv, nblk, num_sms)
    for start in range(0, len(pairs), w):
        window = pairs[start:start + w]
        for j in range(nblk):
            for b, g in window:
                out.append((b, g, j))
    return out
