"""Pins for the tile-order definitions (integer, exhaustive).  CPU only."""
import pytest

from oracle import tile_order as T


@pytest.mark.parametrize("order", T.ORDERS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,nb,G", [(1, 2, 1, 1), (1, 8, 5, 1), (2, 3, 4, 1), (4, 128, 3, 1), (1, 64, 32, 1),
                                      (1, 8, 5, 4), (2, 6, 4, 3), (1, 64, 32, 8), (3, 2, 1, 2)])
def test_orders_are_bijections(order, causal, B, H, nb, G):
    seen = {T.unit_to_tile(order, u, B, H, nb, causal, G) for u in range(B * H * nb)}
    assert seen == {(b, h, m) for b in range(B) for h in range(H) for m in range(nb)}


@pytest.mark.parametrize("B,Hq,G,nb", [(1, 16, 4, 130), (2, 6, 3, 257), (1, 64, 8, 65)])
def test_causal_gqa_head_first_runs_each_acc_longest_first(B, Hq, G, nb):
    """Each ACC's G * nb units are consecutive, and inside the ACC the units
    come in non-increasing causal length (block index descending), every
    head of the group at each length."""
    seq = [T.unit_to_tile(T.HEAD_FIRST, u, B, Hq, nb, True, G) for u in range(B * Hq * nb)]
    upa = G * nb
    for a in range(B * Hq // G):
        acc = seq[a * upa:(a + 1) * upa]
        assert {(b, h // G) for b, h, _ in acc} == {divmod(a, Hq // G)}
        ms = [m for _, _, m in acc]
        assert ms == sorted(ms, reverse=True)
        for i in range(0, upa, G):
            assert sorted(h % G for _, h, _ in acc[i:i + G]) == list(range(G))


@pytest.mark.parametrize("causal", [False, True])
def test_head_first_finishes_a_head_before_the_next(causal):
    B, H, nb = 2, 6, 7
    seq = [T.unit_to_tile(T.HEAD_FIRST, u, B, H, nb, causal) for u in range(B * H * nb)]
    for i in range(0, len(seq), nb):  # each run of nb units is one (b, h)
        assert len({(b, h) for b, h, _ in seq[i:i + nb]}) == 1
    if causal:  # longest (last) block first inside each head
        assert [m for _, _, m in seq[:nb]] == list(range(nb - 1, -1, -1))


def test_head_first_keeps_a_gqa_group_together():
    """Query heads of one KV group (contiguous groups) are consecutive."""
    B, Hq, Hkv, nb = 1, 16, 4, 3
    G = Hq // Hkv
    groups = [T.unit_to_tile(T.HEAD_FIRST, u, B, Hq, nb, False)[1] // G for u in range(B * Hq * nb)]
    assert groups == sorted(groups)


def test_block_first_cycles_heads_innermost():
    B, H, nb = 1, 5, 4
    seq = [T.unit_to_tile(T.BLOCK_FIRST, u, B, H, nb, False) for u in range(H * nb)]
    assert [h for _, h, _ in seq[:H]] == list(range(H))
    assert {m for _, _, m in seq[:H]} == {0}


def test_naive_head_first_has_the_head_first_linear_order():
    """Equal except for causal GQA, where naive head-first keeps the linear
    (head, block) order of a one-CTA-per-unit launch."""
    for u in range(2 * 3 * 4):
        assert (T.unit_to_tile(T.NAIVE_HEAD_FIRST, u, 2, 3, 4, True)
                == T.unit_to_tile(T.HEAD_FIRST, u, 2, 3, 4, True))
        assert (T.unit_to_tile(T.NAIVE_HEAD_FIRST, u, 2, 6, 4, False, 2)
                == T.unit_to_tile(T.HEAD_FIRST, u, 2, 6, 4, False, 2))
    assert ([T.unit_to_tile(T.NAIVE_HEAD_FIRST, u, 1, 4, 3, True, 2) for u in range(4)]
            == [(0, 0, 2), (0, 0, 1), (0, 0, 0), (0, 1, 2)])


@pytest.mark.parametrize("B", [1, 2, 4])
@pytest.mark.parametrize("H", [8, 128])
@pytest.mark.parametrize("X", [1, 4, 8])
def test_swizzle_is_a_bijection(B, H, X):
    nb = 16
    seen = {T.swizzled_head_first(w, B, H, nb, X) for w in range(B * H * nb)}
    assert len(seen) == B * H * nb
    assert all(0 <= b < B and 0 <= h < H and 0 <= m < nb for b, h, m in seen)


def test_swizzle_figure10_each_head_on_one_xcd():
    """Figure 10 of the detail page: 8 query heads, 128 row blocks, 4 XCDs; with
    round-robin dispatch (WG w runs on XCD w % 4) every head lands on one XCD."""
    H, nb, X = 8, 128, 4
    xcd_of_head = {}
    for w in range(H * nb):
        _, h, _ = T.swizzled_head_first(w, 1, H, nb, X)
        xcd_of_head.setdefault(h, set()).add(w % X)
    assert all(len(s) == 1 for s in xcd_of_head.values())
    # two heads per XCD, each XCD used
    per_xcd = {}
    for h, s in xcd_of_head.items():
        per_xcd.setdefault(next(iter(s)), []).append(h)
    assert sorted(len(v) for v in per_xcd.values()) == [2, 2, 2, 2]


def test_swizzle_with_one_xcd_is_naive_head_first():
    B, H, nb = 2, 8, 9
    for w in range(B * H * nb):
        assert T.swizzled_head_first(w, B, H, nb, 1) == T.unit_to_tile(T.HEAD_FIRST, w, B, H, nb, False)


def test_swizzle_printed_batch_line_is_not_a_bijection_for_two_batches():
    """The page's per-batch id ``wid // BATCH`` (read literally) collides for
    BATCH = 2; this is why the reading ``wid % (H * blocks)`` is used."""
    B, H, nb, X = 2, 8, 4, 4

    def literal(wid):
        wpb = wid // B
        hpx = H // X
        head = (wpb % X) * hpx + wpb // (X * nb)
        block = (wpb % (X * nb)) // X
        batch = (wid // (nb * H)) % B
        return batch, head, block

    assert len({literal(w) for w in range(B * H * nb)}) < B * H * nb
    assert len({T.swizzled_head_first(w, B, H, nb, X) for w in range(B * H * nb)}) == B * H * nb


def test_swizzle_rejects_heads_not_divisible_by_xcds():
    with pytest.raises(ValueError):
        T.swizzled_head_first(0, 1, 12, 4, 8)


def test_chiplet_swizzle_is_a_permutation():
    for X, grid in [(8, 64), (4, 4096)]:
        assert sorted(T.swizzle_chiplet(w, grid, X) for w in range(grid)) == list(range(grid))


@pytest.mark.parametrize("B,Hq,Hkv,nb", [(1, 128, 128, 4), (1, 64, 8, 3), (3, 8, 1, 2), (2, 6, 3, 5)])
@pytest.mark.parametrize("causal", [False, True])
def test_die_split_partitions_units_by_acc(B, Hq, Hkv, nb, causal):
    seqs = [T.die_split_sequence(d, B, Hq, Hkv, nb, causal) for d in (0, 1)]
    every = [x for s in seqs for x in s]
    assert sorted(every) == sorted((b, h, m) for b in range(B) for h in range(Hq) for m in range(nb))
    G = Hq // Hkv
    for d, seq in enumerate(seqs):  # each ACC lives on exactly one die
        assert all(((b * Hkv + h // G) % 2) == d for b, h, _ in seq)


def test_die_split_each_die_is_head_first_over_its_accs():
    """Per die the order is the head-first order restricted to that die's
    ACCs; for one ACC per die it is exactly the head-first order of that ACC."""
    B, Hq, Hkv, nb = 1, 4, 2, 3
    G = Hq // Hkv
    hf = [T.unit_to_tile(T.HEAD_FIRST, u, B, Hq, nb, True, G, whole_entry=False) for u in range(B * Hq * nb)]
    for d in (0, 1):
        assert T.die_split_sequence(d, B, Hq, Hkv, nb, True) == [x for x in hf if x[1] // G == d]


@pytest.mark.parametrize("causal", [False, True])
def test_die_split_with_one_die_is_head_first(causal):
    B, Hq, Hkv, nb = 2, 6, 3, 4
    assert T.die_split_sequence(0, B, Hq, Hkv, nb, causal, dies=1) == [
        T.unit_to_tile(T.HEAD_FIRST, u, B, Hq, nb, causal, Hq // Hkv, whole_entry=False)
        for u in range(B * Hq * nb)]


# ------------------------------------------------------- backward dK/dV order
DKDV_SHAPES = [  # B, Hkv, N, num_sms
    (1, 8, 8192, 152),     # window of all 8 heads
    (1, 8, 16384, 152),    # windows of 4
    (1, 7, 11739, 152),    # windows of 5: a partial last window
    (2, 3, 1000, 152),     # pairs across batch entries, one window
    (1, 8, 32768, 152),    # windows of 2
    (1, 2, 200000, 152),   # long: one pair per window
    (3, 5, 3000, 8),       # few SMs: windows of 1
]


@pytest.mark.parametrize("B,Hkv,N,sms", DKDV_SHAPES)
@pytest.mark.parametrize("order", T.ORDERS)
@pytest.mark.parametrize("causal", [False, True])
def test_dkdv_sequence_is_a_permutation(B, Hkv, N, sms, order, causal):
    nblk = T.num_blocks(N, T.KEY_BLOCK)
    seq = T.dkdv_sequence(order, B, Hkv, N, causal, sms)
    assert sorted(seq) == [(b, g, j) for b in range(B) for g in range(Hkv) for j in range(nblk)]


@pytest.mark.parametrize("B,Hkv,N,sms", DKDV_SHAPES)
def test_causal_head_first_dkdv_windows(B, Hkv, N, sms):
    """Each window holds the fewest consecutive pairs whose blocks number at
    least three times the SMs (or every pair), and runs longest first: the
    key block never decreases inside a window, and within one key block the
    window's pairs appear in increasing order."""
    nblk = T.num_blocks(N, T.KEY_BLOCK)
    w = T.dkdv_window(T.HEAD_FIRST, True, B, Hkv, nblk, sms)
    assert w == min(B * Hkv, max(1, -(-3 * sms // nblk)))
    assert w * nblk >= min(3 * sms, B * Hkv * nblk)
    assert w == 1 or (w - 1) * nblk < 3 * sms
    seq = T.dkdv_sequence(T.HEAD_FIRST, B, Hkv, N, True, sms)
    pos = 0
    for start in range(0, B * Hkv, w):
        width = min(w, B * Hkv - start)
        part = seq[pos:pos + width * nblk]
        pos += width * nblk
        assert {b * Hkv + g for b, g, _ in part} == set(range(start, start + width))
        assert [j for _, _, j in part] == sorted(j for _, _, j in part)
        assert [b * Hkv + g for b, g, _ in part[:width]] == list(range(start, start + width))
    # non-causal and the other orders never interleave pairs
    assert T.dkdv_window(T.HEAD_FIRST, False, B, Hkv, nblk, sms) == 1
    assert T.dkdv_window(T.NAIVE_HEAD_FIRST, True, B, Hkv, nblk, sms) == 1


def test_dkdv_head_first_without_a_window_is_pair_major():
    seq = T.dkdv_sequence(T.HEAD_FIRST, 2, 2, 300, False, 152)
    assert seq == [(0, 0, 0), (0, 0, 1), (0, 0, 2), (0, 1, 0), (0, 1, 1), (0, 1, 2),
                   (1, 0, 0), (1, 0, 1), (1, 0, 2), (1, 1, 0), (1, 1, 1), (1, 1, 2)]
    assert T.dkdv_sequence(T.BLOCK_FIRST, 1, 2, 256, True, 152) == [(0, 0, 0), (0, 1, 0), (0, 0, 1), (0, 1, 1)]


@pytest.mark.parametrize("B,Hq,G,nb", [(1, 16, 4, 5), (2, 6, 3, 4), (1, 64, 8, 32), (1, 64, 8, 64), (3, 8, 2, 64)])
def test_causal_gqa_head_first_over_a_whole_entry_is_block_first(B, Hq, G, nb):
    """When an entry's K/V fit in L2 together (KV heads x row blocks <= 512)
    causal GQA head-first takes the block-first sequence; one block more per
    head and it is ACC by ACC again."""
    assert (Hq // G) * nb <= T.WHOLE_ENTRY_BLOCKS
    for u in range(B * Hq * nb):
        assert (T.unit_to_tile(T.HEAD_FIRST, u, B, Hq, nb, True, G)
                == T.unit_to_tile(T.BLOCK_FIRST, u, B, Hq, nb, True, G))
    big = T.WHOLE_ENTRY_BLOCKS // (Hq // G) + 1
    seq = [T.unit_to_tile(T.HEAD_FIRST, u, 1, Hq, big, True, G) for u in range(Hq * big)]
    assert {h // G for _, h, _ in seq[:G * big]} == {0}  # the first ACC's units come first

