"""Pins for the fp64 oracle: closed forms, brute force, a library routine and
invariants, so that a dropped term, a wrong sign or index or a transposed
operand in the oracle fails at least one test.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

HERE = os.path.dirname(os.path.abspath(__file__))


def _inf(x):
    return -math.inf if x == "-inf" else x


def _golden():
    with open(os.path.join(HERE, "golden", "closed_form.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["attention"], ids=lambda c: c["name"])
def test_closed_form_attention(oracle, case):
    o, lse = oracle.attention_head(case["q"], case["k"], case["v"], case["scale"], case["causal"])
    np.testing.assert_allclose(o, np.array(case["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(case["lse"]), rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", _golden()["merge"], ids=lambda c: c["name"])
def test_closed_form_merge(oracle, case):
    parts = np.array(case["o_parts"], dtype=np.float64)
    lses = np.array([_inf(x) for x in case["lse_parts"]], dtype=np.float64)
    o, lse = oracle.lse_merge(parts, lses)
    np.testing.assert_allclose(o, np.array(case["o"]), rtol=0, atol=1e-12)
    exp_lse = _inf(case["lse"])
    if exp_lse == -math.inf:
        assert lse == -math.inf
    else:
        assert abs(lse - exp_lse) <= 1e-12


def _brute_force(q, k, v, scale, causal):
    """Explicit score matrix, explicit softmax matrix, explicit product P V,
    with plain Python loops (tiny inputs only)."""
    nq, d = len(q), len(q[0])
    nk = len(k)
    S = [[scale * sum(q[i][c] * k[j][c] for c in range(d)) for j in range(nk)] for i in range(nq)]
    mask = [[(not causal) or j <= i for j in range(nk)] for i in range(nq)]
    P, lse = [], []
    for i in range(nq):
        e = [math.exp(S[i][j]) if mask[i][j] else 0.0 for j in range(nk)]
        z = sum(e)
        P.append([x / z for x in e])
        lse.append(math.log(z))
    O = [[sum(P[i][j] * v[j][c] for j in range(nk)) for c in range(d)] for i in range(nq)]
    return np.array(O), np.array(lse), P


@pytest.mark.parametrize("n", [1, 2, 3, 5, 17])
@pytest.mark.parametrize("d", [1, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(oracle, n, d, causal):
    rng = np.random.default_rng(100 * n + d + int(causal))
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref, P = _brute_force(q.tolist(), k.tolist(), v.tolist(), scale, causal)
    for row in P:  # every probability row sums to one
        assert abs(sum(row) - 1.0) <= 1e-13
    o, lse = oracle.attention_head(q, k, v, scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (4, 2), (8, 1)])
def test_matches_torch_sdpa_fp64(oracle, causal, hq, hkv):
    """GQA head grouping and causal alignment against torch's fp64 CPU routine."""
    g = torch.Generator().manual_seed(11 + hq + hkv + int(causal))
    B, N, d = 2, 37, 16
    q = torch.randn(B, hq, N, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, hkv, N, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, hkv, N, d, generator=g, dtype=torch.float64)
    # give every KV head a distinct offset so a wrong head index cannot hide
    v = v + 10.0 * torch.arange(hkv, dtype=torch.float64).view(1, hkv, 1, 1)
    scale = 1.0 / math.sqrt(d)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale,
                                         enable_gqa=(hq != hkv))
    o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), scale, causal)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-11, atol=1e-12)
    # lse against torch.logsumexp of the masked, scaled scores
    kr = k.repeat_interleave(hq // hkv, dim=1)
    s = scale * q @ kr.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -math.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=1e-12, atol=1e-12)


def test_single_key_returns_its_value(oracle):
    rng = np.random.default_rng(1)
    q, k, v = rng.standard_normal((4, 8)), rng.standard_normal((1, 8)), rng.standard_normal((1, 8))
    o, lse = oracle.attention_head(q, k, v, 0.3, False)
    np.testing.assert_allclose(o, np.repeat(v, 4, axis=0), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.3 * q @ k[0], rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_values(oracle, causal):
    rng = np.random.default_rng(2)
    n, d = 9, 4
    q = rng.standard_normal((n, d))
    k = np.repeat(rng.standard_normal((1, d)), n, axis=0)
    v = rng.standard_normal((n, d))
    o, _ = oracle.attention_head(q, k, v, 0.5, causal)
    if causal:
        expect = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]  # prefix means
    else:
        expect = np.repeat(v.mean(axis=0, keepdims=True), n, axis=0)
    np.testing.assert_allclose(o, expect, rtol=1e-13, atol=1e-14)


def test_joint_key_value_permutation_invariance(oracle):
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((5, 6)), rng.standard_normal((11, 6)), rng.standard_normal((11, 6))
    perm = rng.permutation(11)
    o1, l1 = oracle.attention_head(q, k, v, 0.4, False)
    o2, l2 = oracle.attention_head(q, k[perm], v[perm], 0.4, False)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-14)


def test_common_key_shift_only_moves_lse(oracle):
    """Adding u to every key adds scale*q.u to every score of a row: o is
    unchanged and lse moves by exactly that amount."""
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal((5, 6)), rng.standard_normal((13, 6)), rng.standard_normal((13, 6))
    u = rng.standard_normal(6)
    o1, l1 = oracle.attention_head(q, k, v, 0.4, False)
    o2, l2 = oracle.attention_head(q, k + u, v, 0.4, False)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2 - l1, 0.4 * q @ u, rtol=1e-11, atol=1e-12)


def test_empty_key_range(oracle):
    q = np.ones((1, 4))
    k = np.ones((3, 4))
    o, lse = oracle.attention_head(q, k, k, 1.0, False, k_lo=2, k_hi=2)
    assert np.all(o == 0.0) and lse[0] == -math.inf


@pytest.mark.parametrize("seqlen", [0, 1, 63, 64, 65, 1000, 4096])
@pytest.mark.parametrize("splits", [1, 2, 3, 8, 64])
def test_split_ranges_partition_the_keys(oracle, seqlen, splits):
    r = oracle.split_ranges(seqlen, splits)
    assert len(r) == splits
    covered = []
    for lo, hi in r:
        assert 0 <= lo <= hi <= seqlen
        covered.extend(range(lo, hi))
    assert covered == list(range(seqlen))
    chunk = r[0][1] - r[0][0]
    if seqlen:
        assert chunk % 64 == 0 or chunk == seqlen


@pytest.mark.parametrize("splits", [1, 2, 5, 16])
def test_merge_of_split_partials_equals_unsplit(oracle, splits):
    """Merging per-split (o, lse) reproduces attention over the whole range,
    including splits that hold no keys."""
    rng = np.random.default_rng(5 + splits)
    B, hq, hkv, s_max, d = 2, 4, 2, 300, 8
    q = rng.standard_normal((B, hq, d))
    kc = rng.standard_normal((B, hkv, s_max, d))
    vc = rng.standard_normal((B, hkv, s_max, d))
    seqlens = [300, 70]
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle.decode(q, kc, vc, seqlens, scale)
    parts, lses = oracle.decode_partials(q, kc, vc, seqlens, scale, splits)
    o, lse = oracle.lse_merge(parts, lses)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-13)


def test_decode_matches_torch_sdpa_with_lengths(oracle):
    g = torch.Generator().manual_seed(21)
    B, hq, hkv, s_max, d = 3, 8, 2, 50, 16
    q = torch.randn(B, hq, d, generator=g, dtype=torch.float64)
    kc = torch.randn(B, hkv, s_max, d, generator=g, dtype=torch.float64)
    vc = torch.randn(B, hkv, s_max, d, generator=g, dtype=torch.float64)
    seqlens = [50, 17, 1]
    scale = 1 / math.sqrt(d)
    o, _ = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), seqlens, scale)
    for b in range(B):
        n = seqlens[b]
        ref = F.scaled_dot_product_attention(q[b:b + 1, :, None, :], kc[b:b + 1, :, :n],
                                             vc[b:b + 1, :, :n], scale=scale, enable_gqa=True)
        np.testing.assert_allclose(o[b], ref[0, :, 0].numpy(), rtol=1e-11, atol=1e-12)


def test_decode_equals_causal_prefill_row(oracle):
    """Decode of query row i over the first i+1 keys is causal prefill row i."""
    rng = np.random.default_rng(6)
    n, d = 40, 8
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    o_c, l_c = oracle.attention_head(q, k, v, 0.35, True)
    for i in (0, 1, 17, 39):
        o_d, l_d = oracle.decode(q[i][None, None], k[None, None], v[None, None], [i + 1], 0.35)
        np.testing.assert_allclose(o_d[0, 0], o_c[i], rtol=1e-12, atol=1e-13)
        assert abs(l_d[0, 0] - l_c[i]) <= 1e-12


def test_thread_count_does_not_change_results(oracle):
    rng = np.random.default_rng(8)
    q, k, v = rng.standard_normal((33, 8)), rng.standard_normal((50, 8)), rng.standard_normal((50, 8))
    a = oracle.attention_head(q, k, v, 0.3, True, qpos=np.arange(17, 50), nthreads=1)
    b = oracle.attention_head(q, k, v, 0.3, True, qpos=np.arange(17, 50), nthreads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_key_range_partials_merge_to_the_full_causal_attention(oracle):
    """Causal prefill over key ranges: each range's partial (O over the range,
    normalised by its own sum, and its lse) merged with the log-sum-exp
    weights gives the full attention; a row takes only the ranges that start
    at or before it (the later ones attend no key).  The same identity as the
    decode merge, for query rows at every position of a causal prefill."""
    rng = np.random.default_rng(21)
    N, d, C = 37, 8, 10  # ranges [0,10) [10,20) [20,30) [30,37)
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    scale = 0.4
    o_full, lse_full = oracle.attention_head(q, k, v, scale, True)
    starts = list(range(0, N, C))
    parts_o = np.zeros((N, len(starts), d))
    parts_l = np.full((N, len(starts)), -np.inf)
    for s, lo in enumerate(starts):
        o_s, l_s = oracle.attention_head(q, k, v, scale, True, k_lo=lo, k_hi=min(lo + C, N))
        for i in range(N):
            if lo <= i:  # the range holds at least key lo <= i
                parts_o[i, s], parts_l[i, s] = o_s[i], l_s[i]
            else:
                assert l_s[i] == -np.inf  # no key of the range is attended
    o_m, l_m = oracle.lse_merge(parts_o, parts_l)
    assert np.abs(o_m - o_full).max() < 1e-12
    assert np.abs(l_m - lse_full).max() < 1e-12
