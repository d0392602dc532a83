"""GPU parity of the split-KV decode and the log-sum-exp merge against the
fp64 oracle, through the C ABI: ragged and empty sequences, several split
counts (including empty splits), the workspace partials themselves, group
sizes 1..16, and every element of the full decode configurations."""
import gc

import numpy as np
import pytest
import torch

import oracle
from synthetic_inputs import decode_inputs, ragged_seqlens
from tests.gpu_util import assert_close, scale_of, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    from attention_fa2_fwd_sm_gb300 import _build
    _build.build()
    import attention_fa2_fwd_sm_gb300 as A
    A.lib()
    oracle.build()
    return A


def _decode(A, q, kc, vc, seqlens_list, splits):
    dev = q.device
    seqlens = torch.tensor(seqlens_list, dtype=torch.int32, device=dev)
    o, ws, used = A.decode(q, kc, vc, seqlens, num_splits=splits)
    torch.cuda.synchronize()
    A.check(A.attn_device_status(), "device status")
    return o, ws, used


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 7, 16, 0])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_matches_oracle(attn, splits, d):
    dev = torch.device("cuda")
    B, Hq, Hkv, S = 4, 64, 8, 1000
    q, kc, vc = decode_inputs(20 + d, B, Hq, Hkv, S, d, dev)
    lens = [1000, 357, 0, 65]
    o, _, _ = _decode(attn, q, kc, vc, lens, splits)
    o_ref, _ = oracle.decode(to64(q), to64(kc), to64(vc), lens, scale_of(d))
    assert_close(to64(o), o_ref, what=f"d={d} splits={splits}")
    assert torch.count_nonzero(o[2]) == 0  # empty sequence -> zeros


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_decode_group_sizes(attn, G):
    dev = torch.device("cuda")
    Hkv, B, S, d = 4, 2, 700, 128
    q, kc, vc = decode_inputs(30 + G, B, G * Hkv, Hkv, S, d, dev)
    lens = ragged_seqlens(B, S, 9 + G)
    o, _, _ = _decode(attn, q, kc, vc, lens, 3)
    o_ref, _ = oracle.decode(to64(q), to64(kc), to64(vc), lens, scale_of(d))
    assert_close(to64(o), o_ref, what=f"G={G}")


@pytest.mark.parametrize("splits", [2, 5, 16])
def test_workspace_partials_match_the_oracle(attn, splits):
    """The per-split partial states (normalised O_s and lse_s, -inf when the
    split is empty) before the merge."""
    dev = torch.device("cuda")
    B, Hq, Hkv, S, d = 2, 16, 2, 900, 128
    q, kc, vc = decode_inputs(40 + splits, B, Hq, Hkv, S, d, dev)
    lens = [900, 130]
    o, ws, used = _decode(attn, q, kc, vc, lens, splits)
    assert used == splits
    n = B * Hq * splits
    o_bytes = -(-(n * d * 4) // 256) * 256
    wsf = ws.view(torch.float32)
    o_parts = wsf[: n * d].view(B, Hq, splits, d)
    lse_parts = wsf[o_bytes // 4: o_bytes // 4 + n].view(B, Hq, splits)
    po_ref, pl_ref = oracle.decode_partials(to64(q), to64(kc), to64(vc), lens, scale_of(d), splits)
    fin = np.isfinite(pl_ref)
    got_l = to64(lse_parts)
    assert np.array_equal(np.isfinite(got_l), fin)
    assert np.abs(got_l[fin] - pl_ref[fin]).max() <= 1e-3
    assert_close(to64(o_parts)[fin], po_ref[fin], what="partials")
    m_ref, _ = oracle.lse_merge(po_ref, pl_ref)
    assert_close(to64(o), m_ref, what="merged")


def test_split_heuristic_follows_its_rule(attn):
    """attn_decode_num_splits restated from its header: round(floor(5 SMs / 3)
    / (B Hkv)), capped by floor(S / 512) and by 256, at least 1; then doubled
    while every split keeps at least 4096 keys and the grid stays within four
    CTAs per SM.  On a 152-SM GB300 it gives the counts the split sweep
    measured for the decode configurations."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def rule(B, Hkv, S):
        ctas = B * Hkv
        s = max(1, min((5 * sms // 3 + ctas // 2) // ctas, S // 512, 256))
        while 2 * s <= 256 and S // (2 * s) >= 4096 and ctas * 2 * s <= 4 * sms:
            s *= 2
        return s

    for B in (1, 2, 8, 32, 300):
        for S in (1, 511, 4096, 8192, 32768, 131072, 1 << 20):
            assert attn.attn_decode_num_splits(B, 64, 8, S) == rule(B, 8, S), (B, S)
    if sms == 152:
        got = [attn.attn_decode_num_splits(B, 64, 8, S) for B in (1, 8, 32) for S in (8192, 32768, 131072)]
        assert got == [16, 32, 32, 4, 8, 8, 2, 2, 2]


def test_ring_depth_boundary(attn):
    """A split grid of at most one CTA per SM runs the six-stage K/V ring, a
    larger one the three-stage ring; both sides of the boundary match the
    oracle (some of these splits are empty)."""
    dev = torch.device("cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, Hq, Hkv, S, d = 1, 64, 8, 4000, 128
    n = sms // Hkv  # n * Hkv CTAs fit one per SM; n + 1 do not
    q, kc, vc = decode_inputs(52, B, Hq, Hkv, S, d, dev)
    lens = [S - 3]
    o_ref, _ = oracle.decode(to64(q), to64(kc), to64(vc), lens, scale_of(d))
    for splits in (n, n + 1):
        o, _, _ = _decode(attn, q, kc, vc, lens, splits)
        assert_close(to64(o), o_ref, what=f"splits={splits} ({splits * Hkv} CTAs, {sms} SMs)")


def test_split_counts_agree(attn):
    dev = torch.device("cuda")
    B, Hq, Hkv, S, d = 2, 64, 8, 5000, 128
    q, kc, vc = decode_inputs(50, B, Hq, Hkv, S, d, dev)
    lens = [5000, 4097]
    outs = [_decode(attn, q, kc, vc, lens, s)[0].float() for s in (1, 4, 16, 64)]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 2e-2


def test_nan_garbage_past_seqlen_is_ignored(attn):
    """Cache slots past seqlens[b] may hold anything (here NaN): they must not
    leak into the output."""
    dev = torch.device("cuda")
    B, Hq, Hkv, S, d = 2, 16, 2, 300, 128
    q, kc, vc = decode_inputs(60, B, Hq, Hkv, S, d, dev)
    lens = [130, 77]
    kc2, vc2 = kc.clone(), vc.clone()
    for b, n in enumerate(lens):
        kc2[b, :, n:] = float("nan")
        vc2[b, :, n:] = float("nan")
    o, _, _ = _decode(attn, q, kc2, vc2, lens, 2)
    o_ref, _ = oracle.decode(to64(q), to64(kc), to64(vc), lens, scale_of(d))
    assert_close(to64(o), o_ref, what="nan past seqlen")


FULL = [(b, s) for b in (1, 8, 32) for s in (8192, 32768, 131072)]


@pytest.mark.parametrize("B,S", FULL)
def test_full_size_every_element(attn, B, S):
    """The GQA decode configurations (Hq=64, Hkv=8, d=128, batch 1/8/32, KV
    length 8K/32K/128K, the heuristic's split count), every output element
    against the oracle.  The oracle runs on one (batch entry, KV head) pair's
    slices at a time, so only that pair's cache is ever widened to fp64; the
    pairs of one batch entry run on a thread pool (the oracle's C calls
    release the interpreter lock)."""
    from concurrent.futures import ThreadPoolExecutor
    dev = torch.device("cuda")
    Hq, Hkv, d = 64, 8, 128
    G = Hq // Hkv
    q, kc, vc = decode_inputs(70, B, Hq, Hkv, S, d, dev)
    seqlens = torch.full((B,), S, dtype=torch.int32, device=dev)
    try:
        o, _, used = attn.decode(q, kc, vc, seqlens, num_splits=0)
        torch.cuda.synchronize()
        attn.check(attn.attn_device_status(), "device status")
        o64 = to64(o)
        q64 = to64(q)

        def pair(b, g, k64, v64):
            o_ref, _ = oracle.decode(q64[b:b + 1, g * G:(g + 1) * G], k64[None, None], v64[None, None], [S],
                                     scale_of(d))
            return b, g, o_ref

        with ThreadPoolExecutor(max_workers=min(Hkv, oracle.default_threads())) as pool:
            for b in range(B):
                # widen on the device, one batch entry at a time
                kb = kc[b].double().cpu().numpy()
                vb = vc[b].double().cpu().numpy()
                jobs = [pool.submit(pair, b, g, kb[g], vb[g]) for g in range(Hkv)]
                for j in jobs:
                    bb, g, o_ref = j.result()
                    assert_close(o64[bb:bb + 1, g * G:(g + 1) * G], o_ref,
                                 what=f"B={B} S={S} b={bb} g={g} splits={used}")
                del kb, vb
    finally:
        del q, kc, vc
        gc.collect()
        torch.cuda.empty_cache()
