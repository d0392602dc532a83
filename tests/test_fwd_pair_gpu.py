"""GPU parity of the CTA-pair forward (ATTN_FWD_CTA_PAIR: clusters of two
CTAs running 512-row units with cta_group::2 MMAs, d = 128) against the fp64
oracle, through the C ABI: small shapes element by element (ragged tails,
a pair tile half past N, N = 1, GQA, causal, more units than pairs), the
four tile orders bit for bit, agreement with the one-CTA scheme, two
launches at once on two streams, and the bounded-wait give-up."""
import pytest
import torch

import oracle
from synthetic_inputs import prefill_inputs, sample_heads, sample_rows
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


def _run(A, q, k, v, causal, order=0, scheme=None, stream=None):
    scheme = A.FWD_CTA_PAIR if scheme is None else scheme
    o, lse = A.forward(q, k, v, causal=causal, tile_order=order | scheme, stream=stream)
    torch.cuda.synchronize()
    A.check(A.attn_device_status(), "device status")
    return o, lse


SMALL = [
    # B, Hq, Hkv, N, causal
    (1, 2, 2, 256, False),
    (1, 2, 2, 700, True),
    (1, 2, 1, 1, False),
    (1, 3, 3, 129, True),
    (1, 2, 2, 513, True),     # the second unit's first pair tile: rank 0 has row 512, rank 1 none
    (1, 2, 2, 640, False),    # rank 1 of the second unit's first pair tile lies exactly past N
    (2, 4, 2, 1000, True),
    (1, 8, 1, 1537, False),
    (1, 4, 4, 2048, False),
    (3, 32, 8, 600, True),    # more units than pairs: several units per persistent pair
]


@pytest.mark.parametrize("B,Hq,Hkv,N,causal", SMALL)
def test_pair_forward_matches_oracle(attn, B, Hq, Hkv, N, causal):
    dev = torch.device("cuda")
    d = 128
    q, k, v = prefill_inputs(1, B, Hq, Hkv, N, d, dev)
    o, lse = _run(attn, q, k, v, causal)
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), scale_of(d), causal)
    assert_close(to64(o), o_ref, to64(lse), lse_ref, what=f"pair {(B, Hq, Hkv, N, causal)}")


@pytest.mark.parametrize("causal", [False, True])
def test_pair_tile_orders_are_bit_identical_and_correct(attn, causal):
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 1, 64, 8, 2048 + 77, 128
    q, k, v = prefill_inputs(2, B, Hq, Hkv, N, d, dev)
    outs = [_run(attn, q, k, v, causal, order=o) for o in (0, 1, 2, 3)]
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])
    o, lse = outs[0]
    for h in sample_heads(Hq, Hkv):
        g = h // (Hq // Hkv)
        rows = sample_rows(N)
        o_ref, l_ref = oracle.attention_rows(to64(q[0, h, rows]), to64(k[0, g]), to64(v[0, g]), scale_of(d),
                                             causal, rows)
        assert_close(to64(o[0, h, rows]), o_ref, to64(lse[0, h, rows]), l_ref, what=f"head {h}")


@pytest.mark.parametrize("causal", [False, True])
def test_pair_agrees_with_the_single_cta_scheme(attn, causal):
    """Both schemes compute every S and O element with the same K=16 steps in
    the same order; they agree within the forward tolerance, and the test
    records whether they agree bit for bit."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 2, 16, 4, 1500, 128
    q, k, v = prefill_inputs(5, B, Hq, Hkv, N, d, dev)
    o1, l1 = _run(attn, q, k, v, causal, scheme=attn.FWD_SINGLE_CTA)
    o2, l2 = _run(attn, q, k, v, causal, scheme=attn.FWD_CTA_PAIR)
    assert_close(to64(o2), to64(o1), to64(l2), to64(l1), what="pair vs single")
    same = torch.equal(o1, o2) and torch.equal(l1, l2)
    print(f"pair vs single bit-identical: {same}")


def test_pair_and_single_launches_on_two_streams(attn):
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 1, 32, 8, 3000, 128
    q, k, v = prefill_inputs(6, B, Hq, Hkv, N, d, dev)
    ref_p = _run(attn, q, k, v, True, scheme=attn.FWD_CTA_PAIR)
    ref_s = _run(attn, q, k, v, True, scheme=attn.FWD_SINGLE_CTA)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            a = attn.forward(q, k, v, causal=True, tile_order=attn.FWD_CTA_PAIR, stream=s1)
        with torch.cuda.stream(s2):
            b = attn.forward(q, k, v, causal=True, tile_order=attn.FWD_SINGLE_CTA, stream=s2)
        outs.append((a, b))
    torch.cuda.synchronize()
    attn.check(attn.attn_device_status(), "device status")
    for a, b in outs:
        assert torch.equal(a[0], ref_p[0]) and torch.equal(a[1], ref_p[1])
        assert torch.equal(b[0], ref_s[0]) and torch.equal(b[1], ref_s[1])


def test_pair_timeout_is_reported_and_recovered(attn):
    """A zero wait limit makes the pair give up at its first incomplete wait:
    both CTAs leave, the status reads ATTN_ERR_TIMEOUT once, and the next
    launch runs normally."""
    dev = torch.device("cuda")
    q, k, v = prefill_inputs(90, 1, 8, 2, 1000, 128, dev)
    old = attn.attn_set_wait_timeout_ns(0)
    try:
        attn.forward(q, k, v, causal=True, tile_order=attn.FWD_CTA_PAIR)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == attn.ATTN_ERR_TIMEOUT
    finally:
        attn.attn_set_wait_timeout_ns(old)
    assert attn.attn_device_status() == attn.ATTN_OK
    o, lse = _run(attn, q, k, v, True)
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), scale_of(128), True)
    assert_close(to64(o), o_ref, to64(lse), lse_ref, what="after a timeout")


@pytest.mark.parametrize("B,Hq,Hkv,N,causal", [(1, 128, 128, 32768, False), (1, 64, 8, 131072, True)])
def test_pair_full_size_equals_the_single_cta_scheme(attn, B, Hq, Hkv, N, causal):
    """Sizes the forward sweep times with the pair scheme: bit for bit the
    one-CTA result (the same K = 16 steps in the same order), and sampled rows
    of sampled heads against the oracle."""
    import gc
    dev = torch.device("cuda")
    d = 128
    q, k, v = prefill_inputs(12, B, Hq, Hkv, N, d, dev)
    try:
        o1, l1 = _run(attn, q, k, v, causal, scheme=attn.FWD_SINGLE_CTA)
        o2, l2 = _run(attn, q, k, v, causal, scheme=attn.FWD_CTA_PAIR)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        rows = sample_rows(N)
        for h in sample_heads(Hq, Hkv):
            g = h // (Hq // Hkv)
            o_ref, l_ref = oracle.attention_rows(to64(q[0, h, rows]), to64(k[0, g]), to64(v[0, g]), scale_of(d),
                                                 causal, rows)
            assert_close(to64(o2[0, h, rows]), o_ref, to64(l2[0, h, rows]), l_ref, what=f"pair N={N} head {h}")
    finally:
        del q, k, v
        gc.collect()
        torch.cuda.empty_cache()
