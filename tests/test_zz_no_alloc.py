"""attn_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers may not call cudaMalloc or own a workspace buffer -- a plug-in
inside a framework whose memory pool has reserved the whole GPU, a serving
loop that cannot afford an allocation on its critical path, or code whose
own interface cannot pass a workspace through.  For them the library keeps
the split partials in a scratch array built into the library itself.

These tests call that entry point through the C ABI and compare its output
with attn_decode's (which uses a caller-owned workspace) and with the fp64
oracle, within the parity tolerance of the other GPU tests, on two calls in
a row with different inputs, shapes and split counts, so the second call
also shows that what the first one left in the shared scratch does not leak
into it.  This file is collected last on purpose."""
import pytest
import torch

import oracle
from synthetic_inputs import decode_inputs
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


def _noalloc(A, q, kc, vc, seqlens, splits):
    B, Hq, d = q.shape
    Hkv, s_max = kc.shape[1], kc.shape[2]
    o = torch.full_like(q, float("nan"))
    A.check(A.attn_decode_noalloc(q, kc, vc, seqlens, o, B, Hq, Hkv, d, scale_of(d), splits, s_max),
            "attn_decode_noalloc")
    return o


def test_noalloc_matches_attn_decode_on_two_calls_in_a_row(attn):
    dev = torch.device("cuda")
    cases = [
        # (cfg, B, Hq, Hkv, S, d, seqlens, splits)
        (80, 4, 64, 8, 3000, 128, [3000, 1234, 0, 65], 0),  # split count chosen by the library
        (81, 2, 32, 4, 2000, 64, [17, 2000], 7),           # explicit split count, other shape
    ]
    for cfg, B, Hq, Hkv, S, d, lens, splits in cases:
        q, kc, vc = decode_inputs(cfg, B, Hq, Hkv, S, d, dev)
        seqlens = torch.tensor(lens, dtype=torch.int32, device=dev)
        o_ref, _, _ = attn.decode(q, kc, vc, seqlens, num_splits=splits)
        o = _noalloc(attn, q, kc, vc, seqlens, splits)
        torch.cuda.synchronize()
        attn.check(attn.attn_device_status(), "device status")
        assert_close(to64(o), to64(o_ref), what=f"noalloc vs attn_decode (case {cfg})")
        o_oracle, _ = oracle.decode(to64(q), to64(kc), to64(vc), lens, scale_of(d))
        assert_close(to64(o), o_oracle, what=f"noalloc vs the oracle (case {cfg})")


def test_noalloc_refuses_split_counts_beyond_its_scratch(attn):
    dev = torch.device("cuda")
    B, Hq, Hkv, S, d = 32, 64, 8, 4096, 128
    assert attn.attn_decode_workspace_bytes(B, Hq, d, 64) > attn.DECODE_NOALLOC_SCRATCH_BYTES
    q, kc, vc = decode_inputs(82, B, Hq, Hkv, S, d, dev)
    seqlens = torch.full((B,), S, dtype=torch.int32, device=dev)
    o = torch.zeros_like(q)
    rc = attn.attn_decode_noalloc(q, kc, vc, seqlens, o, B, Hq, Hkv, d, scale_of(d), 64, S)
    assert rc == attn.ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0  # nothing was queued
    # with num_splits <= 0 it lowers the split count until the partials fit
    o2 = _noalloc(attn, q, kc, vc, seqlens, 0)
    o_ref, _, _ = attn.decode(q, kc, vc, seqlens, num_splits=1)
    torch.cuda.synchronize()
    assert_close(to64(o2), to64(o_ref), what="noalloc with a lowered split count")


def _heuristic_splits(sms, B, Hkv, S):
    """attn_decode_num_splits's rule as its header states it."""
    ctas = B * Hkv
    s = max(1, min((5 * sms // 3 + ctas // 2) // ctas, S // 512, 256))
    while 2 * s <= 256 and S // (2 * s) >= 4096 and ctas * 2 * s <= 4 * sms:
        s *= 2
    return s


def test_noalloc_lowers_the_heuristic_split_count_to_fit_its_scratch(attn):
    """A shape whose heuristic split count needs more partial storage than the
    built-in scratch holds (group of 16 query heads on 5 KV heads, 816K cached
    keys: 102 splits on a 152-SM GPU, 4.2 MB of partials): with num_splits <= 0
    the call lowers the count one at a time until the partials fit, and its
    output is attn_decode's at that count bit for bit, and the oracle's within
    the parity tolerance."""
    dev = torch.device("cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, Hq, Hkv, S, d = 1, 80, 5, 835584, 128
    cap = attn.DECODE_NOALLOC_SCRATCH_BYTES
    raw = _heuristic_splits(sms, B, Hkv, S)
    assert raw == attn.attn_decode_num_splits(B, Hq, Hkv, S)
    want = raw
    while want > 1 and attn.attn_decode_workspace_bytes(B, Hq, d, want) > cap:
        want -= 1
    if sms == 152:
        assert attn.attn_decode_workspace_bytes(B, Hq, d, raw) > cap and want == raw - 1
    assert attn.attn_decode_workspace_bytes(B, Hq, d, want) <= cap
    q, kc, vc = decode_inputs(83, B, Hq, Hkv, S, d, dev)
    seqlens = torch.full((B,), S, dtype=torch.int32, device=dev)
    try:
        o = _noalloc(attn, q, kc, vc, seqlens, 0)
        o_ref, _, used = attn.decode(q, kc, vc, seqlens, num_splits=want)
        torch.cuda.synchronize()
        attn.check(attn.attn_device_status(), "device status")
        assert used == want
        assert torch.equal(o, o_ref), "noalloc with the lowered count differs from attn_decode at that count"
        q64 = to64(q)
        G = Hq // Hkv
        for g in range(Hkv):
            o_or, _ = oracle.decode(q64[:, g * G:(g + 1) * G], kc[:, g:g + 1].double().cpu().numpy(),
                                    vc[:, g:g + 1].double().cpu().numpy(), [S], scale_of(d))
            assert_close(to64(o[:, g * G:(g + 1) * G]), o_or, what=f"lowered split count {want}, KV head {g}")
    finally:
        del q, kc, vc
        torch.cuda.empty_cache()
