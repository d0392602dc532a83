"""GPU checks of attn_fwd_host, the forward on host-resident tensors whose
copies and kernels overlap in chunks of KV heads: its outputs are bit for bit
those of attn_fwd_ex on device copies of the same inputs (every chunk is an
independent forward problem), for several chunk sizes including a ragged last
chunk, pinned and pageable host memory, GQA, causal and d = 56; and they match
the fp64 oracle."""
import pytest
import torch

import oracle
from synthetic_inputs import prefill_inputs
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


def _host(t, pinned):
    h = t.cpu()
    return h.pin_memory() if pinned else h.clone()


CASES = [
    # B, Hq, Hkv, N, d, causal, kv heads per chunk, pinned
    (2, 8, 2, 300, 128, True, 0, True),
    (2, 8, 2, 300, 128, True, 1, True),
    (2, 8, 2, 300, 128, False, 2, False),
    (1, 6, 6, 1000, 64, False, 4, True),   # chunks of 4 and 2 KV heads
    (1, 6, 6, 1000, 64, True, 5, False),
    (1, 4, 4, 513, 56, True, 3, True),
    (3, 4, 1, 129, 128, False, 0, True),   # one KV head per batch entry: one chunk each
    (1, 2, 2, 1, 64, False, 1, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,chunk,pinned", CASES)
def test_host_forward_is_bit_identical_to_the_device_call(attn, B, Hq, Hkv, N, d, causal, chunk, pinned):
    dev = torch.device("cuda")
    q, k, v = prefill_inputs(3, B, Hq, Hkv, N, d, dev)
    scale = scale_of(d)
    o_dev, lse_dev = attn.forward(q, k, v, causal=causal, scale=scale)
    hq, hk, hv = (_host(t, pinned) for t in (q, k, v))
    o_h = torch.full(q.shape, float("nan"), dtype=q.dtype)
    lse_h = torch.full((B, Hq, N), float("nan"), dtype=torch.float32)
    if pinned:
        o_h, lse_h = o_h.pin_memory(), lse_h.pin_memory()
    o, lse = attn.forward_host(hq, hk, hv, causal=causal, scale=scale, kv_heads_per_chunk=chunk,
                               out=(o_h, lse_h))
    attn.check(attn.attn_device_status(), "device status")
    assert torch.equal(o.view(torch.int16), o_dev.cpu().view(torch.int16))
    assert torch.equal(lse, lse_dev.cpu())


def test_host_forward_matches_the_oracle_and_repeats(attn):
    """Two calls in a row on one workspace with different inputs, the second
    without lse: each result against the oracle."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 1, 8, 2, 700, 128
    scale = scale_of(d)
    ws = torch.empty(attn.attn_fwd_host_workspace_bytes(B, Hq, Hkv, N, d, 1), dtype=torch.uint8, device=dev)
    for seed, causal, with_lse in ((5, True, True), (6, False, False)):
        q, k, v = (t.cpu().pin_memory() for t in prefill_inputs(seed, B, Hq, Hkv, N, d, dev))
        o, lse = attn.forward_host(q, k, v, causal=causal, scale=scale, with_lse=with_lse,
                                   kv_heads_per_chunk=1, workspace=ws)
        attn.check(attn.attn_device_status(), "device status")
        o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), scale, causal)
        if with_lse:
            assert_close(to64(o), o_ref, to64(lse), lse_ref, what=f"seed {seed}")
        else:
            assert lse is None
            assert_close(to64(o), o_ref, what=f"seed {seed}")


def test_host_forward_is_ordered_on_the_callers_stream(attn):
    """Work enqueued on the stream after the call sees the copied-back output,
    and the call waits for work enqueued before it."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 1, 4, 4, 512, 64
    scale = scale_of(d)
    q, k, v = prefill_inputs(8, B, Hq, Hkv, N, d, dev)
    o_ref, _ = attn.forward(q, k, v, causal=False, scale=scale)
    s = torch.cuda.Stream()
    hq, hk, hv = (torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(3))
    o_h = torch.zeros(q.shape, dtype=q.dtype, pin_memory=True)
    back = torch.empty_like(q)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        # fill the host inputs from the device on the same stream, then run
        for src, dst in ((q, hq), (k, hk), (v, hv)):
            dst.copy_(src, non_blocking=True)
        attn.forward_host(hq, hk, hv, scale=scale, with_lse=False, kv_heads_per_chunk=1, out=(o_h, None),
                          stream=s, synchronize=False)
        back.copy_(o_h, non_blocking=True)
    s.synchronize()
    attn.check(attn.attn_device_status(), "device status")
    assert torch.equal(back.view(torch.int16), o_ref.view(torch.int16))


def test_host_buffers_need_no_alignment(attn):
    """Host tensors may start anywhere (here 2 bytes past a 16-byte boundary):
    only the device workspace has an alignment rule."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 1, 4, 2, 333, 64
    q, k, v = prefill_inputs(9, B, Hq, Hkv, N, d, dev)
    o_dev, lse_dev = attn.forward(q, k, v, causal=True, scale=scale_of(d))

    def odd(t):
        flat = torch.empty(t.numel() + 1, dtype=t.dtype, pin_memory=True)
        view = flat[1:].view(t.shape)
        view.copy_(t.cpu())
        return view

    hq, hk, hv = odd(q), odd(k), odd(v)
    o_h, lse_h = odd(torch.zeros_like(q)), torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=True)
    assert hq.data_ptr() % 16 == 2 and o_h.data_ptr() % 16 == 2
    attn.forward_host(hq, hk, hv, causal=True, scale=scale_of(d), kv_heads_per_chunk=1, out=(o_h, lse_h))
    attn.check(attn.attn_device_status(), "device status")
    assert torch.equal(o_h.view(torch.int16), o_dev.cpu().view(torch.int16))
    assert torch.equal(lse_h, lse_dev.cpu())


def test_traced_call_records_an_ordered_timeline(attn):
    """With tracing on, a call records per chunk (copy-in done, kernel
    reached, kernel done, copy-out done); each chunk's times are ordered that
    way, the chunks follow the call's chunk order, and the traced call's
    outputs are those of an untraced one."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 2, 8, 4, 700, 128
    q, k, v = prefill_inputs(4, B, Hq, Hkv, N, d, dev)
    hq, hk, hv = (_host(t, True) for t in (q, k, v))
    o0, lse0 = attn.forward_host(hq, hk, hv, kv_heads_per_chunk=1)
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_host_trace_read()  # nothing traced yet
    attn.check(attn.attn_fwd_host_trace(1), "trace on")
    try:
        o1, lse1 = attn.forward_host(hq, hk, hv, kv_heads_per_chunk=1)
        tl = attn.attn_fwd_host_trace_read()
    finally:
        attn.check(attn.attn_fwd_host_trace(0), "trace off")
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)) and torch.equal(lse0, lse1)
    assert len(tl) == B * Hkv
    # Each mark is recorded on its stream before the event that other streams
    # wait on, so the order holds exactly.
    for c, (cin, kin, kout, cout) in enumerate(tl):
        assert 0.0 <= cin <= kin <= kout <= cout, (c, tl[c])
        if c >= 2:  # a slot is refilled only after the chunk two back has left it
            assert cin >= tl[c - 2][2], (c, tl[c], tl[c - 2])
    assert len(attn.attn_fwd_host_trace_read(capacity=3)) == 3


def test_host_forward_with_the_pair_scheme(attn):
    """The tile-scheme flag reaches the chunks' kernels: attn_fwd_host with
    ATTN_FWD_CTA_PAIR gives the device call's result bit for bit."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 1, 8, 4, 900, 128
    q, k, v = prefill_inputs(12, B, Hq, Hkv, N, d, dev)
    o_dev, lse_dev = attn.forward(q, k, v, causal=True, tile_order=attn.FWD_CTA_PAIR)
    hq, hk, hv = (_host(t, True) for t in (q, k, v))
    o, lse = attn.forward_host(hq, hk, hv, causal=True, tile_order=attn.FWD_CTA_PAIR, kv_heads_per_chunk=1)
    attn.check(attn.attn_device_status(), "device status")
    assert torch.equal(o.view(torch.int16), o_dev.cpu().view(torch.int16))
    assert torch.equal(lse, lse_dev.cpu())


def test_host_forward_at_the_bench_size_is_bit_identical(attn):
    """The end-to-end call the benchmark times: MHA B=1, H=128, N=131072,
    d=128, non-causal, head-first, pinned host buffers and the library's
    default chunking.  Its outputs equal attn_fwd's on the same inputs bit for
    bit (the device result is itself compared with the oracle at this size in
    the forward tests)."""
    dev = torch.device("cuda")
    B, H, N, d = 1, 128, 131072, 128
    scale = scale_of(d)

    def pinned(t):
        return torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)

    q, k, v = prefill_inputs(11, B, H, H, N, d, dev)
    o_dev, lse_dev = attn.forward(q, k, v, causal=False, scale=scale)
    attn.check(attn.attn_device_status(), "device status")
    hq, hk, hv = pinned(q), pinned(k), pinned(v)
    o_ref, lse_ref = pinned(o_dev), pinned(lse_dev)
    del q, k, v, o_dev, lse_dev
    torch.cuda.empty_cache()
    try:
        o, lse = attn.forward_host(hq, hk, hv, causal=False, scale=scale, kv_heads_per_chunk=0)
        attn.check(attn.attn_device_status(), "device status")
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse, lse_ref)
    finally:
        del hq, hk, hv, o_ref, lse_ref
        torch.cuda.empty_cache()
