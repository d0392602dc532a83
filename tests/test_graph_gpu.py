"""CUDA-graph capture of the entry points.  A serving loop captures one step
(a prefill, a decode step, a ragged decode step, a prefill from host buffers)
once and replays it with new contents in the same buffers; every replay must give bit for bit what an
eager call on those contents gives.  The ragged decode builds its work list
on the device, so a captured step stays valid when the sequence lengths
change between replays; the forward's persistent scheduler resets its
counters at the end of every launch, so one captured launch replays any
number of times."""
import math

import pytest
import torch

from synthetic_inputs import decode_inputs, prefill_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    from attention_fa2_fwd_sm_gb300 import _build
    _build.build()
    import attention_fa2_fwd_sm_gb300 as A
    A.lib()
    return A


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _replays_match(attn, step, outs, refill, reps=3):
    """Warm up eagerly, capture `step`, then per replay: refill the inputs,
    replay, keep the outputs, run `step` eagerly on the same inputs, compare."""
    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    for rep in range(reps):
        refill(rep)
        g.replay()
        torch.cuda.synchronize()
        got = [o.clone() for o in outs]
        step()
        torch.cuda.synchronize()
        for a, b in zip(got, outs):
            assert torch.equal(_bits(a), _bits(b)), f"replay {rep} differs from the eager call"
    attn.check(attn.attn_device_status(), "device status")


@pytest.mark.parametrize("causal", [False, True])
def test_forward_replays_in_a_cuda_graph(attn, causal):
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 2, 8, 2, 1000, 128
    q, k, v = prefill_inputs(40, B, Hq, Hkv, N, d, dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    scale = 1 / math.sqrt(d)

    def step():
        attn.check(attn.attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, attn.ORDER_HEAD_FIRST),
                   "attn_fwd_ex")

    def refill(rep):
        for dst, src in zip((q, k, v), prefill_inputs(41 + rep, B, Hq, Hkv, N, d, dev)):
            dst.copy_(src)

    _replays_match(attn, step, (o, lse), refill)


def test_decode_step_replays_in_a_cuda_graph(attn):
    dev = torch.device("cuda")
    B, Hq, Hkv, S, d = 4, 64, 8, 3000, 128
    q, kc, vc = decode_inputs(50, B, Hq, Hkv, S, d, dev)
    seqlens = torch.tensor([S, 1, 1500, 2047], dtype=torch.int32, device=dev)
    splits = attn.attn_decode_num_splits(B, Hq, Hkv, S)
    wbytes = attn.attn_decode_workspace_bytes(B, Hq, d, splits)
    ws = torch.empty(max(wbytes, 16), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)

    def step():
        attn.check(attn.attn_decode(q, kc, vc, seqlens, o, B, Hq, Hkv, d, d ** -0.5, splits, S, ws, wbytes),
                   "attn_decode")

    def refill(rep):
        for dst, src in zip((q, kc, vc), decode_inputs(51 + rep, B, Hq, Hkv, S, d, dev)):
            dst.copy_(src)
        seqlens.copy_(torch.tensor([[S, 7, 0, 64], [2, S, 1000, 999], [S, S, S, 1]][rep], dtype=torch.int32))

    _replays_match(attn, step, (o,), refill)


def test_ragged_decode_step_replays_with_new_lengths(attn):
    dev = torch.device("cuda")
    B, Hq, Hkv, S, d = 6, 32, 8, 5000, 128
    q, kc, vc = decode_inputs(60, B, Hq, Hkv, S, d, dev)
    seqlens = torch.tensor([S, 0, 10, 2000, 64, 65], dtype=torch.int32, device=dev)
    nbytes = attn.attn_decode_varlen_workspace_bytes(B, Hq, Hkv, d)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)

    def step():
        attn.check(attn.attn_decode_varlen(q, kc, vc, seqlens, o, B, Hq, Hkv, d, d ** -0.5, S, ws, nbytes),
                   "attn_decode_varlen")

    lens = [[1, 1, 1, 1, 1, 1], [S, S, 0, 0, S, 4096], [0, 0, 0, 0, 0, 0]]

    def refill(rep):
        q.copy_(decode_inputs(61 + rep, B, Hq, Hkv, S, d, dev)[0])
        seqlens.copy_(torch.tensor(lens[rep], dtype=torch.int32))

    _replays_match(attn, step, (o,), refill)


def test_host_buffer_forward_replays_in_a_cuda_graph(attn):
    """attn_fwd_host forks its copy and compute streams off the capturing
    stream and joins them back, so the whole overlapped pipeline (copy-in,
    kernels, copy-out) becomes one graph that reads the pinned host inputs
    at replay time."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 1, 6, 3, 777, 64
    hq, hk, hv = (t.cpu().pin_memory() for t in prefill_inputs(70, B, Hq, Hkv, N, d, dev))
    o = torch.empty(hq.shape, dtype=hq.dtype, pin_memory=True)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=True)
    nbytes = attn.attn_fwd_host_workspace_bytes(B, Hq, Hkv, N, d, 1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def step():
        attn.check(attn.attn_fwd_host(hq, hk, hv, o, lse, B, Hq, Hkv, N, d, d ** -0.5, True,
                                      attn.ORDER_HEAD_FIRST, 1, ws, nbytes), "attn_fwd_host")

    def refill(rep):
        for dst, src in zip((hq, hk, hv), prefill_inputs(71 + rep, B, Hq, Hkv, N, d, "cpu")):
            dst.copy_(src)

    _replays_match(attn, step, (o, lse), refill)
