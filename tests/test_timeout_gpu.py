"""The bounded device waits: with a wait limit of zero every wait that is not
already satisfied runs out, the kernel leaves cleanly (copies drained, TMEM
freed), attn_device_status reports ATTN_ERR_TIMEOUT, and the next call with
the normal limit is correct again.  Nothing faults, traps or hangs."""
import pytest
import torch

import oracle
from synthetic_inputs import decode_inputs, prefill_inputs
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


# Both forward instantiations (d <= 64 and d = 128): every role of a CTA leaves
# its loop once one wait gives up, and the next launch runs normally.
@pytest.mark.parametrize("d", [64, 128])
def test_forward_timeout_is_reported_and_recovered(attn, d):
    dev = torch.device("cuda")
    q, k, v = prefill_inputs(90, 1, 8, 2, 1000, d, dev)
    old = attn.attn_set_wait_timeout_ns(0)
    try:
        attn.forward(q, k, v, causal=True)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == attn.ATTN_ERR_TIMEOUT
    finally:
        attn.attn_set_wait_timeout_ns(old)
    assert attn.attn_device_status() == attn.ATTN_OK  # cleared by the read
    o, lse = attn.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    o_ref, l_ref = oracle.attention(to64(q), to64(k), to64(v), scale_of(d), True)
    assert_close(to64(o), o_ref, to64(lse), l_ref, what="after timeout")


def test_decode_timeout_is_reported_and_recovered(attn):
    dev = torch.device("cuda")
    q, kc, vc = decode_inputs(91, 2, 16, 2, 3000, 128, dev)
    seqlens = torch.tensor([3000, 1500], dtype=torch.int32, device=dev)
    old = attn.attn_set_wait_timeout_ns(0)
    try:
        attn.decode(q, kc, vc, seqlens, num_splits=3)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == attn.ATTN_ERR_TIMEOUT
    finally:
        attn.attn_set_wait_timeout_ns(old)
    o, _, _ = attn.decode(q, kc, vc, seqlens, num_splits=3)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    o_ref, _ = oracle.decode(to64(q), to64(kc), to64(vc), [3000, 1500], scale_of(128))
    assert_close(to64(o), o_ref, what="after timeout")
