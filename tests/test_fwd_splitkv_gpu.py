"""GPU parity of the split-KV forward (attn_fwd_splitkv: every head's keys in
ranges, fp32 partials per range, then the log-sum-exp merge) against the fp64
oracle, through the C ABI: small shapes element by element (several range
counts, ranges that end past N, N = 1, GQA, causal rows before a range's
start, d = 56/64/128), the workspace partials of one head against the oracle
over each key range, agreement with attn_fwd, a long causal GQA context on
sampled rows, and the bounded-wait give-up."""
import gc

import numpy as np
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


def _run(A, q, k, v, causal, splits):
    o, lse, ws = A.forward_splitkv(q, k, v, causal=causal, kv_splits=splits)
    torch.cuda.synchronize()
    A.check(A.attn_device_status(), "device status")
    return o, lse, ws


SMALL = [
    # B, Hq, Hkv, N, d, causal, kv_splits
    (1, 2, 2, 1000, 128, True, 3),
    (1, 2, 2, 1000, 64, False, 2),
    (2, 4, 2, 700, 128, True, 4),
    (1, 8, 1, 1537, 56, True, 3),
    (1, 2, 2, 300, 128, False, 8),   # 128-key ranges: 3 of them
    (1, 3, 3, 129, 64, True, 2),     # the second range holds one key
    (1, 2, 2, 1, 128, False, 4),     # one range
    (2, 16, 16, 1100, 56, True, 5),  # more units than SMs
    (1, 4, 4, 2048, 128, False, 0),  # the library's choice (one range)
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,splits", SMALL)
def test_splitkv_matches_oracle(attn, B, Hq, Hkv, N, d, causal, splits):
    dev = torch.device("cuda")
    q, k, v = prefill_inputs(8, B, Hq, Hkv, N, d, dev)
    o, lse, _ = _run(attn, q, k, v, causal, splits)
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), scale_of(d), causal)
    assert_close(to64(o), o_ref, to64(lse), lse_ref, what=f"split-KV {(B, Hq, Hkv, N, d, causal, splits)}")


@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_partials_match_the_oracle_per_key_range(attn, causal):
    """The workspace holds, per range s, O over the range normalised by its own
    sum and its lse ([ranges][B * Hq][N][d], then [ranges][B * Hq][N]); a
    causal row before a range's start attends nothing there (lse -inf)."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d, splits = 1, 2, 1, 900, 128, 3
    q, k, v = prefill_inputs(9, B, Hq, Hkv, N, d, dev)
    o, lse, ws = _run(attn, q, k, v, causal, splits)
    chunk = -(-(-(-N // splits)) // 128) * 128  # ceil(N / splits) rounded up to 128
    n_rng = -(-N // chunk)
    rows = B * Hq * N
    o_bytes = -(-(rows * n_rng * d * 4) // 256) * 256
    wsf = ws.view(torch.float32)
    po = wsf[: rows * n_rng * d].view(n_rng, B * Hq, N, d)
    pl = wsf[o_bytes // 4: o_bytes // 4 + rows * n_rng].view(n_rng, B * Hq, N)
    h = 1
    for s in range(n_rng):
        lo, hi = s * chunk, min((s + 1) * chunk, N)
        o_s, l_s = oracle.attention_head(to64(q[0, h]), to64(k[0, 0]), to64(v[0, 0]), scale_of(d), causal,
                                         k_lo=lo, k_hi=hi)
        rows_s = np.arange(N) >= lo if causal else np.ones(N, dtype=bool)
        got_l = to64(pl[s, h])[rows_s]
        assert np.abs(got_l - l_s[rows_s]).max() <= 1e-3, f"range {s}"
        assert_close(to64(po[s, h])[rows_s], o_s[rows_s], what=f"range {s} partial O")
        if causal:
            assert np.all(l_s[~rows_s] == -np.inf)


def test_splitkv_agrees_with_the_forward(attn):
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 1, 16, 4, 4096 + 77, 128
    q, k, v = prefill_inputs(10, B, Hq, Hkv, N, d, dev)
    o1, l1 = attn.forward(q, k, v, causal=True)
    for splits in (2, 5):
        o2, l2, _ = _run(attn, q, k, v, True, splits)
        assert_close(to64(o2), to64(o1), to64(l2), to64(l1), what=f"split-KV ({splits}) vs attn_fwd")


@pytest.mark.parametrize("name,Hq,Hkv,d,causal", [("gqa", 64, 8, 128, True), ("mha", 128, 128, 128, False),
                                                  ("deepseek", 128, 128, 56, True)])
def test_splitkv_long_context_sampled_rows(attn, name, Hq, Hkv, d, causal):
    """The long-context configurations the split is for and the benchmark
    times, at 128K keys (two 64K-key ranges by the library's rule at d = 128):
    GQA 64/8 causal, MHA 128 heads, and the DeepSeek-like d = 56 causal; on
    sampled rows of sampled heads."""
    dev = torch.device("cuda")
    B, N = 1, 131072
    q, k, v = prefill_inputs(11, B, Hq, Hkv, N, d, dev)
    try:
        if d == 128:
            assert attn.attn_fwd_splitkv_workspace_bytes(B, Hq, N, d, 0) == B * Hq * N * 2 * (d + 1) * 4
        o, lse, ws = _run(attn, q, k, v, causal, 0)
        del ws
        for h in sample_heads(Hq, Hkv):
            g = h // (Hq // Hkv)
            rows = sample_rows(N)
            o_ref, l_ref = oracle.attention_rows(to64(q[0, h, rows]), to64(k[0, g]), to64(v[0, g]), scale_of(d),
                                                 causal, rows)
            assert_close(to64(o[0, h, rows]), o_ref, to64(lse[0, h, rows]), l_ref, what=f"{name} 128K head {h}")
    finally:
        del q, k, v
        gc.collect()
        torch.cuda.empty_cache()


def test_splitkv_timeout_is_reported_and_recovered(attn):
    dev = torch.device("cuda")
    q, k, v = prefill_inputs(91, 1, 8, 2, 1000, 64, dev)
    old = attn.attn_set_wait_timeout_ns(0)
    try:
        attn.forward_splitkv(q, k, v, causal=True, kv_splits=3)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == attn.ATTN_ERR_TIMEOUT
    finally:
        attn.attn_set_wait_timeout_ns(old)
    assert attn.attn_device_status() == attn.ATTN_OK
    o, lse, _ = _run(attn, q, k, v, True, 3)
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), scale_of(64), True)
    assert_close(to64(o), o_ref, to64(lse), lse_ref, what="after a timeout")
