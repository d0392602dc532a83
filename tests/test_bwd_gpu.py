"""GPU parity of the backward pass against the fp64 oracle, through the C ABI.

The kernels take the GPU forward pass's own output and log-sum-exp (as a
training step would) and the oracle computes the exact gradient from the same
bf16 q, k, v, dO.  Small shapes are compared element by element (several
blocks, ragged tails, N = 1, GQA, causal, d = 56/64/128); a larger shape and
the backward sweep's full sizes on sampled rows and through identities of the
softmax Jacobian.  Structural
identities are checked bit for bit: the three tile orders, and d = 56
against explicit zero padding to 64."""
import gc

import numpy as np
import pytest
import torch

import oracle
from synthetic_inputs import output_grad, prefill_inputs, sample_heads, sample_rows
from tests.gpu_util import scale_of, to64

pytestmark = pytest.mark.gpu

# Gradient tolerance.  Against the exact gradient the kernels round P and dS
# to bf16 before their products (relative 2^-9 each), use the forward's bf16 O
# in Delta = rowsum(dO * O) and round the results to bf16; over the sums
# these stay near 2^-8 of the gradient's size.  The bar: relative L2 error
# per tensor <= 1e-2 and every element within 3e-2 of the tensor's largest
# magnitude, both with an absolute floor of 1e-3 per element (below bf16's
# resolution for values near 1).  The floor covers gradients that are exactly
# zero in exact arithmetic (a single attended key gives dq = dk = 0), where
# the kernel returns rounding noise: Delta uses the forward's bf16 O, so
# dP - Delta is zero only up to rounding.
REL_L2 = 1e-2
MAX_REL = 3e-2
FLOOR = 1e-3


def assert_grad_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    scale = max(np.max(np.abs(ref)), FLOOR)
    err = np.abs(got - ref)
    rel_l2 = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), FLOOR * np.sqrt(ref.size))
    assert rel_l2 <= REL_L2, f"{what}: relative L2 error {rel_l2:.3e}"
    assert np.max(err) <= MAX_REL * scale, f"{what}: max error {np.max(err):.3e} (scale {scale:.3e})"


@pytest.fixture(scope="module")
def attn():
    from attention_fa2_fwd_sm_gb300 import _build
    _build.build()
    import attention_fa2_fwd_sm_gb300 as A
    A.lib()
    oracle.build()
    return A


def _fwd_bwd(A, q, k, v, dout, causal, order=0, scale=None):
    d = q.shape[-1]
    scale = scale_of(d) if scale is None else scale
    o, lse = A.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = A.backward(q, k, v, o, lse, dout, causal=causal, scale=scale, tile_order=order)
    torch.cuda.synchronize()
    assert A.attn_device_status() == A.ATTN_OK
    return dq, dk, dv


SMALL = [  # B, Hq, Hkv, N, d, causal
    (1, 2, 2, 128, 64, False),
    (1, 2, 2, 300, 128, True),
    (2, 4, 2, 257, 64, True),
    (1, 3, 1, 1, 128, False),
    (1, 2, 2, 200, 56, True),
    (1, 4, 4, 640, 128, False),
    (1, 16, 16, 1024, 64, True),    # more units than SMs in both passes
    (1, 16, 2, 1100, 128, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", SMALL)
def test_small_shapes_match_the_oracle(attn, B, Hq, Hkv, N, d, causal):
    dev = torch.device("cuda")
    q, k, v = prefill_inputs(21, B, Hq, Hkv, N, d, dev)
    dout = output_grad(21, B, Hq, N, d, dev)
    dq, dk, dv = _fwd_bwd(attn, q, k, v, dout, causal)
    rq, rk, rv = oracle.attention_bwd(to64(q), to64(k), to64(v), to64(dout), scale_of(d), causal)
    what = f"{(B, Hq, Hkv, N, d, causal)}"
    assert_grad_close(to64(dq), rq, "dq " + what)
    assert_grad_close(to64(dk), rk, "dk " + what)
    assert_grad_close(to64(dv), rv, "dv " + what)


@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(1, 8, 2, 700, 128), (2, 16, 2, 300, 64), (1, 6, 2, 257, 56)])
def test_query_head_split_of_the_dkdv_pass(attn, B, Hq, Hkv, N, d):
    """Non-causal grouped-query problems with few dK/dV units split each KV
    head's query heads when the workspace holds the partials (causal ones
    never do): the split and the unsplit
    pass (the minimum workspace) both match the oracle, agree within fp32
    rounding on dK and dV, and give the same dQ bit for bit."""
    dev = torch.device("cuda")
    causal = False
    q, k, v = prefill_inputs(24, B, Hq, Hkv, N, d, dev)
    dout = output_grad(24, B, Hq, N, d, dev)
    scale = scale_of(d)
    o, lse = attn.forward(q, k, v, causal=causal, scale=scale)
    base = attn.attn_bwd_workspace_bytes(B, Hq, N)
    ex = attn.attn_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, causal)
    assert ex > base, "this shape is split"
    assert attn.attn_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, True) == base, "causal never splits"
    rq, rk, rv = oracle.attention_bwd(to64(q), to64(k), to64(v), to64(dout), scale, causal)
    got = {}
    for name, nbytes in (("split", ex), ("unsplit", base)):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        grads = attn.backward(q, k, v, o, lse, dout, causal=causal, scale=scale, workspace=ws)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == attn.ATTN_OK
        what = f"{name} {(B, Hq, Hkv, N, d, causal)}"
        for g, r, nm in zip(grads, (rq, rk, rv), ("dq", "dk", "dv")):
            assert_grad_close(to64(g), r, nm + " " + what)
        got[name] = grads
    assert torch.equal(got["split"][0], got["unsplit"][0]), "dQ does not depend on the dK/dV split"
    for a, b in zip(got["split"][1:], got["unsplit"][1:]):
        diff = (a.float() - b.float()).abs().max().item()
        assert diff <= 2e-2 * max(b.float().abs().max().item(), 1e-3), diff


@pytest.mark.parametrize("scale", [1.0, 0.02])
@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_other_scales_match_the_oracle(attn, scale, d, causal):
    """Scales far from 1/sqrt(d): peaked rows (1.0) and nearly uniform ones (0.02)."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N = 1, 4, 2, 300
    q, k, v = prefill_inputs(23, B, Hq, Hkv, N, d, dev)
    dout = output_grad(23, B, Hq, N, d, dev)
    dq, dk, dv = _fwd_bwd(attn, q, k, v, dout, causal, scale=scale)
    rq, rk, rv = oracle.attention_bwd(to64(q), to64(k), to64(v), to64(dout), scale, causal)
    what = f"scale {scale}, d {d}, causal {causal}"
    assert_grad_close(to64(dq), rq, "dq " + what)
    assert_grad_close(to64(dk), rk, "dk " + what)
    assert_grad_close(to64(dv), rv, "dv " + what)


@pytest.mark.parametrize("causal", [False, True])
def test_tile_orders_are_bit_identical(attn, causal):
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 1, 32, 8, 1500, 128
    q, k, v = prefill_inputs(22, B, Hq, Hkv, N, d, dev)
    dout = output_grad(22, B, Hq, N, d, dev)
    ref = _fwd_bwd(attn, q, k, v, dout, causal, order=0)
    for order in (1, 2):
        got = _fwd_bwd(attn, q, k, v, dout, causal, order=order)
        for a, b in zip(got, ref):
            assert torch.equal(a, b), f"order {order}"


@pytest.mark.parametrize("N", [16384, 16385])
def test_causal_gqa_dq_order_on_both_sides_of_the_whole_entry_rule(attn, N):
    """The dQ pass takes the forward's 256-row units: 8 KV heads of 64 such
    blocks (16384 keys) fit in L2 together and run the block-first sequence
    under head-first; one more key keeps the ACC-by-ACC order.  Every order
    gives the same gradients bit for bit, and dQ matches the oracle on
    sampled rows of sampled heads."""
    dev = torch.device("cuda")
    B, Hq, Hkv, d = 1, 16, 8, 64
    G = Hq // Hkv
    q, k, v = prefill_inputs(27, B, Hq, Hkv, N, d, dev)
    dout = output_grad(27, B, Hq, N, d, dev)
    got = _fwd_bwd(attn, q, k, v, dout, True, order=0)
    for order in (1, 2):
        other = _fwd_bwd(attn, q, k, v, dout, True, order=order)
        for a, b in zip(other, got):
            assert torch.equal(a, b), f"order {order}"
    rows = sample_rows(N)
    for h in sample_heads(Hq, Hkv):
        g = h // G
        rq, _, _ = oracle.attention_bwd_head(to64(q[0, h, rows]), to64(k[0, g]), to64(v[0, g]),
                                             to64(dout[0, h, rows]), scale_of(d), True, qpos=rows)
        assert_grad_close(to64(got[0][0, h, rows]), rq, f"dq N={N} head {h}")


def test_causal_dkdv_windows_with_a_partial_last_window(attn):
    """Causal head-first dK/dV runs windows of (batch, KV head) pairs longest
    first, sized to cover the SMs three times.  Seven KV heads with windows of
    five leave a partial last window.  Every order computes each block the
    same way, so the gradients equal block-first's bit for bit, and dV of each
    KV head sums to the group's dO."""
    dev = torch.device("cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nblk = -(-3 * sms // 5)
    assert -(-3 * sms // nblk) == 5
    B, Hq, Hkv, N, d = 1, 14, 7, nblk * 128 - 37, 64
    G = Hq // Hkv
    q, k, v = prefill_inputs(26, B, Hq, Hkv, N, d, dev)
    dout = output_grad(26, B, Hq, N, d, dev)
    got = _fwd_bwd(attn, q, k, v, dout, True, order=0)
    ref = _fwd_bwd(attn, q, k, v, dout, True, order=1)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    dv32 = got[2].float()
    for g in range(Hkv):
        want = dout[0, g * G:(g + 1) * G].float().sum((0, 1))
        assert torch.allclose(dv32[0, g].sum(0), want, rtol=1e-2, atol=1e-2 * want.abs().max().item())


def test_concurrent_launches_of_both_head_dims(attn):
    """Backward launches of both head dimensions draw their scheduler slots
    from one sequence, so launches running at once on two streams never share
    a slot: every gradient equals that of a launch run alone."""
    dev = torch.device("cuda")
    B, H, N = 1, 4, 1024
    data = {}
    for d in (64, 128):
        q, k, v = prefill_inputs(60 + d, B, H, H, N, d, dev)
        dout = output_grad(60 + d, B, H, N, d, dev)
        o, lse = attn.forward(q, k, v, causal=True)
        data[d] = (q, k, v, o, lse, dout)
    ref = {d: attn.backward(*data[d], causal=True) for d in data}
    torch.cuda.synchronize()
    nbytes = {d: attn.attn_bwd_workspace_bytes_ex(B, H, H, N, d, True) for d in data}
    streams = {d: torch.cuda.Stream() for d in data}
    runs = []
    for _ in range(6):
        for d in data:
            q, k, v, o, lse, dout = data[d]
            ws = torch.empty(nbytes[d], dtype=torch.uint8, device=dev)
            grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
            attn.check(attn.attn_bwd(q, k, v, o, dout, lse, *grads, B, H, H, N, d, d ** -0.5, True, 0, ws,
                                     nbytes[d], streams[d].cuda_stream), "attn_bwd")
            runs.append((d, grads, ws))
    torch.cuda.synchronize()
    attn.check(attn.attn_device_status(), "device status")
    for d, grads, _ in runs:
        for a, b in zip(grads, ref[d]):
            assert torch.equal(a, b), f"d={d}"


def test_d56_equals_zero_padding_to_64(attn):
    dev = torch.device("cuda")
    B, H, N = 1, 4, 700
    q, k, v = prefill_inputs(23, B, H, H, N, 56, dev)
    dout = output_grad(23, B, H, N, 56, dev)
    scale = scale_of(56)
    g56 = _fwd_bwd(attn, q, k, v, dout, True, scale=scale)
    pad = lambda t: torch.nn.functional.pad(t, (0, 8)).contiguous()
    g64 = _fwd_bwd(attn, pad(q), pad(k), pad(v), pad(dout), True, scale=scale)
    for a, b in zip(g56, g64):
        assert torch.equal(a, b[..., :56])
        assert torch.count_nonzero(b[..., 56:]) == 0


@pytest.mark.parametrize("causal", [False, True])
def test_larger_shape_sampled_rows_and_identities(attn, causal):
    """GQA 32/4 heads, N = 4096: dq on sampled rows of sampled heads, dk and dv
    of one KV head in full, and the Jacobian identities on every head:
    sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i per KV head."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 1, 32, 4, 4096, 128
    G = Hq // Hkv
    q, k, v = prefill_inputs(24, B, Hq, Hkv, N, d, dev)
    dout = output_grad(24, B, Hq, N, d, dev)
    dq, dk, dv = _fwd_bwd(attn, q, k, v, dout, causal)
    scale = scale_of(d)
    g = Hkv - 1
    rk = np.zeros((N, d))
    rv = np.zeros((N, d))
    rows = sample_rows(N)
    for h in range(g * G, (g + 1) * G):
        rq, rkh, rvh = oracle.attention_bwd_head(to64(q[0, h]), to64(k[0, g]), to64(v[0, g]), to64(dout[0, h]),
                                                 scale, causal)
        rk += rkh
        rv += rvh
        if h in sample_heads(Hq, Hkv) or h == g * G:
            assert_grad_close(to64(dq[0, h, rows]), rq[rows], f"dq head {h}")
    assert_grad_close(to64(dk[0, g]), rk, "dk")
    assert_grad_close(to64(dv[0, g]), rv, "dv")
    dk32, dv32 = dk.float(), dv.float()
    for gg in range(Hkv):
        norm = torch.linalg.vector_norm(dk32[0, gg]).item()
        assert torch.linalg.vector_norm(dk32[0, gg].sum(0)).item() <= 1e-2 * norm
        want = dout[0, gg * G:(gg + 1) * G].float().sum((0, 1))
        assert torch.allclose(dv32[0, gg].sum(0), want, rtol=1e-2, atol=1e-2 * want.abs().max().item())


FULL_BWD = [
    # the backward sweep's configurations: name, B, Hq, Hkv, N, d, causal
    ("mha", 1, 128, 128, 8192, 128, False),
    ("gqa", 1, 64, 8, 8192, 128, False),
    ("gqa", 1, 64, 8, 8192, 128, True),
    ("mha", 1, 128, 128, 32768, 128, False),
    ("gqa", 1, 64, 8, 32768, 128, False),
    ("gqa", 1, 64, 8, 32768, 128, True),
    ("deepseek", 1, 128, 128, 32768, 56, True),
]


@pytest.mark.parametrize("name,B,Hq,Hkv,N,d,causal", FULL_BWD)
def test_full_size_sampled(attn, name, B, Hq, Hkv, N, d, causal):
    """Full sizes, in the launch configuration the sweep times (head-first,
    the library's own workspace choice): dQ on sampled rows of sampled heads
    against the oracle (a row of dQ needs only its own query row); on every KV
    head the identities that hold at any size, sum_j dK_j = 0 and sum_j dV_j =
    the group's summed dO; at 8K one KV head's dK and dV in full."""
    dev = torch.device("cuda")
    cfg = {"mha": 31, "gqa": 32, "deepseek": 33}[name] + (4 if causal else 0)
    q, k, v = prefill_inputs(cfg, B, Hq, Hkv, N, d, dev)
    dout = output_grad(cfg, B, Hq, N, d, dev)
    scale = scale_of(d)
    G = Hq // Hkv
    try:
        dq, dk, dv = _fwd_bwd(attn, q, k, v, dout, causal)
        rows = sample_rows(N)
        for h in sample_heads(Hq, Hkv):
            g = h // G
            rq, _, _ = oracle.attention_bwd_head(to64(q[0, h, rows]), to64(k[0, g]), to64(v[0, g]),
                                                 to64(dout[0, h, rows]), scale, causal, qpos=rows)
            assert_grad_close(to64(dq[0, h, rows]), rq, f"{name} N={N} dq head {h}")
        dk32, dv32 = dk.float(), dv.float()
        for gg in range(Hkv):
            norm = torch.linalg.vector_norm(dk32[0, gg]).item()
            assert torch.linalg.vector_norm(dk32[0, gg].sum(0)).item() <= 1e-2 * norm, f"sum dK, KV head {gg}"
            want = dout[0, gg * G:(gg + 1) * G].float().sum((0, 1))
            assert torch.allclose(dv32[0, gg].sum(0), want, rtol=1e-2, atol=1e-2 * want.abs().max().item()), \
                f"sum dV, KV head {gg}"
        if N <= 8192:
            g = Hkv - 1
            rk = np.zeros((N, d))
            rv = np.zeros((N, d))
            for h in range(g * G, (g + 1) * G):
                _, rkh, rvh = oracle.attention_bwd_head(to64(q[0, h]), to64(k[0, g]), to64(v[0, g]),
                                                        to64(dout[0, h]), scale, causal)
                rk += rkh
                rv += rvh
            assert_grad_close(to64(dk[0, g]), rk, f"{name} N={N} dk")
            assert_grad_close(to64(dv[0, g]), rv, f"{name} N={N} dv")
    finally:
        del q, k, v, dout
        gc.collect()
        torch.cuda.empty_cache()


def test_single_key_gives_zero_q_and_k_gradients(attn):
    """N = 1: o = v, so dq = dk = 0 exactly (here: rounding noise far below
    the floor) and dv = dO summed over the group."""
    dev = torch.device("cuda")
    q, k, v = prefill_inputs(25, 2, 4, 2, 1, 64, dev)
    dout = output_grad(25, 2, 4, 1, 64, dev)
    dq, dk, dv = _fwd_bwd(attn, q, k, v, dout, False)
    assert dq.abs().max().item() <= FLOOR and dk.abs().max().item() <= FLOOR
    want = dout.float().view(2, 2, 2, 1, 64).sum(2)
    assert torch.allclose(dv.float(), want, rtol=1e-2, atol=1e-2)


def test_backward_argument_errors(attn):
    dev = torch.device("cuda")
    q, k, v = prefill_inputs(26, 1, 2, 2, 128, 64, dev)
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 128), dtype=torch.float32, device=dev)
    g = [torch.empty_like(t) for t in (q, k, v)]
    ws = torch.empty(attn.attn_bwd_workspace_bytes(1, 2, 128), dtype=torch.uint8, device=dev)
    call = lambda **kw: attn.attn_bwd(q, k, v, o, q, kw.get("lse", lse), *g, 1, 2, 2, 128, kw.get("d", 64),
                                      0.125, False, kw.get("order", 0), kw.get("ws", ws),
                                      kw.get("ws_bytes", ws.numel()))
    assert call(lse=None) == attn.ATTN_ERR_ARG
    assert call(order=3) == attn.ATTN_ERR_ARG
    assert call(ws_bytes=ws.numel() - 1) == attn.ATTN_ERR_WORKSPACE
    assert call(ws=None) == attn.ATTN_ERR_WORKSPACE
    assert call(d=96) == attn.ATTN_ERR_UNSUPPORTED


# The backward's passes leave cleanly when a wait gives up: with a wait limit
# of zero every role of the dK/dV and dQ kernels leaves its loop at the first
# wait that is not already satisfied (copies drained, MMAs committed, TMEM
# freed), attn_device_status reports ATTN_ERR_TIMEOUT, and the next call is
# correct.  The CTAs that gave up still reset their scheduler slot, so 65 more
# calls (every slot again) stay bit-identical.  Non-causal GQA with few units
# runs the split dK/dV pass and its reduction.
@pytest.mark.parametrize("d,causal", [(64, True), (128, True), (128, False)])
def test_backward_timeout_is_reported_and_recovered(attn, d, causal):
    dev = torch.device("cuda")
    B, Hq, Hkv, N = 1, 8, 2, 700
    q, k, v = prefill_inputs(92, B, Hq, Hkv, N, d, dev)
    dout = output_grad(92, B, Hq, N, d, dev)
    scale = scale_of(d)
    o, lse = attn.forward(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    old = attn.attn_set_wait_timeout_ns(0)
    try:
        attn.backward(q, k, v, o, lse, dout, causal=causal, scale=scale)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == attn.ATTN_ERR_TIMEOUT
    finally:
        attn.attn_set_wait_timeout_ns(old)
    assert attn.attn_device_status() == attn.ATTN_OK  # cleared by the read
    grads = attn.backward(q, k, v, o, lse, dout, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    refs = oracle.attention_bwd(to64(q), to64(k), to64(v), to64(dout), scale, causal)
    for got, ref, name in zip(grads, refs, ("dq", "dk", "dv")):
        assert_grad_close(to64(got), ref, f"{name} after timeout")
    for i in range(65):
        again = attn.backward(q, k, v, o, lse, dout, causal=causal, scale=scale)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(again, grads)), f"call {i}"
    assert attn.attn_device_status() == attn.ATTN_OK
