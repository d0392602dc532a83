"""Pins of the backward oracle (gradients of attention), CPU only.

The gradient has a plain definition (the chain rule of the forward
definition), so the pins are things the mathematics fixes, independent of
the oracle's own code: central finite differences of the oracle's forward
(itself pinned), autograd of PyTorch's fp64 CPU attention (a library
routine), and identities of the softmax Jacobian."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _rand(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def _loss(q, k, v, dout, scale, causal):
    o, _ = oracle.attention_head(q, k, v, scale, causal)
    return float(np.sum(o * dout))


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_differences(causal):
    nq, nk, d, scale = 6, 6, 5, 0.7
    q, k, v, dout = _rand(1, nq, d), _rand(2, nk, d), _rand(3, nk, d), _rand(4, nq, d)
    dq, dk, dv = oracle.attention_bwd_head(q, k, v, dout, scale, causal)
    h = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            lp = _loss(**{**args, name: xp}, dout=dout, scale=scale, causal=causal)
            lm = _loss(**{**args, name: xm}, dout=dout, scale=scale, causal=causal)
            num[idx] = (lp - lm) / (2 * h)
        assert np.max(np.abs(num - g)) <= 1e-8 * max(1.0, np.max(np.abs(g))), name


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (6, 1)])
def test_gradients_match_autograd_of_library_attention(causal, hq, hkv):
    B, N, d, scale = 2, 11, 8, 0.35
    g = torch.Generator().manual_seed(7)
    q = torch.randn(B, hq, N, d, generator=g, dtype=torch.float64, requires_grad=True)
    k = torch.randn(B, hkv, N, d, generator=g, dtype=torch.float64, requires_grad=True)
    v = torch.randn(B, hkv, N, d, generator=g, dtype=torch.float64, requires_grad=True)
    dout = torch.randn(B, hq, N, d, generator=g, dtype=torch.float64)
    o = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale, enable_gqa=hq != hkv)
    o.backward(dout)
    dq, dk, dv = oracle.attention_bwd(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(),
                                      dout.numpy(), scale, causal)
    for mine, ref in ((dq, q.grad), (dk, k.grad), (dv, v.grad)):
        np.testing.assert_allclose(mine, ref.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_jacobian_identities(causal):
    """Each row's ds sums to zero over its keys, so the key gradients sum to
    zero; each row's probabilities sum to one, so the value gradients sum to
    the sum of the output gradients."""
    nq = nk = 40
    d = 16
    q, k, v, dout = _rand(5, nq, d), _rand(6, nk, d), _rand(7, nk, d), _rand(8, nq, d)
    dq, dk, dv = oracle.attention_bwd_head(q, k, v, dout, 0.25, causal)
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(0), dout.sum(0), rtol=1e-12, atol=1e-12)
    # shifting every key by one vector leaves the output, hence dq, unchanged
    dq2, _, _ = oracle.attention_bwd_head(q, k + _rand(9, 1, d), v, dout, 0.25, causal)
    np.testing.assert_allclose(dq2, dq, rtol=1e-9, atol=1e-11)


def test_single_key_and_first_causal_row():
    """One key: o = v regardless of q and k, so dq = dk = 0 and dv = sum dO.
    The first causal row sees only key 0, so its dq is 0."""
    q, k, v, dout = _rand(10, 3, 4), _rand(11, 1, 4), _rand(12, 1, 4), _rand(13, 3, 4)
    dq, dk, dv = oracle.attention_bwd_head(q, k, v, dout, 1.0)
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_allclose(dv[0], dout.sum(0), rtol=1e-14)
    q, k, v, dout = _rand(14, 5, 4), _rand(15, 5, 4), _rand(16, 5, 4), _rand(17, 5, 4)
    dq, _, _ = oracle.attention_bwd_head(q, k, v, dout, 1.0, causal=True)
    assert np.all(dq[0] == 0) and np.any(dq[1] != 0)


def test_two_key_closed_form():
    """Two keys with scores 0 and log 3 (p = 1/4, 3/4), q = e_0, k_1 = log3 e_0:
    dp = <dO, v_j>, D = sum p dp, ds = p (dp - D), dq = ds_1 * k_1 (scale 1)."""
    q = np.array([[1.0, 0.0]])
    k = np.array([[0.0, 0.0], [math.log(3), 0.0]])
    v = np.array([[1.0, 2.0], [5.0, -2.0]])
    dout = np.array([[1.0, 1.0]])
    dq, dk, dv = oracle.attention_bwd_head(q, k, v, dout, 1.0)
    # dp = (3, 3): equal, so ds = 0 and every q/k gradient vanishes
    assert np.allclose(dq, 0) and np.allclose(dk, 0)
    np.testing.assert_allclose(dv, [[0.25, 0.25], [0.75, 0.75]], rtol=1e-14)
    dout = np.array([[1.0, 0.0]])  # dp = (1, 5), D = 4, ds = (1/4 * -3, 3/4 * 1) = (-0.75, 0.75)
    dq, dk, dv = oracle.attention_bwd_head(q, k, v, dout, 1.0)
    np.testing.assert_allclose(dq, [[0.75 * math.log(3), 0.0]], rtol=1e-13)
    np.testing.assert_allclose(dk, [[-0.75, 0.0], [0.75, 0.0]], rtol=1e-13)
