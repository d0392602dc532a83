"""Planted mistakes: compile mutated copies of the oracle source (on the CPU)
and check that the pins reject each one.  This shows the pins are strong
enough that a dropped term, an off-by-one, a swapped operand or a wrong sign
cannot pass unnoticed."""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "drop_scale": ("s[j - lo] = jb->scale * dot;", "s[j - lo] = dot;"),
    "causal_off_by_one": ("int64_t last = jb->qpos[i] + 1;", "int64_t last = jb->qpos[i];"),
    "values_from_keys": ("const double *vj = jb->v + j * d;", "const double *vj = jb->k + j * d;"),
    "lse_without_max": ("jb->lse[i] = m + log(l);", "jb->lse[i] = log(l);"),
    "no_normalisation": ("for (int64_t c = 0; c < d; ++c) oi[c] /= l;", ""),
    "merge_weight_sign": ("double w = exp(lse_parts[s] - L);", "double w = exp(L - lse_parts[s]);"),
    # backward
    "bwd_drop_delta": ("const double ds = p[j] * (dp - D);", "const double ds = p[j] * dp;"),
    "bwd_dk_from_keys": ("dkj[c] += jb->scale * ds * qi[c];", "dkj[c] += jb->scale * ds * krow[c];"),
    "bwd_dq_without_scale": ("dqi[c] += jb->scale * ds * krow[c];", "dqi[c] += ds * krow[c];"),
    "bwd_dv_from_queries": ("dvj[c] += p[j] * gi[c];", "dvj[c] += p[j] * qi[c];"),
    "bwd_causal_off_by_one": ("if (jb->causal && jb->qpos[i] + 1 < hi) hi = jb->qpos[i] + 1;",
                              "if (jb->causal && jb->qpos[i] < hi) hi = jb->qpos[i];"),
    "bwd_unnormalised_p": ("for (int64_t j = 0; j < hi; ++j) p[j] /= l;", ""),
}


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", str(path),
                    "-o", str(so), "-lm"], check=True)
    return str(so)


def _pins_pass():
    """A compact subset of the pins: SDPA (causal and GQA), closed forms, merge."""
    ok = True
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1, 4, 9, 8, generator=g, dtype=torch.float64)
    k = torch.randn(1, 2, 9, 8, generator=g, dtype=torch.float64)
    v = torch.randn(1, 2, 9, 8, generator=g, dtype=torch.float64)
    for causal in (False, True):
        ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=0.3, enable_gqa=True)
        o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), 0.3, causal)
        ok &= np.allclose(o, ref.numpy(), rtol=1e-11, atol=1e-12)
    o, lse = oracle.attention_head([[1.0, 0.0]], [[0.0, 0.0], [math.log(3), 0.0]],
                                   [[1.0, 2.0], [5.0, -2.0]], 1.0)
    ok &= np.allclose(o, [[4.0, -1.0]], atol=1e-12) and abs(lse[0] - math.log(4)) < 1e-12
    o, lse = oracle.attention_head([[1.0]], [[1000.0], [0.0]], [[7.0], [1.0]], 1.0)
    ok &= abs(lse[0] - 1000.0) < 1e-9
    mo, ml = oracle.lse_merge(np.array([[1.0, 2.0], [5.0, -2.0]]), np.array([0.0, math.log(3)]))
    ok &= np.allclose(mo, [4.0, -1.0], atol=1e-12) and abs(ml - math.log(4)) < 1e-12
    # backward: autograd of the library's fp64 attention (causal and GQA)
    for causal in (False, True):
        qg, kg, vg = (t.clone().requires_grad_(True) for t in (q, k, v))
        dout = torch.randn(1, 4, 9, 8, generator=g, dtype=torch.float64)
        F.scaled_dot_product_attention(qg, kg, vg, is_causal=causal, scale=0.3,
                                       enable_gqa=True).backward(dout)
        got = oracle.attention_bwd(q.numpy(), k.numpy(), v.numpy(), dout.numpy(), 0.3, causal)
        for mine, ref in zip(got, (qg.grad, kg.grad, vg.grad)):
            ok &= np.allclose(mine, ref.numpy(), rtol=1e-10, atol=1e-12)
    return bool(ok)


def test_unmutated_oracle_passes_the_subset():
    assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, monkeypatch, name):
    so = _build_mutant(tmp_path, name)
    real = oracle._load()
    lib = ctypes.CDLL(so)
    for fn in ("oracle_attention_head", "oracle_lse_merge", "oracle_default_threads",
               "oracle_attention_bwd_head"):
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
        getattr(lib, fn).restype = getattr(real, fn).restype
    monkeypatch.setattr(oracle, "_lib", lib)
    assert not _pins_pass(), f"mutant {name} passed the pins"
