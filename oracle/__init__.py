"""fp64 CPU oracle for the attention hot path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only users.  The product path (the CUDA
library and its Python binding) never imports, links or runs anything here,
and this package imports nothing from the product.

The arithmetic lives in ``attn_oracle.c`` (the plain definition of attention,
row by row, in double precision, its gradient by the chain rule, and the
log-sum-exp merge); this module only
builds it with gcc, marshals numpy arrays and applies the readings that the
pages leave open:

* per-head tensors are ``[B, H, N, d]`` (detail page, section 4 notation:
  Q, K, V in R^{N x d} per head);
* grouped-query attention uses contiguous groups: query head ``h`` reads
  KV head ``h // G`` with ``G = Hq // Hkv`` (kernbench2 "Fused Grouped-Query
  Attention" introduction: each KV head shared by a group of G query heads);
* causal masking keeps key ``j`` for query ``i`` iff ``j <= i`` (equal query
  and key lengths, so top-left and bottom-right alignment coincide);
* decode is one query row per (batch, query head) against ``seqlens[b]``
  keys (kernbench2, same section: a decode step has T_q = 1);
* split-KV decode cuts the key range into ``num_splits`` chunks of
  ``ceil(seqlen / num_splits)`` keys rounded up to 64; an empty chunk has
  ``lse = -inf`` and weight 0 in the merge (kernbench2 "Inference with
  Long-Context Length", Case 4: KV split with a reduction of (m, l, O)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``liboracle.so`` with gcc (plain -O2)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_attention_head.argtypes = [
            _D, _D, _D, _I64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_double, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _D, _D,
            ctypes.c_int]
        lib.oracle_attention_head.restype = ctypes.c_int
        lib.oracle_lse_merge.argtypes = [_D, _D, ctypes.c_int64, ctypes.c_int64, _D, _D]
        lib.oracle_lse_merge.restype = ctypes.c_int
        lib.oracle_attention_bwd_head.argtypes = [
            _D, _D, _D, _D, _I64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_double, ctypes.c_int, _D, _D, _D, ctypes.c_int]
        lib.oracle_attention_bwd_head.restype = ctypes.c_int
        lib.oracle_default_threads.argtypes = []
        lib.oracle_default_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    """Worker threads used when ``nthreads=0`` (all online host cores)."""
    return int(_load().oracle_default_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_D)


def attention_head(q, k, v, scale, causal=False, qpos=None, k_lo=0, k_hi=None, nthreads=0):
    """One head: ``q [nq, d]``, ``k, v [nk, d]`` -> ``(o [nq, d], lse [nq])`` in fp64.

    ``qpos[i]`` is the absolute position of query row i (default ``0..nq-1``);
    keys attended are ``[k_lo, k_hi)`` and, when ``causal``, ``j <= qpos[i]``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, d = q.shape
    nk = k.shape[0]
    if k.shape != (nk, d) or v.shape != (nk, d):
        raise ValueError("k and v must be [nk, d] with the d of q")
    if k_hi is None:
        k_hi = nk
    if qpos is None:
        qpos = np.arange(nq, dtype=np.int64)
    qpos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
    o = np.zeros((nq, d), dtype=np.float64)
    lse = np.zeros((nq,), dtype=np.float64)
    rc = _load().oracle_attention_head(
        _ptr(q), _ptr(k), _ptr(v), qpos.ctypes.data_as(_I64), nq, nk, d, float(scale),
        int(bool(causal)), int(k_lo), int(k_hi), _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attention_head rejected its arguments")
    return o, lse


def attention_bwd_head(q, k, v, dout, scale, causal=False, qpos=None, nthreads=0):
    """Gradients of one head for output gradient ``dout [nq, d]``:
    ``(dq [nq, d], dk [nk, d], dv [nk, d])`` in fp64 (chain rule of the
    forward definition; see ``attn_oracle.c``)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    nq, d = q.shape
    nk = k.shape[0]
    if k.shape != (nk, d) or v.shape != (nk, d) or dout.shape != (nq, d):
        raise ValueError("k, v must be [nk, d] and dout [nq, d] with the d of q")
    if qpos is None:
        qpos = np.arange(nq, dtype=np.int64)
    qpos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
    dq = np.zeros((nq, d), dtype=np.float64)
    dk = np.zeros((nk, d), dtype=np.float64)
    dv = np.zeros((nk, d), dtype=np.float64)
    rc = _load().oracle_attention_bwd_head(
        _ptr(q), _ptr(k), _ptr(v), _ptr(dout), qpos.ctypes.data_as(_I64), nq, nk, d, float(scale),
        int(bool(causal)), _ptr(dq), _ptr(dk), _ptr(dv), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attention_bwd_head rejected its arguments")
    return dq, dk, dv


def kv_head_of(h: int, hq: int, hkv: int) -> int:
    """KV head read by query head ``h`` (contiguous groups of ``hq // hkv``)."""
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return h // (hq // hkv)


def attention(q, k, v, scale, causal=False, nthreads=0):
    """Full forward: ``q [B, Hq, N, d]``, ``k, v [B, Hkv, Nk, d]`` -> ``(o, lse)``."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, hq, n, d = q.shape
    hkv = k.shape[1]
    o = np.zeros_like(q)
    lse = np.zeros((B, hq, n), dtype=np.float64)
    for b in range(B):
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            o[b, h], lse[b, h] = attention_head(q[b, h], k[b, g], v[b, g], scale, causal,
                                                nthreads=nthreads)
    return o, lse


def attention_bwd(q, k, v, dout, scale, causal=False, nthreads=0):
    """Full backward: ``q, dout [B, Hq, N, d]``, ``k, v [B, Hkv, N, d]`` ->
    ``(dq, dk, dv)``; the gradient of a KV head is the sum over the query
    heads that read it."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, hq, _, _ = q.shape
    hkv = k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            dq[b, h], dkh, dvh = attention_bwd_head(q[b, h], k[b, g], v[b, g], dout[b, h], scale,
                                                    causal, nthreads=nthreads)
            dk[b, g] += dkh
            dv[b, g] += dvh
    return dq, dk, dv


def attention_rows(q_rows, k_head, v_head, scale, causal, positions, nthreads=0):
    """Selected rows of one head: ``q_rows [r, d]`` at absolute ``positions``."""
    return attention_head(q_rows, k_head, v_head, scale, causal, qpos=positions,
                          nthreads=nthreads)


def decode(q, kcache, vcache, seqlens, scale, nthreads=0):
    """Decode: ``q [B, Hq, d]``, caches ``[B, Hkv, S_max, d]``, ``seqlens [B]``."""
    q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
    B, hq, d = q.shape
    hkv = kc.shape[1]
    o = np.zeros((B, hq, d), dtype=np.float64)
    lse = np.zeros((B, hq), dtype=np.float64)
    for b in range(B):
        n = int(seqlens[b])
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            ob, lb = attention_head(q[b, h][None, :], kc[b, g], vc[b, g], scale, False,
                                    k_lo=0, k_hi=n, nthreads=1 if nthreads == 0 else nthreads)
            o[b, h], lse[b, h] = ob[0], lb[0]
    return o, lse


def split_ranges(seqlen: int, num_splits: int, granule: int = 64):
    """Key ranges of the split-KV decode: chunks of ceil(seqlen/splits) keys
    rounded up to ``granule``; trailing chunks may be empty."""
    if num_splits <= 0:
        raise ValueError("num_splits must be positive")
    per = -(-seqlen // num_splits) if seqlen > 0 else 0
    chunk = -(-per // granule) * granule
    out = []
    for s in range(num_splits):
        lo = min(s * chunk, seqlen)
        hi = min((s + 1) * chunk, seqlen)
        out.append((lo, hi))
    return out


def varlen_plan(seqlens, max_seqlen: int, hkv: int, target: int, min_chunk: int = 512, granule: int = 64):
    """Work list of the ragged multi-user decode (integer arithmetic): one chunk
    size for the whole batch, C = max(min_chunk, ceil(T * hkv / target) rounded
    up to ``granule``) with T the total number of attended keys; sequence b is
    cut into ceil(len_b / C) chunks [c C, min(c C + C, len_b)).  Returns
    ``(C, [(b, lo, hi), ...])`` in batch order.  This splits the KV sequence of
    each user as the kernbench2 decode family does (statically sharded KV,
    partial states reduced per user); the chunk rule is this library's reading
    (the pages size shards by device count, which has no one-GPU analogue)."""
    lens = [min(max(int(n), 0), int(max_seqlen)) for n in seqlens]
    total = sum(lens)
    c = -(-total * int(hkv) // int(target))
    c = -(-c // granule) * granule
    c = max(c, min_chunk)
    items = []
    for b, n in enumerate(lens):
        for lo in range(0, n, c):
            items.append((b, lo, min(lo + c, n)))
    return c, items


def decode_partials(q, kcache, vcache, seqlens, scale, num_splits):
    """Per-split partial states: ``o_parts [B, Hq, S, d]`` (each normalised by its
    own sum) and ``lse_parts [B, Hq, S]`` (-inf for an empty split)."""
    q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
    B, hq, d = q.shape
    hkv = kc.shape[1]
    o_parts = np.zeros((B, hq, num_splits, d), dtype=np.float64)
    lse_parts = np.zeros((B, hq, num_splits), dtype=np.float64)
    for b in range(B):
        for s, (lo, hi) in enumerate(split_ranges(int(seqlens[b]), num_splits)):
            for h in range(hq):
                g = kv_head_of(h, hq, hkv)
                ob, lb = attention_head(q[b, h][None, :], kc[b, g], vc[b, g], scale, False,
                                        k_lo=lo, k_hi=hi, nthreads=1)
                o_parts[b, h, s], lse_parts[b, h, s] = ob[0], lb[0]
    return o_parts, lse_parts


def lse_merge(o_parts, lse_parts):
    """Merge partial states over the second-to-last axis of ``o_parts [..., S, d]``."""
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    *lead, S, d = o_parts.shape
    flat_o = o_parts.reshape(-1, S, d)
    flat_l = lse_parts.reshape(-1, S)
    out = np.zeros((flat_o.shape[0], d), dtype=np.float64)
    out_lse = np.zeros((flat_o.shape[0],), dtype=np.float64)
    lib = _load()
    for r in range(flat_o.shape[0]):
        po = np.ascontiguousarray(flat_o[r])
        pl = np.ascontiguousarray(flat_l[r])
        row = np.zeros((d,), dtype=np.float64)
        lse = np.zeros((1,), dtype=np.float64)
        if lib.oracle_lse_merge(_ptr(po), _ptr(pl), S, d, _ptr(row), _ptr(lse)) != 0:
            raise ValueError("oracle_lse_merge rejected its arguments")
        out[r], out_lse[r] = row, lse[0]
    if not lead:
        return out[0], float(out_lse[0])
    return out.reshape(*lead, d), out_lse.reshape(*lead)
