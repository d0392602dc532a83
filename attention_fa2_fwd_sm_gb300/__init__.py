"""Python binding of libattn.so (fused attention for GB300 / sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/attn.h``.  The functions take
torch tensors (for device memory and the current stream) and return the
library's status code; ``check`` turns a non-zero code into an exception.
There is no fallback: if ``libattn.so`` cannot be loaded, importing the
functions raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

ATTN_OK = 0
ATTN_ERR_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_WORKSPACE = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_TIMEOUT = -5

ORDER_HEAD_FIRST = 0
ORDER_BLOCK_FIRST = 1
ORDER_NAIVE_HEAD_FIRST = 2
ORDER_DIE_SPLIT_HEAD_FIRST = 3
ORDERS = {"head_first": ORDER_HEAD_FIRST, "block_first": ORDER_BLOCK_FIRST,
          "naive_head_first": ORDER_NAIVE_HEAD_FIRST,
          "die_split_head_first": ORDER_DIE_SPLIT_HEAD_FIRST}
# forward tile schemes, OR-ed into tile_order (0: the library's choice)
FWD_SINGLE_CTA = 0x100
FWD_CTA_PAIR = 0x200
SCHEMES = {"auto": 0, "single": FWD_SINGLE_CTA, "pair": FWD_CTA_PAIR}

# Every symbol include/attn.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_LL = ctypes.c_longlong
_SZ = ctypes.c_size_t
_IP = ctypes.POINTER(ctypes.c_int)
_FP = ctypes.POINTER(ctypes.c_float)
SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_fwd_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "attn_fwd_host": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _SZ, _P]),
    "attn_fwd_host_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "attn_fwd_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "attn_fwd_splitkv_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "attn_fwd_host_trace": (_I, [_I]),
    "attn_fwd_host_trace_read": (_LL, [_FP, _LL]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "attn_bwd_workspace_bytes": (_SZ, [_I, _I, _I]),
    "attn_bwd_workspace_bytes_ex": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "attn_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "attn_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _P]),
    "attn_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "attn_decode_varlen": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "attn_decode_varlen_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "attn_decode_num_splits": (_I, [_I, _I, _I, _I]),
    "attn_tile_map": (_I, [_I, _I, _I, _I, _I, _I, _LL, _IP, _IP, _IP]),
    "attn_tile_map_die_split": (_I, [_I, _I, _I, _I, _I, _I, _LL, _IP, _IP, _IP]),
    "attn_bwd_tile_map": (_I, [_I, _I, _I, _I, _I, _I, _LL, _IP, _IP, _IP]),
    "attn_die_map": (_I, [_IP, _I, _FP]),
    "attn_fwd_units": (_LL, [_I, _I, _I]),
    "attn_device_status": (_I, [_P]),
    "attn_set_wait_timeout_ns": (_LL, [_LL]),
    "attn_strerror": (ctypes.c_char_p, [_I]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_version": (_I, []),
}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = f"{what}: {strerror(code)} ({code})" if what else f"{strerror(code)} ({code})"
        if code == ATTN_ERR_CUDA:
            msg += f" [{attn_last_error()}]"
        super().__init__(msg)


def lib():
    """Load libattn.so (raises OSError / RuntimeError when it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "attention_fa2_fwd_sm_gb300._build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().attn_strerror(int(code)).decode()


def check(code: int, what: str = "") -> None:
    if code != ATTN_OK:
        raise AttnError(code, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, stream=None) -> int:
    return lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                          float(scale), int(bool(causal)), _stream(stream))


def attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, tile_order, stream=None) -> int:
    return lib().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                             float(scale), int(bool(causal)), int(tile_order), _stream(stream))


def attn_fwd_host(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, tile_order, kv_heads_per_chunk,
                  workspace, workspace_bytes, stream=None) -> int:
    return lib().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, float(scale),
                               int(bool(causal)), int(tile_order), int(kv_heads_per_chunk), _ptr(workspace),
                               int(workspace_bytes), _stream(stream))


def attn_fwd_host_workspace_bytes(B, Hq, Hkv, N, d, kv_heads_per_chunk=0) -> int:
    return int(lib().attn_fwd_host_workspace_bytes(B, Hq, Hkv, N, d, kv_heads_per_chunk))


def attn_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, kv_splits, workspace, workspace_bytes,
                     stream=None) -> int:
    return lib().attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, float(scale),
                                  int(bool(causal)), int(kv_splits), _ptr(workspace), int(workspace_bytes),
                                  _stream(stream))


def attn_fwd_splitkv_workspace_bytes(B, Hq, N, d, kv_splits=0) -> int:
    return int(lib().attn_fwd_splitkv_workspace_bytes(B, Hq, N, d, kv_splits))


def forward_splitkv(q, k, v, causal=False, scale=None, kv_splits=0, workspace=None, with_lse=True, stream=None):
    """Allocate outputs (and a workspace when none is given) and run
    attn_fwd_splitkv on ``[B, H, N, d]`` bf16 CUDA tensors; returns
    ``(o, lse, workspace)``."""
    import torch
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = d ** -0.5
    nbytes = attn_fwd_splitkv_workspace_bytes(B, Hq, N, d, kv_splits)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if with_lse else None
    check(attn_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, kv_splits, workspace, nbytes,
                           stream), "attn_fwd_splitkv")
    return o, lse, workspace


def attn_fwd_host_trace(enable) -> int:
    return int(lib().attn_fwd_host_trace(int(bool(enable))))


def attn_fwd_host_trace_read(capacity=None):
    """Per-chunk timeline of the last traced attn_fwd_host call on the current
    device: a list of (copy-in done, kernel reached, kernel done, copy-out
    done) in ms from the call's start.  Raises when there is none."""
    n = int(lib().attn_fwd_host_trace_read(None, 0))
    if n < 0:
        check(n, "attn_fwd_host_trace_read")
    cap = n if capacity is None else min(n, int(capacity))
    buf = (ctypes.c_float * (4 * max(cap, 1)))()
    got = int(lib().attn_fwd_host_trace_read(buf, cap))
    if got < 0:
        check(got, "attn_fwd_host_trace_read")
    return [tuple(buf[4 * c: 4 * c + 4]) for c in range(cap)]


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal, tile_order,
             workspace, workspace_bytes, stream=None) -> int:
    return lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                          _ptr(dv), B, Hq, Hkv, N, d, float(scale), int(bool(causal)), int(tile_order),
                          _ptr(workspace), int(workspace_bytes), _stream(stream))


def attn_bwd_workspace_bytes(B, Hq, N) -> int:
    return int(lib().attn_bwd_workspace_bytes(B, Hq, N))


def attn_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, causal) -> int:
    return int(lib().attn_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, int(bool(causal))))


def attn_decode(q, kcache, vcache, seqlens, o, B, Hq, Hkv, d, scale, num_splits, max_seqlen,
                workspace=None, workspace_bytes=0, stream=None) -> int:
    return lib().attn_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(o), B, Hq,
                             Hkv, d, float(scale), int(num_splits), int(max_seqlen),
                             _ptr(workspace), int(workspace_bytes), _stream(stream))


def attn_decode_noalloc(q, kcache, vcache, seqlens, o, B, Hq, Hkv, d, scale, num_splits, max_seqlen,
                        stream=None) -> int:
    """attn_decode for callers that cannot allocate device memory: the split
    partials go to a scratch array built into the library (see attn.h)."""
    return lib().attn_decode_noalloc(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(o), B,
                                     Hq, Hkv, d, float(scale), int(num_splits), int(max_seqlen),
                                     _stream(stream))


DECODE_NOALLOC_SCRATCH_BYTES = 4194304


def attn_decode_varlen(q, kcache, vcache, seqlens, o, B, Hq, Hkv, d, scale, max_seqlen, workspace,
                       workspace_bytes, stream=None) -> int:
    return lib().attn_decode_varlen(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(o), B, Hq, Hkv,
                                    d, float(scale), int(max_seqlen), _ptr(workspace), int(workspace_bytes),
                                    _stream(stream))


def attn_decode_varlen_workspace_bytes(B, Hq, Hkv, d) -> int:
    return int(lib().attn_decode_varlen_workspace_bytes(B, Hq, Hkv, d))


def decode_varlen(q, kcache, vcache, seqlens, scale=None, workspace=None, stream=None):
    """Allocate the output (and a workspace when none is given) and run
    attn_decode_varlen; returns ``(o, workspace)``."""
    import torch
    B, Hq, d = q.shape
    Hkv, s_max = kcache.shape[1], kcache.shape[2]
    if scale is None:
        scale = d ** -0.5
    nbytes = attn_decode_varlen_workspace_bytes(B, Hq, Hkv, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    check(attn_decode_varlen(q, kcache, vcache, seqlens, o, B, Hq, Hkv, d, scale, s_max, workspace,
                             workspace.numel(), stream), "attn_decode_varlen")
    return o, workspace


def attn_decode_workspace_bytes(B, Hq, d, num_splits) -> int:
    return int(lib().attn_decode_workspace_bytes(B, Hq, d, num_splits))


def attn_decode_num_splits(B, Hq, Hkv, max_seqlen) -> int:
    return int(lib().attn_decode_num_splits(B, Hq, Hkv, max_seqlen))


def attn_tile_map(tile_order, B, Hq, Hkv, N, causal, unit):
    b, h, m = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = lib().attn_tile_map(int(tile_order), B, Hq, Hkv, N, int(bool(causal)), int(unit),
                             ctypes.byref(b), ctypes.byref(h), ctypes.byref(m))
    check(rc, "attn_tile_map")
    return b.value, h.value, m.value


def attn_tile_map_die_split(B, Hq, Hkv, N, causal, die, k):
    """(b, h, m) of the k-th unit of die `die` under the die-split order, or
    None when that die has no k-th unit of its own."""
    b, h, m = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = lib().attn_tile_map_die_split(B, Hq, Hkv, N, int(bool(causal)), int(die), int(k),
                                       ctypes.byref(b), ctypes.byref(h), ctypes.byref(m))
    if rc == ATTN_ERR_ARG:
        return None
    check(rc, "attn_tile_map_die_split")
    return b.value, h.value, m.value


def attn_bwd_tile_map(tile_order, B, Hkv, N, causal, num_sms, unit):
    """(b, g, j) of dK/dV unit `unit`: batch entry, KV head, 128-key block."""
    b, g, j = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = lib().attn_bwd_tile_map(int(tile_order), B, Hkv, N, int(bool(causal)), int(num_sms), int(unit),
                                 ctypes.byref(b), ctypes.byref(g), ctypes.byref(j))
    check(rc, "attn_bwd_tile_map")
    return b.value, g.value, j.value


def attn_die_map(capacity=256):
    """(die of each SM id, stats) of the current device, as the die-split order
    uses it; stats = (measured, min |corr|, near clk, far clk)."""
    dies = (ctypes.c_int * capacity)()
    stats = (ctypes.c_float * 4)()
    n = lib().attn_die_map(dies, capacity, stats)
    if n < 0:
        check(n, "attn_die_map")
    return list(dies[:min(n, capacity)]), tuple(stats)


def attn_fwd_units(B, Hq, N) -> int:
    return int(lib().attn_fwd_units(B, Hq, N))


def attn_device_status(stream=None) -> int:
    return lib().attn_device_status(_stream(stream))


def attn_set_wait_timeout_ns(ns: int) -> int:
    return int(lib().attn_set_wait_timeout_ns(int(ns)))


def attn_last_error() -> str:
    return lib().attn_last_error().decode()


def attn_version() -> int:
    return int(lib().attn_version())


# ----------------------------------------------------------- torch helpers
def forward(q, k, v, causal=False, scale=None, tile_order=ORDER_HEAD_FIRST, with_lse=True,
            stream=None):
    """Allocate outputs and run attn_fwd_ex on ``[B, H, N, d]`` bf16 CUDA tensors."""
    import torch
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = d ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if with_lse else None
    check(attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, tile_order, stream),
          "attn_fwd_ex")
    return o, lse


def forward_host(q, k, v, causal=False, scale=None, tile_order=ORDER_HEAD_FIRST, with_lse=True,
                 kv_heads_per_chunk=0, workspace=None, out=None, device=None, stream=None, synchronize=True):
    """Run attn_fwd_host on ``[B, H, N, d]`` bf16 CPU tensors (pinned for overlap).

    Allocates pinned outputs (unless ``out = (o, lse)`` is given) and a device
    workspace (unless given); with ``synchronize`` it waits for the stream, so
    the outputs are ready on return.  Returns ``(o, lse)``."""
    import torch
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = d ** -0.5
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    nbytes = attn_fwd_host_workspace_bytes(B, Hq, Hkv, N, d, kv_heads_per_chunk)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    if out is None:
        o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        lse = torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=True) if with_lse else None
    else:
        o, lse = out
    check(attn_fwd_host(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, tile_order, kv_heads_per_chunk,
                        workspace, nbytes, stream), "attn_fwd_host")
    if synchronize:
        torch.cuda.current_stream(dev).synchronize() if stream is None else torch.cuda.synchronize(dev)
    return o, lse


def backward(q, k, v, o, lse, dout, causal=False, scale=None, tile_order=ORDER_HEAD_FIRST, workspace=None,
             stream=None):
    """Allocate gradients (and a workspace when none is given) and run attn_bwd
    on ``[B, H, N, d]`` bf16 CUDA tensors; returns ``(dq, dk, dv)``."""
    import torch
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = d ** -0.5
    nbytes = attn_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, causal)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    else:
        nbytes = min(nbytes, workspace.numel() * workspace.element_size())
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    check(attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal, tile_order,
                   workspace, nbytes, stream), "attn_bwd")
    return dq, dk, dv


def decode(q, kcache, vcache, seqlens, num_splits=0, scale=None, workspace=None, stream=None):
    """Allocate the output (and a workspace when none is given) and run attn_decode."""
    import torch
    B, Hq, d = q.shape
    Hkv, s_max = kcache.shape[1], kcache.shape[2]
    if scale is None:
        scale = d ** -0.5
    splits = num_splits if num_splits > 0 else attn_decode_num_splits(B, Hq, Hkv, s_max)
    nbytes = attn_decode_workspace_bytes(B, Hq, d, splits)
    if workspace is None and nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    check(attn_decode(q, kcache, vcache, seqlens, o, B, Hq, Hkv, d, scale, splits, s_max,
                      workspace, nbytes, stream), "attn_decode")
    return o, workspace, splits
