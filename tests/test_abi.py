"""CPU-only checks of the C-ABI library: it builds, loads, exports every
declared symbol, validates arguments on the host before any CUDA call, and
its scheduler agrees with the tile-order definitions.  No kernel runs."""
import os
import re

import pytest

import attention_fa2_fwd_sm_gb300 as attn
from attention_fa2_fwd_sm_gb300 import _build
from oracle import tile_order as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
A16 = 0x10000  # a fake 16-byte-aligned address: never dereferenced by these calls


@pytest.fixture(scope="module")
def L():
    _build.build()
    return attn.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text))


def test_every_declared_symbol_is_exported(L):
    names = _declared_functions()
    assert "attn_fwd" in names and "attn_decode" in names
    for n in names:
        assert hasattr(L, n), n
    assert names == set(attn.SIGNATURES), "binding and header disagree"


def test_noalloc_scratch_size_agrees_with_the_header(L):
    """The binding's copy of the built-in scratch size is the header's value
    (the library itself checks the header against its own constant when it
    compiles)."""
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    m = re.search(r"#define\s+ATTN_DECODE_NOALLOC_SCRATCH_BYTES\s+(\d+)u?", text)
    assert m, "ATTN_DECODE_NOALLOC_SCRATCH_BYTES not found in attn.h"
    assert int(m.group(1)) == attn.DECODE_NOALLOC_SCRATCH_BYTES


def test_fwd_host_trace_read_checks_its_buffer(L):
    # a capacity without a buffer is refused before any CUDA call
    assert L.attn_fwd_host_trace_read(None, 4) == attn.ATTN_ERR_ARG
    assert L.attn_fwd_host_trace_read(None, -1) == attn.ATTN_ERR_ARG


def test_version_and_messages(L):
    assert attn.attn_version() >= 100
    for code in (0, -1, -2, -3, -4, -5):
        assert attn.strerror(code) and attn.strerror(code) != "unknown status code"
    assert attn.strerror(-99) == "unknown status code"


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(attn, "_lib", None)
    monkeypatch.setattr(attn, "LIB_PATH", "/nonexistent/libattn.so")
    with pytest.raises(RuntimeError):
        attn.lib()


@pytest.mark.parametrize("order", T.ORDERS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Hkv,N", [(1, 2, 2, 256), (2, 3, 3, 300), (1, 8, 8, 4096), (3, 5, 5, 1),
                                       (1, 8, 2, 1300), (2, 6, 3, 600), (1, 64, 8, 2048),
                                       (1, 64, 8, 16384), (1, 64, 8, 16385), (1, 8, 2, 70000)])
def test_scheduler_matches_the_definitions(L, order, causal, B, H, Hkv, N):
    nb = T.num_blocks(N, 256)
    assert attn.attn_fwd_units(B, H, N) == B * H * nb
    for u in range(B * H * nb):
        assert (attn.attn_tile_map(order, B, H, Hkv, N, causal, u)
                == T.unit_to_tile(order, u, B, H, nb, causal, H // Hkv))


@pytest.mark.parametrize("order", T.ORDERS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hkv,N,sms", [(1, 8, 8192, 152), (1, 7, 11739, 152), (2, 3, 1000, 152),
                                         (1, 8, 32768, 152), (3, 5, 3000, 8), (1, 1, 1, 152)])
def test_dkdv_scheduler_matches_the_definition(L, order, causal, B, Hkv, N, sms):
    seq = T.dkdv_sequence(order, B, Hkv, N, causal, sms)
    for u, want in enumerate(seq):
        assert attn.attn_bwd_tile_map(order, B, Hkv, N, causal, sms, u) == want
    with pytest.raises(attn.AttnError):
        attn.attn_bwd_tile_map(order, B, Hkv, N, causal, sms, len(seq))


def test_dkdv_scheduler_rejects_bad_arguments(L):
    for args in [(3, 1, 2, 256, True, 152, 0), (0, 1, 2, 256, True, 0, 0), (0, 0, 2, 256, True, 152, 0),
                 (0, 1, 2, 256, True, 152, -1)]:
        with pytest.raises(attn.AttnError):
            attn.attn_bwd_tile_map(*args)


def test_scheduler_rejects_bad_units(L):
    with pytest.raises(attn.AttnError):
        attn.attn_tile_map(0, 1, 2, 2, 256, False, 2)
    with pytest.raises(attn.AttnError):
        attn.attn_tile_map(7, 1, 2, 2, 256, False, 0)
    with pytest.raises(attn.AttnError):
        attn.attn_tile_map(0, 1, 6, 4, 256, True, 0)  # Hq % Hkv != 0


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 8, 8, 300), (1, 64, 8, 1024), (3, 6, 3, 257), (1, 4, 1, 256)])
def test_die_split_scheduler_matches_the_definition(L, causal, B, Hq, Hkv, N):
    nb = T.num_blocks(N, 256)
    for die in (0, 1):
        want = T.die_split_sequence(die, B, Hq, Hkv, nb, causal)
        got = [attn.attn_tile_map_die_split(B, Hq, Hkv, N, causal, die, k) for k in range(len(want))]
        assert got == want
        assert attn.attn_tile_map_die_split(B, Hq, Hkv, N, causal, die, len(want)) is None


def test_tile_map_rejects_the_die_split_order(L):
    with pytest.raises(attn.AttnError):
        attn.attn_tile_map(3, 1, 2, 2, 256, False, 0)
    assert attn.attn_tile_map_die_split(1, 2, 2, 256, False, 2, 0) is None  # no die 2
    assert attn.attn_tile_map_die_split(1, 2, 2, 256, False, 0, -1) is None


def _fwd(**kw):
    a = dict(q=A16, k=A16, v=A16, o=A16, lse=None, B=1, Hq=2, Hkv=2, N=256, d=64, scale=0.125,
             causal=False, tile_order=0, stream=0)
    a.update(kw)
    return attn.attn_fwd_ex(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"],
                            a["N"], a["d"], a["scale"], a["causal"], a["tile_order"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_ERR_ARG),
    (dict(o=A16 + 8), attn.ATTN_ERR_ARG),
    (dict(lse=A16 + 2), attn.ATTN_ERR_ARG),
    (dict(B=0), attn.ATTN_ERR_ARG),
    (dict(N=-5), attn.ATTN_ERR_ARG),
    (dict(Hq=3, Hkv=2), attn.ATTN_ERR_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_ARG),
    (dict(tile_order=4), attn.ATTN_ERR_ARG),
    (dict(tile_order=-1), attn.ATTN_ERR_ARG),
    (dict(B=1 << 16, Hq=256, Hkv=256, N=1 << 16), attn.ATTN_ERR_ARG),  # 2^33 work units
    (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=256), attn.ATTN_ERR_UNSUPPORTED),
])
def test_forward_argument_errors(L, kw, code):
    assert _fwd(**kw) == code


def _dec(**kw):
    a = dict(q=A16, k=A16, v=A16, seqlens=A16, o=A16, B=2, Hq=64, Hkv=8, d=128, scale=0.1,
             splits=4, s_max=1024, ws=A16, ws_bytes=1 << 30, stream=0)
    a.update(kw)
    return attn.attn_decode(a["q"], a["k"], a["v"], a["seqlens"], a["o"], a["B"], a["Hq"], a["Hkv"],
                            a["d"], a["scale"], a["splits"], a["s_max"], a["ws"], a["ws_bytes"],
                            a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(seqlens=None), attn.ATTN_ERR_ARG),
    (dict(k=A16 + 4), attn.ATTN_ERR_ARG),
    (dict(Hq=60, Hkv=8), attn.ATTN_ERR_ARG),
    (dict(s_max=0), attn.ATTN_ERR_ARG),
    (dict(splits=257), attn.ATTN_ERR_ARG),
    (dict(scale=-1.0), attn.ATTN_ERR_ARG),
    (dict(d=56), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Hq=64, Hkv=2), attn.ATTN_ERR_UNSUPPORTED),
    (dict(ws=None), attn.ATTN_ERR_WORKSPACE),
    (dict(ws_bytes=100), attn.ATTN_ERR_WORKSPACE),
    (dict(ws=A16 + 8), attn.ATTN_ERR_WORKSPACE),
])
def test_decode_argument_errors(L, kw, code):
    assert _dec(**kw) == code


def test_workspace_size(L):
    assert attn.attn_decode_workspace_bytes(2, 64, 128, 1) == 0
    n = 2 * 64 * 4
    o_bytes = -(-(n * 128 * 4) // 256) * 256
    assert attn.attn_decode_workspace_bytes(2, 64, 128, 4) == o_bytes + n * 4


def test_wait_timeout_setting_round_trips(L):
    old = attn.attn_set_wait_timeout_ns(12345)
    assert attn.attn_set_wait_timeout_ns(old) == 12345


def test_build_is_for_sm103a():
    assert "arch=compute_103a,code=sm_103a" in _build.ARCH


def test_noalloc_decode_refuses_on_the_host(L):
    """Refusals happen before any CUDA call (no device needed)."""
    p = (A16, A16, A16, A16, A16)
    # 32 x 64 heads x 64 splits of 129 floats needs far more than the built-in scratch
    assert attn.attn_decode_workspace_bytes(32, 64, 128, 64) > attn.DECODE_NOALLOC_SCRATCH_BYTES
    assert attn.attn_decode_noalloc(*p, 32, 64, 8, 128, 0.1, 64, 4096, 0) == attn.ATTN_ERR_WORKSPACE
    assert attn.attn_decode_noalloc(None, *p[1:], 2, 64, 8, 128, 0.1, 4, 1024, 0) == attn.ATTN_ERR_ARG
    assert attn.attn_decode_noalloc(*p, 2, 64, 8, 56, 0.1, 4, 1024, 0) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_decode_noalloc(*p, 2, 64, 8, 128, 0.1, 300, 1024, 0) == attn.ATTN_ERR_ARG


def _bwd(**kw):
    a = dict(q=A16, k=A16, v=A16, o=A16, dout=A16, lse=A16, dq=A16, dk=A16, dv=A16, B=1, Hq=2, Hkv=2, N=256,
             d=64, scale=0.125, causal=False, order=0, ws=A16, ws_bytes=1 << 20, stream=0)
    a.update(kw)
    return attn.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"],
                         a["B"], a["Hq"], a["Hkv"], a["N"], a["d"], a["scale"], a["causal"], a["order"],
                         a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_ERR_ARG),
    (dict(dout=A16 + 2), attn.ATTN_ERR_ARG),
    (dict(lse=None), attn.ATTN_ERR_ARG),
    (dict(lse=A16 + 2), attn.ATTN_ERR_ARG),
    (dict(dk=None), attn.ATTN_ERR_ARG),
    (dict(Hq=3, Hkv=2), attn.ATTN_ERR_ARG),
    (dict(scale=-1.0), attn.ATTN_ERR_ARG),
    (dict(order=3), attn.ATTN_ERR_ARG),
    (dict(d=32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(ws=None), attn.ATTN_ERR_WORKSPACE),
    (dict(ws=A16 + 4), attn.ATTN_ERR_WORKSPACE),
    (dict(ws_bytes=2 * 2 * 256 * 4 - 1), attn.ATTN_ERR_WORKSPACE),
])
def test_backward_argument_errors(L, kw, code):
    assert _bwd(**kw) == code


def test_backward_workspace_size(L):
    assert attn.attn_bwd_workspace_bytes(1, 2, 256) == 2 * 2 * 256 * 4
    assert attn.attn_bwd_workspace_bytes(2, 3, 129) == 2 * 2 * 3 * 256 * 4  # rows padded to 128
    assert attn.attn_bwd_workspace_bytes(0, 2, 256) == 0
    # the dK/dV query-head split: the smallest s dividing G with >= 912 units, else G
    base = attn.attn_bwd_workspace_bytes(1, 64, 8192)
    assert attn.attn_bwd_workspace_bytes_ex(1, 128, 128, 8192, 128, 0) == attn.attn_bwd_workspace_bytes(1, 128, 8192)
    assert attn.attn_bwd_workspace_bytes_ex(1, 64, 8, 32768, 128, 0) == attn.attn_bwd_workspace_bytes(1, 64, 32768)
    # GQA 64/8 at 8K: 8 * 64 = 512 units, s = 2 gives 1024; causal never splits
    assert attn.attn_bwd_workspace_bytes_ex(1, 64, 8, 8192, 128, 0) == (base + 255) // 256 * 256 + 8 * 8 * 2 * 8192 * 128
    assert attn.attn_bwd_workspace_bytes_ex(1, 64, 8, 8192, 128, 1) == base
    # 2 KV heads of 3 blocks (6 units), G = 3: no divisor reaches 912, s = G
    base = attn.attn_bwd_workspace_bytes(1, 6, 300)
    assert attn.attn_bwd_workspace_bytes_ex(1, 6, 2, 300, 56, 0) == (base + 255) // 256 * 256 + 8 * 2 * 3 * 300 * 56
    assert attn.attn_bwd_workspace_bytes_ex(1, 6, 4, 300, 56, 0) == 0  # Hq % Hkv != 0


def _dvl(**kw):
    a = dict(q=A16, k=A16, v=A16, seqlens=A16, o=A16, B=2, Hq=64, Hkv=8, d=128, scale=0.1, s_max=1024,
             ws=A16, ws_bytes=1 << 30, stream=0)
    a.update(kw)
    return attn.attn_decode_varlen(a["q"], a["k"], a["v"], a["seqlens"], a["o"], a["B"], a["Hq"], a["Hkv"],
                                   a["d"], a["scale"], a["s_max"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_ERR_ARG),
    (dict(seqlens=A16 + 2), attn.ATTN_ERR_ARG),
    (dict(B=0), attn.ATTN_ERR_ARG),
    (dict(Hq=12, Hkv=8), attn.ATTN_ERR_ARG),
    (dict(s_max=0), attn.ATTN_ERR_ARG),
    (dict(scale=float("inf")), attn.ATTN_ERR_ARG),
    (dict(d=56), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Hq=64, Hkv=2), attn.ATTN_ERR_UNSUPPORTED),
    (dict(ws=None), attn.ATTN_ERR_WORKSPACE),
    (dict(ws=A16 + 8), attn.ATTN_ERR_WORKSPACE),
])
def test_varlen_decode_argument_errors(L, kw, code):
    assert _dvl(**kw) == code


def _fh(**kw):
    a = dict(q=A16, k=A16, v=A16, o=A16, lse=None, B=1, Hq=4, Hkv=2, N=100, d=64, scale=0.1, causal=0, order=0,
             chunk=0, ws=A16, ws_bytes=1 << 30, stream=0)
    a.update(kw)
    return attn.attn_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"], a["d"],
                              a["scale"], a["causal"], a["order"], a["chunk"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_ERR_ARG),
    (dict(o=None), attn.ATTN_ERR_ARG),
    (dict(lse=A16 + 2), attn.ATTN_ERR_ARG),
    (dict(B=0), attn.ATTN_ERR_ARG),
    (dict(Hq=3), attn.ATTN_ERR_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_ARG),
    (dict(order=4), attn.ATTN_ERR_ARG),
    (dict(chunk=3), attn.ATTN_ERR_ARG),  # more KV heads than Hkv
    (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(ws=None), attn.ATTN_ERR_WORKSPACE),
    (dict(ws=A16 + 8), attn.ATTN_ERR_WORKSPACE),
    (dict(chunk=1, ws_bytes=2 * (2 * 25600 + 2 * 12800 + 1024) - 1), attn.ATTN_ERR_WORKSPACE),
])
def test_host_forward_argument_errors(L, kw, code):
    """Host-buffer forward: host pointers need no alignment, but every other
    check runs before any CUDA call, as for the device entry points."""
    assert _fh(**kw) == code


def test_host_forward_workspace_size(L):
    # one slot: q, k, v, o (bf16) and lse (fp32) of one chunk, each rounded up to 256 bytes; two slots
    def slot(gc, G, N, d):
        r = lambda x: (x + 255) // 256 * 256
        q, kv, l = gc * G * N * d * 2, gc * N * d * 2, gc * G * N * 4
        return r(q) + 2 * r(kv) + r(q) + r(l)
    assert attn.attn_fwd_host_workspace_bytes(1, 4, 2, 100, 56, 1) == 2 * slot(1, 2, 100, 56)
    assert attn.attn_fwd_host_workspace_bytes(1, 4, 2, 100, 64, 2) == 2 * slot(2, 2, 100, 64)
    # default chunk: the fewest KV heads holding 304 work units of 256 query rows, at most Hkv
    assert attn.attn_fwd_host_workspace_bytes(1, 128, 128, 32768, 128, 0) == 2 * slot(3, 1, 32768, 128)
    assert attn.attn_fwd_host_workspace_bytes(1, 128, 128, 1024, 128, 0) == 2 * slot(76, 1, 1024, 128)
    assert attn.attn_fwd_host_workspace_bytes(8, 64, 8, 32768, 128, 0) == 2 * slot(1, 8, 32768, 128)
    assert attn.attn_fwd_host_workspace_bytes(1, 64, 8, 512, 128, 0) == 2 * slot(8, 8, 512, 128)
    assert attn.attn_fwd_host_workspace_bytes(1, 4, 2, 100, 64, 3) == 0
    assert attn.attn_fwd_host_workspace_bytes(1, 4, 2, 100, 32, 1) == 0


def test_forward_tile_scheme_flags_are_validated(L):
    """The scheme flags ride in tile_order; the pair scheme is d = 128 only.
    All refused on the host, before any CUDA call."""
    args = lambda order, d: (A16, A16, A16, A16, None, 1, 2, 2, 256, d, 0.125, 0, order, 0)
    assert attn.attn_fwd_ex(*args(attn.FWD_CTA_PAIR, 64)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_fwd_ex(*args(attn.FWD_CTA_PAIR | 1, 56)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_fwd_ex(*args(attn.FWD_CTA_PAIR | attn.FWD_SINGLE_CTA, 128)) == attn.ATTN_ERR_ARG
    assert attn.attn_fwd_ex(*args(0x400, 128)) == attn.ATTN_ERR_ARG
    assert attn.attn_fwd_ex(*args(attn.FWD_CTA_PAIR | 4, 128)) == attn.ATTN_ERR_ARG
    assert attn.attn_fwd_ex(*args(-1, 128)) == attn.ATTN_ERR_ARG
    # the backward pass takes plain orders only
    assert _bwd(order=attn.FWD_SINGLE_CTA, d=128) == attn.ATTN_ERR_ARG


def test_splitkv_workspace_and_argument_errors(L):
    # N = 1000, 3 ranges: ceil(1000 / 3) = 334 keys, rounded up to 384 -> 3 ranges
    rows = 1 * 2 * 1000
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 2, 1000, 64, 3) == rows * 3 * 64 * 4 + rows * 3 * 4
    # 4 ranges asked of 300 keys: 128-key ranges -> 3 ranges
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 1, 300, 128, 4) == 300 * 3 * 128 * 4 + 300 * 3 * 4
    # the library's choice: K + V of one head in 32 MiB -> 65536 keys at d = 128
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 1, 65536, 128, 0) == 65536 * 128 * 4 + 65536 * 4
    two = 131072 * 2
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 1, 131072, 128, 0) == two * 128 * 4 + two * 4
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 1, 1000, 128, 65) == 0
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 1, 1000, 32, 2) == 0
    args = lambda **kw: dict(dict(q=A16, k=A16, v=A16, o=A16, lse=None, B=1, Hq=2, Hkv=2, N=256, d=64, scale=0.125,
                                  causal=0, s=2, ws=A16, wb=1 << 30), **kw)
    call = lambda a: attn.attn_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"],
                                          a["d"], a["scale"], a["causal"], a["s"], a["ws"], a["wb"], 0)
    assert call(args(s=65)) == attn.ATTN_ERR_ARG
    assert call(args(q=None)) == attn.ATTN_ERR_ARG
    assert call(args(Hq=3)) == attn.ATTN_ERR_ARG
    assert call(args(d=32)) == attn.ATTN_ERR_UNSUPPORTED
    assert call(args(ws=None)) == attn.ATTN_ERR_WORKSPACE
    assert call(args(wb=100)) == attn.ATTN_ERR_WORKSPACE
