"""GPU parity of the ragged multi-user decode (attn_decode_varlen) through the
C ABI: outputs against the fp64 oracle, the device work list against the
oracle's plan (integers, bit-exact), and agreement with attn_decode."""
import numpy as np
import pytest
import torch

import oracle
from synthetic_inputs import decode_inputs
from tests.gpu_util import assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    from attention_fa2_fwd_sm_gb300 import _build
    _build.build()
    import attention_fa2_fwd_sm_gb300 as A
    A.lib()
    oracle.build()
    return A


def _target():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return max(1, (5 * sms) // 3)


CASES = [  # Hq, Hkv, d, s_max, seqlens
    (64, 8, 128, 20000, [0, 1, 63, 64, 65, 1000, 4096, 20000, 130]),
    (32, 2, 64, 3000, [3000, 17, 0, 2999, 512, 513]),
    (8, 8, 128, 5000, [5000, 4, 2500]),
    (64, 8, 128, 32768, [32768, 100, 2000, 0, 5000, 64, 777, 32767]),
]


@pytest.mark.parametrize("Hq,Hkv,d,s_max,lens", CASES)
def test_ragged_batches_match_the_oracle_and_the_plan(attn, Hq, Hkv, d, s_max, lens):
    dev = torch.device("cuda")
    B = len(lens)
    q, kc, vc = decode_inputs(41, B, Hq, Hkv, s_max, d, dev)
    seq = torch.tensor(lens, dtype=torch.int32, device=dev)
    o, ws = attn.decode_varlen(q, kc, vc, seq)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    o_ref, _ = oracle.decode(to64(q), to64(kc), to64(vc), lens, d ** -0.5)
    assert_close(to64(o), o_ref, what=f"varlen {lens}")
    # the work list the device built, read from the documented workspace head
    c_ref, items_ref = oracle.varlen_plan(lens, s_max, Hkv, _target())
    head = ws[: 4 * (2 + 2 * B + 3 * len(items_ref))].view(torch.int32).cpu().tolist()
    assert head[0] == len(items_ref) and head[1] == c_ref
    items = [tuple(head[2 + 2 * B + 3 * i: 5 + 2 * B + 3 * i]) for i in range(head[0])]
    assert items == items_ref
    first = [sum(1 for b2, _, _ in items_ref if b2 < b) for b in range(B)]
    assert head[2:2 + B] == first
    assert head[2 + B:2 + 2 * B] == [sum(1 for b2, _, _ in items_ref if b2 == b) for b in range(B)]


def test_agrees_with_the_split_decode(attn):
    dev = torch.device("cuda")
    lens = [9000, 10, 4100, 0, 7000]
    B, Hq, Hkv, d, s_max = len(lens), 64, 8, 128, 9000
    q, kc, vc = decode_inputs(42, B, Hq, Hkv, s_max, d, dev)
    seq = torch.tensor(lens, dtype=torch.int32, device=dev)
    o_v, _ = attn.decode_varlen(q, kc, vc, seq)
    o_s, _, _ = attn.decode(q, kc, vc, seq)
    torch.cuda.synchronize()
    diff = (o_v.float() - o_s.float()).abs().max().item()
    assert diff <= 2e-2
    assert torch.count_nonzero(o_v[3]) == 0  # empty sequence -> zeros in both
    assert torch.count_nonzero(o_s[3]) == 0


def test_all_sequences_empty_gives_zeros(attn):
    dev = torch.device("cuda")
    q, kc, vc = decode_inputs(43, 4, 16, 4, 256, 64, dev)
    seq = torch.zeros(4, dtype=torch.int32, device=dev)
    o, ws = attn.decode_varlen(q, kc, vc, seq)
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0
    assert ws[:8].view(torch.int32).tolist() == [0, 512]


def test_two_calls_in_a_row_reuse_the_workspace(attn):
    dev = torch.device("cuda")
    B, Hq, Hkv, d, s_max = 3, 16, 2, 128, 4000
    q, kc, vc = decode_inputs(44, B, Hq, Hkv, s_max, d, dev)
    ws = None
    for lens in ([4000, 1, 300], [0, 4000, 2222]):
        seq = torch.tensor(lens, dtype=torch.int32, device=dev)
        o, ws = attn.decode_varlen(q, kc, vc, seq, workspace=ws)
        torch.cuda.synchronize()
        o_ref, _ = oracle.decode(to64(q), to64(kc), to64(vc), lens, d ** -0.5)
        assert_close(to64(o), o_ref, what=f"{lens}")


def test_many_users_per_plan_thread(attn):
    """600 users: the plan kernel's threads each take several sequences."""
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(45)
    lens = torch.randint(0, 700, (600,), generator=g).tolist()
    lens[7] = 0
    lens[599] = 700
    B, Hq, Hkv, d, s_max = len(lens), 8, 2, 64, 700
    q, kc, vc = decode_inputs(46, B, Hq, Hkv, s_max, d, dev)
    seq = torch.tensor(lens, dtype=torch.int32, device=dev)
    o, ws = attn.decode_varlen(q, kc, vc, seq)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    c_ref, items_ref = oracle.varlen_plan(lens, s_max, Hkv, _target())
    head = ws[:8].view(torch.int32).tolist()
    assert head == [len(items_ref), c_ref]
    o_ref, _ = oracle.decode(to64(q), to64(kc), to64(vc), lens, d ** -0.5)
    assert_close(to64(o), o_ref, what="600 users")


BENCH_WORKLOADS = [
    # the ragged workloads the benchmark times (Hq=64, Hkv=8, d=128): name, s_max, seqlens
    ("one 64K user + 15 of 2K", 65536, [65536] + [2048] * 15),
    ("64 users uniform in [1, 16K]", 16384, None),  # lengths drawn from a seeded generator
    ("8 users of 32K", 32768, [32768] * 8),
]


@pytest.mark.parametrize("name,s_max,lens", BENCH_WORKLOADS)
def test_benchmark_workloads_every_element(attn, name, s_max, lens):
    """Every output element of the benchmark's ragged workloads against the
    oracle, one user at a time (only that user's keys are widened to fp64;
    users run on a thread pool, the oracle's C calls release the interpreter
    lock); the device work list equals the oracle's plan."""
    import gc
    from concurrent.futures import ThreadPoolExecutor
    dev = torch.device("cuda")
    Hq, Hkv, d = 64, 8, 128
    if lens is None:
        g = torch.Generator().manual_seed(47)
        lens = torch.randint(1, s_max + 1, (64,), generator=g).tolist()
    B = len(lens)
    q, kc, vc = decode_inputs(48, B, Hq, Hkv, s_max, d, dev)
    seq = torch.tensor(lens, dtype=torch.int32, device=dev)
    try:
        o, ws = attn.decode_varlen(q, kc, vc, seq)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == attn.ATTN_OK
        c_ref, items_ref = oracle.varlen_plan(lens, s_max, Hkv, _target())
        assert ws[:8].view(torch.int32).tolist() == [len(items_ref), c_ref]
        o64, q64 = to64(o), to64(q)

        def user(b):
            n = lens[b]
            kb = kc[b, :, :n].double().cpu().numpy()
            vb = vc[b, :, :n].double().cpu().numpy()
            o_ref, _ = oracle.decode(q64[b:b + 1], kb[None], vb[None], [n], d ** -0.5)
            return b, o_ref

        with ThreadPoolExecutor(max_workers=min(8, oracle.default_threads())) as pool:
            for b, o_ref in pool.map(user, range(B)):
                assert_close(o64[b:b + 1], o_ref, what=f"{name}: user {b}, {lens[b]} keys")
    finally:
        del q, kc, vc
        gc.collect()
        torch.cuda.empty_cache()


def test_timeout_is_reported_and_recovered(attn):
    """With a wait limit of zero the work-list decode gives up at its first
    unsatisfied wait (the planner and the merge have none), the status reads
    ATTN_ERR_TIMEOUT, and the next call matches the oracle."""
    dev = torch.device("cuda")
    lens = [3000, 0, 17, 2500]
    B, Hq, Hkv, d, s_max = len(lens), 16, 2, 128, 3000
    q, kc, vc = decode_inputs(49, B, Hq, Hkv, s_max, d, dev)
    seq = torch.tensor(lens, dtype=torch.int32, device=dev)
    old = attn.attn_set_wait_timeout_ns(0)
    try:
        attn.decode_varlen(q, kc, vc, seq)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == attn.ATTN_ERR_TIMEOUT
    finally:
        attn.attn_set_wait_timeout_ns(old)
    o, _ = attn.decode_varlen(q, kc, vc, seq)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    o_ref, _ = oracle.decode(to64(q), to64(kc), to64(vc), lens, d ** -0.5)
    assert_close(to64(o), o_ref, what="varlen after timeout")
