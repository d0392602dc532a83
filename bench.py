"""Benchmark of the attention hot path on GB300 (one JSON line on stdout).

A step is one pass of the whole hot path over one batch of synthetic input:
one forward (prefill) call on the largest MHA workload (B=1, H=128, d=128,
N=131072, non-causal, head-first order) and one split-KV decode call on the
largest GQA decode workload (B=32, Hq=64, Hkv=8, d=128, 131072 cached keys
per sequence).  ``value`` is the forward TFLOP/s (4*B*H*N^2*d algorithmic
flops per call / the call's CUDA-event time); the decode figures are
reported in the ``decode`` object.  Inputs are larger than L2 (16 GiB and
17 GB), so no flush is needed between steps.

``--impl reference`` times the fp64 CPU oracle instead (on a bounded sample
of the same forward workload: a number of query rows of one head), reported
in the same unit.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (% BF16 peak); GQA decode KV GB/s (% HBM) and us/step"
FWD = dict(B=1, H=128, N=131072, d=128, causal=False)
DEC = dict(B=32, Hq=64, Hkv=8, S=131072, d=128)


# DRAM bytes (read + write) per launch measured with ncu for the kernels as
# they stand in the listed sources (profiles/ holds the summaries and the
# commands).  Each capture is one launch of a reduced case of the bench's
# workload -- fewer query heads at the same N for the forward, fewer
# sequences at the same cache length and split count for decode -- and is
# scaled to the bench's launch by the units it processes (heads, sequences):
# each head's K/V stream and each sequence's cache are read independently of
# the others, so the traffic grows in proportion.  A value is reported only
# while the sources hash to the recorded digest; after any change to them the
# bench reports null until re-captured.
MEASURED_TRAFFIC = {
    "fwd": {"files": ["fwd_sm103.cu", "fwd_kernel.cuh", "sm103_ptx.cuh", "tile_order.cuh"],
            "sha256": "626ffe5cb89f1d68ca23e7c4ef3fb4fdac10b19be70ad8e3701681b0a63a40c2",
            # MHA B=1 d=128 non-causal, head-first, H = Hq = Hkv = 16 at N = 131072
            # (one-pass capture of dram__bytes_read.sum + dram__bytes_write.sum)
            "capture": {"B": 1, "H": 16, "N": 131072, "d": 128, "causal": False,
                        "order": "head_first", "bytes": 6157949440 + 607378944}},
    "decode": {"files": ["decode_sm103.cu", "sm103_ptx.cuh"],
               "sha256": "6f39ea2abaa39f9696161823dd1c557c1c34c647d8e0f320046c8e0792c4e869",
               # GQA decode Hq=64 Hkv=8 d=128, B=4 sequences of 131072 keys, 2 splits
               # (the heuristic's count at B=32), decode kernel only
               "capture": {"B": 4, "S": 131072, "splits": 2, "bytes": 2147686144 + 3055104}},
}


def measured_traffic(kind):
    """The ncu-measured traffic entry for `kind` if the kernel sources are
    unchanged since the capture, else None."""
    import hashlib
    entry = MEASURED_TRAFFIC[kind]
    if entry["sha256"] is None or entry["capture"]["bytes"] is None:
        return None
    h = hashlib.sha256()
    for f in entry["files"]:
        with open(os.path.join(ROOT, "attention_fa2_fwd_sm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return entry["capture"] if h.hexdigest() == entry["sha256"] else None


def fwd_traffic(B, H, N, d, causal, order):
    """DRAM bytes per forward launch of an MHA problem (Hq = Hkv = H), scaled
    from the reduced-head capture by B * H; None when no capture applies."""
    c = measured_traffic("fwd")
    if not c or (N, d, bool(causal), order) != (c["N"], c["d"], c["causal"], c["order"]):
        return None
    return round(c["bytes"] * (B * H) / (c["B"] * c["H"]))


def decode_traffic(B, S, splits):
    """DRAM bytes per decode-kernel launch, scaled from the reduced-batch
    capture by B; None when no capture applies."""
    c = measured_traffic("decode")
    if not c or (S, splits) != (c["S"], c["splits"]):
        return None
    return round(c["bytes"] * B / c["B"])


def fwd_flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks of the default
    process group (the values unchanged when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in values]
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replica_throughput(work_per_rank, world, seconds):
    """Whole-job throughput of `world` independent replicas that each did
    `work_per_rank` in at most `seconds` (the slowest rank's time)."""
    return world * work_per_rank / seconds


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_gpu(args):
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    from synthetic_inputs import decode_inputs, prefill_inputs

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or ws > 1:
        _build.build()
    attn.lib()

    B, H, N, d, causal = FWD["B"], FWD["H"], args.n, FWD["d"], FWD["causal"]
    order = attn.ORDERS[args.order]
    q, k, v = prefill_inputs(11, B, H, H, N, d, dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(d)
    Bd, Hq, Hkv, S, dd = args.dec_batch, DEC["Hq"], DEC["Hkv"], args.dec_len, DEC["d"]
    qd, kc, vc = decode_inputs(70, Bd, Hq, Hkv, S, dd, dev)
    seqlens = torch.full((Bd,), S, dtype=torch.int32, device=dev)
    splits = attn.attn_decode_num_splits(Bd, Hq, Hkv, S)
    wbytes = attn.attn_decode_workspace_bytes(Bd, Hq, dd, splits)
    wsp = torch.empty(max(wbytes, 16), dtype=torch.uint8, device=dev)
    od = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    dscale = 1.0 / math.sqrt(dd)

    def prefill():
        attn.check(attn.attn_fwd_ex(q, k, v, o, lse, B, H, H, N, d, scale, causal, order, sh), "attn_fwd")

    def decode():
        attn.check(attn.attn_decode(qd, kc, vc, seqlens, od, Bd, Hq, Hkv, dd, dscale, splits, S, wsp,
                                    wbytes, sh), "attn_decode")

    def barrier():
        torch.cuda.synchronize(dev)
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        prefill()
        decode()
    barrier()
    attn.check(attn.attn_device_status(sh), "warm-up status")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(K):
            ev[i][0].record(stream)
            prefill()
            ev[i][1].record(stream)
            decode()
            ev[i][2].record(stream)
        end.record(stream)
        barrier()
    attn.check(attn.attn_device_status(sh), "timed-region status")
    total_ms = start.elapsed_time(end)
    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]

    total_ms, fwd_sum, dec_sum = max_over_ranks([total_ms, sum(fwd_ms), sum(dec_ms)], dev)

    flops = fwd_flops(B, H, N, d, causal)
    fwd_avg_s = fwd_sum / K / 1e3
    value = replica_throughput(flops, ws, fwd_avg_s) / 1e12
    peaks, peak_src = load_peaks()
    per_gpu = flops / fwd_avg_s / 1e12
    dec_bytes = 2 * Bd * Hkv * S * dd * 2 + 2 * Bd * Hq * dd * 2
    dec_avg_s = dec_sum / K / 1e3
    dec_gbs = dec_bytes / dec_avg_s / 1e9

    fwd_bytes = fwd_traffic(B, H, N, d, causal, args.order)
    long_step = fwd_avg_s * K >= 4.0  # the forward alone keeps the GPU busy for seconds
    if long_step and peaks.get("bf16_tflops_sustained"):
        peak_fwd, peak_kind = peaks["bf16_tflops_sustained"], "sustained (the forward runs back to back for seconds)"
    else:
        peak_fwd, peak_kind = peaks["bf16_tflops"], "burst"
    dec_traffic = decode_traffic(Bd, S, splits)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"MHA forward B={B} H={H} N={N} d={d} non-causal, {args.order} order"
                               f" + GQA decode B={Bd} Hq={Hq} Hkv={Hkv} S={S} d={dd}",
                   "B": B, "H": H, "seq_len": N, "head_dim": d, "causal": causal,
                   "tile_order": args.order, "decode_batch": Bd, "decode_kv_len": S,
                   "decode_splits": splits, "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2 (no flush)"},
        # The forward runs back to back for the whole timed region (about 0.8 s a
        # launch at N = 131072, tens of seconds in all, under the power cap), so
        # its denominator is the sustained bf16 figure; the burst fraction is
        # reported beside it.
        "roofline": {"bound": "tensor", "achieved": round(per_gpu, 2),
                     "peak": peak_fwd, "unit": "TFLOP/s",
                     "frac": round(per_gpu / peak_fwd, 4), "traffic": fwd_bytes,
                     "peak_source": f"{peak_src} bf16 {peak_kind}", "kernel": "fwd_kernel<128, 0>",
                     "frac_of_burst": round(per_gpu / peaks["bf16_tflops"], 4),
                     "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch "
                                        "with fewer heads at the same N, scaled by the head count"
                                        if fwd_bytes else None)},
        "decode": {"value": round(dec_gbs, 1), "unit": "GB/s", "us_per_step": round(dec_avg_s * 1e6, 2),
                   "frac_hbm": round(dec_gbs / peaks["hbm_gbs"], 4), "hbm_peak_gbs": peaks["hbm_gbs"],
                   "bytes_per_step": dec_bytes, "traffic": dec_traffic},
        "gpu_launches": K * (1 + (2 if splits > 1 else 1)),
        "clocks": clk.summary(),
    }

    # -- tile-order ablation (same workload, each order timed alone) --
    if args.ablation and rank == 0:
        abl = {}
        for name, oid in attn.ORDERS.items():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            attn.check(attn.attn_fwd_ex(q, k, v, o, lse, B, H, H, N, d, scale, causal, oid, sh), "warm")
            reps = 2 if N >= 131072 else 3
            e0.record(stream)
            for _ in range(reps):
                attn.check(attn.attn_fwd_ex(q, k, v, o, lse, B, H, H, N, d, scale, causal, oid, sh), "abl")
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / reps
            abl[name] = {"ms": round(ms, 3), "tflops": round(flops / (ms / 1e3) / 1e12, 2)}
        result["ablation"] = abl
        # 1 warm-up + the timed launches per order (plus the die map's one-off probe)
        result["gpu_launches_ablation"] = (1 + reps) * len(attn.ORDERS)

    # -- end to end through the C ABI with host buffers --
    if args.e2e and rank == 0:
        def pinned_copy(t):  # straight into page-locked memory (no pageable intermediate)
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            return h
        hq_, hk_, hv_ = (pinned_copy(t) for t in (q, k, v))
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        wbytes_h = attn.attn_fwd_host_workspace_bytes(B, H, H, N, d, 0)
        ws_h = torch.empty(wbytes_h, dtype=torch.uint8, device=dev)
        # the library's default chunk: the fewest KV heads holding 304 work units (256 rows of a head)
        gc = max(1, min(-(-304 // -(-N // 256)), H))
        chunks = B * -(-H // gc)
        reps = max(2, min(K, 5))

        def e2e_step():
            attn.check(attn.attn_fwd_host(hq_, hk_, hv_, ho, hl, B, H, H, N, d, scale, causal, order, 0,
                                          ws_h, wbytes_h, sh), "e2e")

        e2e_step()
        torch.cuda.synchronize(dev)
        with ClockSampler(local) as e2e_clk:
            # events between the calls (on the calls' own stream) give each
            # call's device-side span without synchronising the host
            marks = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
            t0 = time.perf_counter()
            marks[0].record(stream)
            for i in range(reps):
                e2e_step()
                marks[i + 1].record(stream)
            torch.cuda.synchronize(dev)
            e2e_s = (time.perf_counter() - t0) / reps
        per_call_ms = [round(marks[i].elapsed_time(marks[i + 1]), 3) for i in range(reps)]
        attn.check(attn.attn_device_status(sh), "e2e status")
        result["e2e"] = {"value": round(flops / e2e_s / 1e12, 2), "unit": "TFLOP/s",
                         "h2d_bytes_per_step": 3 * q.numel() * 2,
                         "d2h_bytes_per_step": o.numel() * 2 + lse.numel() * 4,
                         "steps": reps, "ms_per_step": round(e2e_s * 1e3, 3), "per_call_ms": per_call_ms,
                         # the SM clock while these calls ran: the e2e loop comes after
                         # seconds of forward work, later than the step's own samples
                         "clocks": e2e_clk.summary(),
                         "api": "attn_fwd_host (C ABI): pinned host buffers, copies overlapped with the"
                                " kernels in chunks of KV heads"}
        result["gpu_launches_e2e"] = (reps + 1) * chunks
        # The same bytes moved with no kernels, inputs in and outputs out on two
        # streams as the pipeline overlaps them: when this approaches
        # ms_per_step, the host link and not the kernels sets the pace.
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def copies():
            with torch.cuda.stream(s_in):
                for dst, src in ((q, hq_), (k, hk_), (v, hv_)):
                    dst.copy_(src, non_blocking=True)
            with torch.cuda.stream(s_out):
                ho.copy_(o, non_blocking=True)
                hl.copy_(lse, non_blocking=True)

        copies()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(2):
            copies()
        torch.cuda.synchronize(dev)
        copy_ms = (time.perf_counter() - t0) / 2 * 1e3
        result["e2e"]["copy_only_ms"] = round(copy_ms, 3)
        # One more call with the library's per-chunk timeline switched on.
        attn.check(attn.attn_fwd_host_trace(1), "trace on")
        try:
            e2e_step()
            timeline = attn.attn_fwd_host_trace_read()
        finally:
            attn.check(attn.attn_fwd_host_trace(0), "trace off")
        result["e2e"]["timeline"] = timeline_summary(timeline, copy_ms)
        result["gpu_launches_e2e"] += chunks

    if args.cpu_baseline and rank == 0:
        result["cpu_baseline"] = cpu_baseline(q, k, v, scale, causal, args.cpu_seconds)

    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result if rank == 0 else None


def timeline_summary(tl, copy_only_ms):
    """Summary of an attn_fwd_host timeline (per chunk: copy-in done, kernel
    reached, kernel done, copy-out done; ms from the call's start).
    kernel_busy_ms is the union of the chunks' kernel intervals, idle_ms the
    rest of the call, and overlap_frac the share of the copy-only time that
    the call hid behind its kernels: (kernel_busy + copy_only - wall) /
    copy_only."""
    wall = max(t[3] for t in tl)
    spans = sorted((t[1], t[2]) for t in tl)
    busy, cur_s, cur_e, gaps = 0.0, None, None, []
    for s, e in spans:
        if cur_e is None or s > cur_e:
            if cur_e is not None:
                busy += cur_e - cur_s
                gaps.append(s - cur_e)
            cur_s, cur_e = s, e
        else:
            cur_e = max(cur_e, e)
    busy += cur_e - cur_s
    kernel_sum = sum(t[2] - t[1] for t in tl)
    waits_on_copy = sum(max(0.0, tl[c][0] - tl[c - 1][2]) for c in range(1, len(tl)))
    return {"chunks": len(tl), "wall_ms": round(wall, 3), "kernel_busy_ms": round(busy, 3),
            "kernel_ms_sum": round(kernel_sum, 3), "idle_ms": round(wall - busy, 3),
            "first_kernel_ms": round(spans[0][0], 3), "after_last_kernel_ms": round(wall - cur_e, 3),
            "max_gap_ms": round(max(gaps), 3) if gaps else 0.0,
            "copy_in_late_ms": round(waits_on_copy, 3),
            "overlap_frac": round(max(0.0, min(1.0, (busy + copy_only_ms - wall) / copy_only_ms)), 4)
            if copy_only_ms > 0 else None}


def _oracle_sample_rate(q_rows, k_head, v_head, scale, causal, positions, budget_s):
    """Time the oracle on growing row counts until the budget is spent."""
    import numpy as np

    import oracle
    oracle.build()
    threads = oracle.default_threads()
    N, d = k_head.shape
    rows_done, secs = 0, 0.0
    step = max(threads, 16)
    total_rows = q_rows.shape[0]
    i = 0
    while secs < budget_s and i < total_rows:
        n = min(step, total_rows - i)
        t0 = time.perf_counter()
        oracle.attention_rows(q_rows[i:i + n], k_head, v_head, scale, causal, positions[i:i + n])
        secs += time.perf_counter() - t0
        rows_done += n
        i += n
        step = min(step * 2, 4096)
    flops_per_row = 4.0 * N * d
    return rows_done, secs, rows_done * flops_per_row / secs / 1e12, threads


def cpu_baseline(q, k, v, scale, causal, budget_s):
    """The fp64 oracle as it stands, on rows of head 0 of the same workload."""
    import numpy as np
    N = q.shape[2]
    rows = N
    positions = np.arange(rows, dtype=np.int64)
    qh = q[0, 0, :rows].double().cpu().numpy()
    kh = k[0, 0].double().cpu().numpy()
    vh = v[0, 0].double().cpu().numpy()
    n_rows, secs, tflops, threads = _oracle_sample_rate(qh, kh, vh, scale, causal, positions, budget_s)
    return {"value": round(tflops, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_rows} query rows of head 0 (N={N}, d={q.shape[3]}) in {secs:.1f} s; "
                      f"rate extrapolated to the whole call"}


def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores (rank 0 only)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import numpy as np
    import torch

    from synthetic_inputs import prefill_inputs
    B, H, N, d, causal = FWD["B"], FWD["H"], args.n, FWD["d"], FWD["causal"]
    # only head 0 is needed for the sample: draw the same tensors on the CPU
    q, k, v = prefill_inputs(11, B, 1, 1, N, d, "cpu")
    scale = 1.0 / math.sqrt(d)
    rows = min(N, 8192)
    qh = q[0, 0, :rows].double().numpy()
    kh, vh = k[0, 0].double().numpy(), v[0, 0].double().numpy()
    pos = np.arange(rows, dtype=np.int64)
    per_step = max(1.0, args.ref_seconds)
    for _ in range(args.warmup):
        _oracle_sample_rate(qh, kh, vh, scale, causal, pos, per_step / 4)
    rates, total_s, total_rows, threads = [], 0.0, 0, 1
    for _ in range(args.steps):
        n, s, r, threads = _oracle_sample_rate(qh, kh, vh, scale, causal, pos, per_step)
        rates.append(r)
        total_s += s
        total_rows += n
    value = statistics.mean(rates)
    flops_call = fwd_flops(B, H, N, d, causal)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_s / args.steps * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"MHA forward B={B} H={H} N={N} d={d} non-causal (fp64 oracle, "
                               f"sampled rows of head 0)", "B": B, "H": H, "seq_len": N,
                   "head_dim": d, "causal": causal},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{total_rows} query rows over {args.steps} steps; a whole call "
                                   f"({flops_call:.3g} flop) would take {flops_call / value / 1e12:.3g} s"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _l2_flush_buffer(torch, dev):
    """A buffer twice the L2 size; writing it evicts the previous call's data."""
    props = torch.cuda.get_device_properties(dev)
    return torch.empty(2 * max(props.L2_cache_size, 128 << 20), dtype=torch.uint8, device=dev)


def _time_calls(torch, fn, reps, flush=None, stream=None):
    """Median CUDA-event time (ms) of ``fn`` over ``reps`` calls, each after an
    optional L2 flush outside the events."""
    times = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def run_decode_sweep(args):
    """Decode configurations (H_Q=64, H_KV=8, d=128; batch x KV length) with
    num_splits swept; one JSON line per configuration."""
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    from synthetic_inputs import decode_inputs
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    flush = _l2_flush_buffer(torch, dev)
    stream = torch.cuda.current_stream(dev)
    Hq, Hkv, d = DEC["Hq"], DEC["Hkv"], DEC["d"]
    for B in (1, 8, 32):
        for S in (8192, 32768, 131072):
            q, kc, vc = decode_inputs(70, B, Hq, Hkv, S, d, dev)
            seqlens = torch.full((B,), S, dtype=torch.int32, device=dev)
            o = torch.empty_like(q)
            nbytes = 2 * B * Hkv * S * d * 2 + 2 * B * Hq * d * 2
            heur = attn.attn_decode_num_splits(B, Hq, Hkv, S)
            cands = sorted({1, 2, 3, 4, 5, 6, 8, 12, 16, 19, 24, 32, 38, 48, 64, heur})
            res = {}
            for sp in cands:
                if sp > 1 and -(-S // sp) < 64:
                    continue
                wb = attn.attn_decode_workspace_bytes(B, Hq, d, sp)
                ws = torch.empty(max(wb, 16), dtype=torch.uint8, device=dev)
                fn = lambda: attn.check(attn.attn_decode(q, kc, vc, seqlens, o, B, Hq, Hkv, d, d ** -0.5,
                                                         sp, S, ws, wb, stream.cuda_stream), "decode")
                for _ in range(3):
                    fn()
                ms = _time_calls(torch, fn, args.steps, flush, stream)
                res[sp] = {"us": round(ms * 1e3, 2), "gbs": round(nbytes / (ms / 1e3) / 1e9, 1)}
            best = max(res, key=lambda k: res[k]["gbs"])
            print(json.dumps({"mode": "decode-sweep", "B": B, "S": S, "bytes": nbytes,
                              "heuristic_splits": heur, "heuristic": res.get(heur),
                              "best_splits": best, "best": res[best],
                              "frac_hbm_best": round(res[best]["gbs"] / peaks["hbm_gbs"], 4),
                              "splits": res, "l2": "flushed before every call"}), flush=True)
            del q, kc, vc
            torch.cuda.empty_cache()


def run_fwd_sweep(args):
    """Forward configurations of the pages' sweeps, each with every tile
    order; one JSON line per configuration."""
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    from synthetic_inputs import prefill_inputs
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    stream = torch.cuda.current_stream(dev)
    configs = []
    for N in (8192, 32768, 131072):
        configs.append(("mha", 1, 128, 128, N, 128, False))
    for N in (8192, 32768, 131072):
        for causal in (False, True):
            configs.append(("gqa", 1, 64, 8, N, 128, causal))
    for N in (32768, 131072):
        configs.append(("deepseek", 1, 128, 128, N, 56, True))
    for name, B, Hq, Hkv, N, d, causal in configs:
        q, k, v = prefill_inputs(11, B, Hq, Hkv, N, d, dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
        flops = fwd_flops(B, Hq, N, d, causal)
        out = {"mode": "fwd-sweep", "config": name, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d,
               "causal": causal, "flops": flops}
        reps = 3 if N >= 131072 else args.steps
        for oname, oid in attn.ORDERS.items():
            fn = lambda: attn.check(attn.attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, d, d ** -0.5, causal,
                                                     oid, stream.cuda_stream), "fwd")
            fn()
            ms = _time_calls(torch, fn, reps, None, stream)
            tf = flops / (ms / 1e3) / 1e12
            out[oname] = {"ms": round(ms, 3), "tflops": round(tf, 1),
                          "frac": round(tf / peaks["bf16_tflops"], 4)}
            if d == 56:
                out[oname]["tflops_padded_d64"] = round(tf * 64 / 56, 1)
        if d == 128:
            # the CTA-pair scheme (cta_group::2) in the head-first and block-first orders
            for oname in ("head_first", "block_first"):
                oid = attn.ORDERS[oname] | attn.FWD_CTA_PAIR
                fn = lambda: attn.check(attn.attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, d, d ** -0.5, causal,
                                                         oid, stream.cuda_stream), "fwd pair")
                fn()
                ms = _time_calls(torch, fn, reps, None, stream)
                tf = flops / (ms / 1e3) / 1e12
                out["pair_" + oname] = {"ms": round(ms, 3), "tflops": round(tf, 1),
                                        "frac": round(tf / peaks["bf16_tflops"], 4)}
        print(json.dumps(out), flush=True)
        del q, k, v, o, lse
        torch.cuda.empty_cache()


def run_fwd_one(args):
    """One forward configuration in one tile order: W warm-up launches, then K
    timed launches (median); one JSON line.  Used for per-configuration
    profiles (the sizes are flags)."""
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    from synthetic_inputs import prefill_inputs
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    stream = torch.cuda.current_stream(dev)
    B, Hq, Hkv, N, d, causal = args.batch, args.hq, args.hkv, args.n, args.head_dim, args.causal
    q, k, v = prefill_inputs(12, B, Hq, Hkv, N, d, dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    oid = attn.ORDERS[args.order] | attn.SCHEMES[args.scheme]
    fn = lambda: attn.check(attn.attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, d, d ** -0.5, causal, oid,
                                             stream.cuda_stream), "fwd")
    for _ in range(args.warmup):
        fn()
    ms = _time_calls(torch, fn, args.steps, None, stream)
    flops = fwd_flops(B, Hq, N, d, causal)
    tf = flops / (ms / 1e3) / 1e12
    print(json.dumps({"mode": "fwd-one", "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "causal": causal,
                      "order": args.order, "scheme": args.scheme, "ms": round(ms, 4), "tflops": round(tf, 1),
                      "frac": round(tf / peaks["bf16_tflops"], 4), "launches": args.warmup + args.steps}),
          flush=True)


def run_fwd_splitkv(args):
    """The sub-ACC split (attn_fwd_splitkv) against the plain head-first
    forward on the long configurations: MHA and causal GQA at N = 131072
    (d = 128) and the DeepSeek-like d = 56 causal one; W warm-up calls, then
    K timed calls (median).  One JSON line per configuration."""
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    from synthetic_inputs import prefill_inputs
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    stream = torch.cuda.current_stream(dev)
    configs = [("mha", 1, 128, 128, 131072, 128, False), ("gqa", 1, 64, 8, 131072, 128, True),
               ("deepseek", 1, 128, 128, 131072, 56, True)]
    if args.hq != FWD["H"] or args.n != FWD["N"]:  # one configuration from the flags
        configs = [("one", args.batch, args.hq, args.hkv, args.n, args.head_dim, args.causal)]
    for name, B, Hq, Hkv, N, d, causal in configs:
        q, k, v = prefill_inputs(12, B, Hq, Hkv, N, d, dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
        flops = fwd_flops(B, Hq, N, d, causal)
        out = {"mode": "fwd-splitkv", "config": name, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "causal": causal}
        fn = lambda: attn.check(attn.attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, d, d ** -0.5, causal, 0,
                                                 stream.cuda_stream), "fwd")
        for _ in range(args.warmup):
            fn()
        ms = _time_calls(torch, fn, args.steps, None, stream)
        out["plain"] = {"ms": round(ms, 3), "tflops": round(flops / (ms / 1e3) / 1e12, 1)}
        for sp in (0, 1, 2, 4, 8):
            wb = attn.attn_fwd_splitkv_workspace_bytes(B, Hq, N, d, sp)
            ws = torch.empty(wb, dtype=torch.uint8, device=dev)
            fn = lambda: attn.check(attn.attn_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, N, d, d ** -0.5, causal, sp,
                                                          ws, wb, stream.cuda_stream), "splitkv")
            for _ in range(args.warmup):
                fn()
            ms = _time_calls(torch, fn, args.steps, None, stream)
            out[f"splits{sp}"] = {"ms": round(ms, 3), "tflops": round(flops / (ms / 1e3) / 1e12, 1),
                                  "workspace_gb": round(wb / 1e9, 2)}
            del ws
            torch.cuda.empty_cache()
        print(json.dumps(out), flush=True)
        del q, k, v, o, lse
        torch.cuda.empty_cache()


def bwd_flops(B, H, N, d, causal):
    """Algorithmic backward work: five products of 2*N*N*d per head (dV, dP,
    dK, dQ and the recomputed S), half of that causal."""
    f = 10.0 * B * H * N * N * d
    return f / 2 if causal else f


def run_bwd_one(args):
    """The backward pass of one configuration in one tile order: W warm-up
    calls, then K timed calls (median); one JSON line."""
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    from synthetic_inputs import output_grad, prefill_inputs
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    stream = torch.cuda.current_stream(dev)
    B, Hq, Hkv, N, d, causal = args.batch, args.hq, args.hkv, args.n, args.head_dim, args.causal
    if args.order not in ("head_first", "block_first", "naive_head_first"):
        raise SystemExit("the backward pass takes head_first, block_first or naive_head_first")
    q, k, v = prefill_inputs(13, B, Hq, Hkv, N, d, dev)
    dout = output_grad(13, B, Hq, N, d, dev)
    o, lse = attn.forward(q, k, v, causal=causal, scale=d ** -0.5)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = attn.attn_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, causal)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    oid = attn.ORDERS[args.order]
    fn = lambda: attn.check(attn.attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, d ** -0.5,
                                          causal, oid, ws, nbytes, stream.cuda_stream), "bwd")
    for _ in range(args.warmup):
        fn()
    ms = _time_calls(torch, fn, args.steps, None, stream)
    tf = bwd_flops(B, Hq, N, d, causal) / (ms / 1e3) / 1e12
    print(json.dumps({"mode": "bwd-one", "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "causal": causal,
                      "order": args.order, "ms": round(ms, 4), "tflops": round(tf, 1),
                      "frac": round(tf / peaks["bf16_tflops"], 4),
                      # pre-pass, dK/dV, dQ; plus the partials' sum when the dK/dV pass splits
                      "launches_per_call": 3 + int(nbytes > attn.attn_bwd_workspace_bytes(B, Hq, N)),
                      "calls": args.warmup + args.steps}), flush=True)


def run_decode_one(args):
    """GQA decode (Hq=64, Hkv=8, d=128) of one batch size and KV length with
    the heuristic's split count (or --dec-splits): W warm-up calls, then K
    timed calls (median), the L2 flushed before each; one JSON line."""
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    from synthetic_inputs import decode_inputs
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    flush = _l2_flush_buffer(torch, dev)
    stream = torch.cuda.current_stream(dev)
    Hq, Hkv, d = DEC["Hq"], DEC["Hkv"], DEC["d"]
    B, S = args.dec_batch, args.dec_len
    q, kc, vc = decode_inputs(70, B, Hq, Hkv, S, d, dev)
    seqlens = torch.full((B,), S, dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    sp = args.dec_splits if args.dec_splits > 0 else attn.attn_decode_num_splits(B, Hq, Hkv, S)
    wb = attn.attn_decode_workspace_bytes(B, Hq, d, sp)
    ws = torch.empty(max(wb, 16), dtype=torch.uint8, device=dev)
    fn = lambda: attn.check(attn.attn_decode(q, kc, vc, seqlens, o, B, Hq, Hkv, d, d ** -0.5, sp, S, ws, wb,
                                             stream.cuda_stream), "decode")
    for _ in range(args.warmup):
        fn()
    ms = _time_calls(torch, fn, args.steps, flush, stream)
    nbytes = 2 * B * Hkv * S * d * 2 + 2 * B * Hq * d * 2
    gbs = nbytes / (ms / 1e3) / 1e9
    print(json.dumps({"mode": "decode-one", "B": B, "S": S, "Hq": Hq, "Hkv": Hkv, "d": d, "splits": sp,
                      "us": round(ms * 1e3, 2), "gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                      "l2": "flushed before every call"}), flush=True)


def run_decode_floor(args):
    """What bounds the short decode configurations: each (B, S) timed as is,
    with every sequence empty (the same grid and merge, no keys to read),
    with 64 keys per sequence (one ring stage per CTA that has keys), and the
    same three with one split (one kernel, no merge).  The L2 is flushed
    before every call; one JSON line per configuration."""
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    from synthetic_inputs import decode_inputs
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    flush = _l2_flush_buffer(torch, dev)
    stream = torch.cuda.current_stream(dev)
    Hq, Hkv, d = DEC["Hq"], DEC["Hkv"], DEC["d"]
    for B, S in ((1, 8192), (1, 32768), (8, 8192), (8, 32768)):
        q, kc, vc = decode_inputs(70, B, Hq, Hkv, S, d, dev)
        o = torch.empty_like(q)
        heur = attn.attn_decode_num_splits(B, Hq, Hkv, S)
        out = {"mode": "decode-floor", "B": B, "S": S, "heuristic_splits": heur,
               "bytes": 2 * B * Hkv * S * d * 2 + 2 * B * Hq * d * 2}
        for sp in (heur, 1):
            wb = attn.attn_decode_workspace_bytes(B, Hq, d, sp)
            ws = torch.empty(max(wb, 16), dtype=torch.uint8, device=dev)
            for name, n in (("full", S), ("one_stage", 64), ("empty", 0)):
                seq = torch.full((B,), n, dtype=torch.int32, device=dev)
                fn = lambda: attn.check(attn.attn_decode(q, kc, vc, seq, o, B, Hq, Hkv, d, d ** -0.5, sp, S, ws, wb,
                                                         stream.cuda_stream), "decode")
                for _ in range(args.warmup):
                    fn()
                out[f"{name}_splits{sp}_us"] = round(_time_calls(torch, fn, args.steps, flush, stream) * 1e3, 2)
        # the same flush and events around a one-element torch fill: the floor of any launch here
        one = torch.empty(1, dtype=torch.int32, device=dev)
        fill = lambda: one.fill_(1)
        for _ in range(args.warmup):
            fill()
        out["trivial_kernel_us"] = round(_time_calls(torch, fill, args.steps, flush, stream) * 1e3, 2)
        out["full_gbs"] = round(out["bytes"] / (out[f"full_splits{heur}_us"] * 1e-6) / 1e9, 1)
        out["frac_hbm"] = round(out["full_gbs"] / peaks["hbm_gbs"], 4)
        print(json.dumps(out), flush=True)
        del q, kc, vc
        torch.cuda.empty_cache()


def run_decode_varlen(args):
    """Ragged multi-user decode batches (GQA Hq=64, Hkv=8, d=128): attn_decode
    (split count from max_seqlen) against attn_decode_varlen (chunks from the
    total attended keys).  GB/s counts the attended K/V bytes plus q and o."""
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    from synthetic_inputs import decode_inputs
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    stream = torch.cuda.current_stream(dev)
    Hq, Hkv, d = 64, 8, 128
    g = torch.Generator().manual_seed(77)
    workloads = [
        ("one 64K user + 15 users of 2K", 65536, [65536] + [2048] * 15),
        ("64 users, lengths uniform in [1, 16K]", 16384, torch.randint(1, 16385, (64,), generator=g).tolist()),
        ("8 users of 32K (equal lengths)", 32768, [32768] * 8),
    ]
    for name, s_max, lens in workloads:
        B = len(lens)
        q, kc, vc = decode_inputs(14, B, Hq, Hkv, s_max, d, dev)
        seq = torch.tensor(lens, dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        nbytes = sum(lens) * Hkv * d * 2 * 2 + 2 * B * Hq * d * 2
        splits = attn.attn_decode_num_splits(B, Hq, Hkv, s_max)
        ws_s = torch.empty(max(attn.attn_decode_workspace_bytes(B, Hq, d, splits), 16), dtype=torch.uint8,
                           device=dev)
        ws_v = torch.empty(max(attn.attn_decode_varlen_workspace_bytes(B, Hq, Hkv, d), 16), dtype=torch.uint8,
                           device=dev)
        split_fn = lambda: attn.check(attn.attn_decode(q, kc, vc, seq, o, B, Hq, Hkv, d, d ** -0.5, splits, s_max,
                                                       ws_s, ws_s.numel(), stream.cuda_stream), "decode")
        varlen_fn = lambda: attn.check(attn.attn_decode_varlen(q, kc, vc, seq, o, B, Hq, Hkv, d, d ** -0.5, s_max,
                                                               ws_v, ws_v.numel(), stream.cuda_stream), "varlen")
        out = {"mode": "decode-varlen", "workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d,
               "attended_keys": sum(lens), "bytes": nbytes}
        for key, fn in (("split", split_fn), ("varlen", varlen_fn)):
            for _ in range(args.warmup):
                fn()
            us = _time_calls(torch, fn, args.steps, None, stream) * 1e3
            gbs = nbytes / (us * 1e-6) / 1e9
            out[key] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        out["split"]["splits"] = splits
        out["varlen"]["chunk"] = int(ws_v[4:8].view(torch.int32).item())
        out["varlen"]["chunks"] = int(ws_v[0:4].view(torch.int32).item())
        print(json.dumps(out), flush=True)
        del q, kc, vc
        torch.cuda.empty_cache()


def run_bwd_sweep(args):
    """Backward configurations (MHA, GQA causal and non-causal, DeepSeek-like
    d=56 causal) in the head-first and block-first orders; one JSON line per
    configuration."""
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    from synthetic_inputs import output_grad, prefill_inputs
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    stream = torch.cuda.current_stream(dev)
    configs = []
    for N in (8192, 32768):
        configs.append(("mha", 1, 128, 128, N, 128, False))
        for causal in (False, True):
            configs.append(("gqa", 1, 64, 8, N, 128, causal))
    configs.append(("deepseek", 1, 128, 128, 32768, 56, True))
    for name, B, Hq, Hkv, N, d, causal in configs:
        q, k, v = prefill_inputs(15, B, Hq, Hkv, N, d, dev)
        dout = output_grad(15, B, Hq, N, d, dev)
        o, lse = attn.forward(q, k, v, causal=causal, scale=d ** -0.5)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        nbytes = attn.attn_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, causal)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        flops = bwd_flops(B, Hq, N, d, causal)
        out = {"mode": "bwd-sweep", "config": name, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d,
               "causal": causal, "flops": flops}
        for oname in ("head_first", "block_first"):
            oid = attn.ORDERS[oname]
            fn = lambda: attn.check(attn.attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, d ** -0.5,
                                                  causal, oid, ws, nbytes, stream.cuda_stream), "bwd")
            for _ in range(max(1, args.warmup)):
                fn()
            ms = _time_calls(torch, fn, args.steps, None, stream)
            tf = flops / (ms / 1e3) / 1e12
            out[oname] = {"ms": round(ms, 3), "tflops": round(tf, 1), "frac": round(tf / peaks["bf16_tflops"], 4)}
        print(json.dumps(out), flush=True)
        del q, k, v, dout, o, lse, dq, dk, dv, ws
        torch.cuda.empty_cache()


def run_die_map(args):
    """The SM -> die map the die-split order uses (measured on first use) with
    its calibration statistics; one JSON line."""
    import torch

    import attention_fa2_fwd_sm_gb300 as attn
    from attention_fa2_fwd_sm_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    dies, stats = attn.attn_die_map()
    print(json.dumps({"mode": "die-map", "sms": len(dies), "die1_sms": sum(dies),
                      "measured": stats[0] == 1.0, "min_margin": round(stats[1], 3),
                      "near_clk": round(stats[2], 1), "far_clk": round(stats[3], 1),
                      "die_of_sm": "".join(str(x) for x in dies)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--mode", default="step",
                    choices=["step", "decode-sweep", "decode-one", "decode-floor", "decode-varlen", "fwd-sweep", "fwd-one",
                             "fwd-splitkv",
                             "bwd-one", "bwd-sweep", "die-map"],
                    help="step: the contract's one-line benchmark; the sweeps print one line "
                         "per configuration; fwd-one times one forward configuration")
    ap.add_argument("--batch", type=int, default=1, help="fwd-one: batch")
    ap.add_argument("--hq", type=int, default=FWD["H"], help="fwd-one: query heads")
    ap.add_argument("--hkv", type=int, default=FWD["H"], help="fwd-one: KV heads")
    ap.add_argument("--head-dim", type=int, default=FWD["d"], help="fwd-one: head dimension")
    ap.add_argument("--causal", action="store_true", help="fwd-one: causal mask")
    ap.add_argument("--n", type=int, default=FWD["N"], help="forward sequence length")
    ap.add_argument("--order", default="head_first", choices=["head_first", "block_first",
                                                              "naive_head_first",
                                                              "die_split_head_first"])
    ap.add_argument("--scheme", default="auto", choices=["auto", "single", "pair"],
                    help="fwd-one: forward tile scheme (pair: CTA pairs with cta_group::2 MMAs, d = 128)")
    ap.add_argument("--no-ablation", dest="ablation", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--dec-batch", type=int, default=DEC["B"], help="decode batch")
    ap.add_argument("--dec-len", type=int, default=DEC["S"], help="decode cached keys per sequence")
    ap.add_argument("--dec-splits", type=int, default=0, help="decode-one: split count (0: the heuristic's)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=4.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.mode == "decode-sweep":
        return run_decode_sweep(args)
    if args.mode == "fwd-sweep":
        return run_fwd_sweep(args)
    if args.mode == "fwd-one":
        return run_fwd_one(args)
    if args.mode == "die-map":
        return run_die_map(args)
    if args.mode == "bwd-one":
        return run_bwd_one(args)
    if args.mode == "decode-one":
        return run_decode_one(args)
    if args.mode == "decode-varlen":
        return run_decode_varlen(args)
    if args.mode == "decode-floor":
        return run_decode_floor(args)
    if args.mode == "fwd-splitkv":
        return run_fwd_splitkv(args)
    if args.mode == "bwd-sweep":
        return run_bwd_sweep(args)
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
