"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module draws random numbers and picks sample indices; it holds none of
the attention arithmetic, so both the CUDA path and the fp64 oracle may use
it without sharing any of the method.

Recipe (the pages' workloads are Triton FA sweeps and Llama-3 / DeepSeek-V3
shapes; no dataset is involved): every tensor is i.i.d. N(0, 1) drawn in fp32
from a seeded ``torch.Generator`` and rounded to bf16 (round to nearest even).
Seeds are ``1000 + cfg`` for Q, ``2000 + cfg`` for K, ``3000 + cfg`` for V and
``4000 + cfg`` for the output gradient dO of the backward pass.
Small cases draw on the CPU generator; large ones on the device generator of
the tensor's device (deterministic for a given device and seed).
"""
from __future__ import annotations

import math

import torch

SEED_Q, SEED_K, SEED_V, SEED_DO = 1000, 2000, 3000, 4000


def normal_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """i.i.d. N(0,1) in fp32 from ``seed``, rounded to bf16, on ``device``."""
    device = torch.device(device)
    numel = math.prod(shape)
    gen_dev = device if (device.type == "cuda" and numel > (1 << 22)) else torch.device("cpu")
    g = torch.Generator(device=gen_dev)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, device=gen_dev, dtype=torch.float32)
    return x.to(torch.bfloat16).to(device)


def prefill_inputs(cfg: int, B: int, Hq: int, Hkv: int, N: int, d: int, device="cpu"):
    """q ``[B, Hq, N, d]``, k and v ``[B, Hkv, N, d]``, bf16, contiguous."""
    q = normal_bf16((B, Hq, N, d), SEED_Q + cfg, device)
    k = normal_bf16((B, Hkv, N, d), SEED_K + cfg, device)
    v = normal_bf16((B, Hkv, N, d), SEED_V + cfg, device)
    return q, k, v


def output_grad(cfg: int, B: int, Hq: int, N: int, d: int, device="cpu"):
    """dO ``[B, Hq, N, d]`` bf16 (the backward pass's incoming gradient)."""
    return normal_bf16((B, Hq, N, d), SEED_DO + cfg, device)


def decode_inputs(cfg: int, B: int, Hq: int, Hkv: int, s_max: int, d: int, device="cpu"):
    """q ``[B, Hq, d]``, kcache and vcache ``[B, Hkv, s_max, d]``, bf16."""
    q = normal_bf16((B, Hq, d), SEED_Q + cfg, device)
    kc = normal_bf16((B, Hkv, s_max, d), SEED_K + cfg, device)
    vc = normal_bf16((B, Hkv, s_max, d), SEED_V + cfg, device)
    return q, kc, vc


def ragged_seqlens(B: int, s_max: int, seed: int):
    """Per-sequence lengths in ``[0, s_max]`` with both ends represented."""
    g = torch.Generator().manual_seed(int(seed))
    lens = torch.randint(0, s_max + 1, (B,), generator=g).tolist()
    if B >= 1:
        lens[0] = s_max
    if B >= 2:
        lens[1] = 0 if B > 2 else max(1, s_max // 3)
    return lens


def sample_rows(N: int, n_random: int = 32, seed: int = 7):
    """Row indices for sampled checks: tile edges, the middle, the last row and
    ``n_random`` seeded random rows (deduplicated, sorted)."""
    fixed = [0, 1, 127, 128, 255, 256, N // 2, N - 1]
    g = torch.Generator().manual_seed(int(seed))
    rnd = torch.randint(0, N, (n_random,), generator=g).tolist() if N > 0 else []
    return sorted({r for r in fixed + rnd if 0 <= r < N})


def sample_heads(Hq: int, Hkv: int):
    """Query heads for sampled checks: first, middle and last, plus the first and
    last query head of the first and last KV group."""
    G = Hq // Hkv
    cand = [0, Hq // 2, Hq - 1, G - 1, Hq - G]
    return sorted({h for h in cand if 0 <= h < Hq})
