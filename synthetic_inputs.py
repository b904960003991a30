"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so both the CPU oracle and the CUDA path can take their
inputs from here without sharing any of the method.

Recipe (the same on every machine):
  * one ``torch.Generator`` seeded with ``seed`` draws, in this order,
    Q, K and V as fp32 ``torch.randn`` tensors of shape ``[B, L, H, d]``
    (the pages' ``[bs, seq, heads, head_dim]`` order), each rounded to bf16
    with round-to-nearest-even;
  * when ``k_scale_frac > 0``, the same generator then draws, per batch element,
    ``ceil(k_scale_frac * L)`` token positions uniformly without replacement,
    and K at those positions (all heads) is multiplied by ``k_scale``.  With a
    power-of-two factor (4 in the zigzag workload) the product is exact in bf16.

Workload seeds: the five standard workloads use seeds 1001..1005.
"""
import math

import torch

# The five standard workloads, by what they are.  ``layouts`` lists the token
# assignments each one is run with; ``usp`` gives (Ulysses degree, ring degree).
WORKLOADS = {
    "tiny_noncausal_B1_H2_L512_d64_N4": dict(
        B=1, H=2, L=512, d=64, N=4, causal=False, layouts=("contiguous",),
        seed=1001, k_scale_frac=0.0),
    "causal_B1_H16_L8192_d128_N4": dict(
        B=1, H=16, L=8192, d=128, N=4, causal=True,
        layouts=("contiguous", "striped"), seed=1002, k_scale_frac=0.0),
    "zigzag_B2_H32_L32768_d128_N8_kscaled": dict(
        B=2, H=32, L=32768, d=128, N=8, causal=True, layouts=("zigzag",),
        seed=1003, k_scale_frac=0.01),
    "striped_B1_H8_L131072_d128_N16": dict(
        B=1, H=8, L=131072, d=128, N=16, causal=True,
        layouts=("striped", "contiguous"), seed=1004, k_scale_frac=0.0),
    "usp_U2xR4_zigzag_B1_H16_L262144_d128": dict(
        B=1, H=16, L=262144, d=128, N=4, U=2, causal=True, layouts=("zigzag",),
        seed=1005, k_scale_frac=0.0),
}


def make_qkv(B, L, H, d, seed, k_scale_frac=0.0, k_scale=4.0):
    """Return CPU bf16 tensors (q, k, v) of shape [B, L, H, d] and the scaled-K rows.

    The third value is a ``[B, n]`` int64 tensor of the token positions whose K
    rows were scaled (``n = 0`` when ``k_scale_frac == 0``).
    """
    g = torch.Generator().manual_seed(int(seed))
    q = torch.randn((B, L, H, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((B, L, H, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((B, L, H, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    n = int(math.ceil(k_scale_frac * L)) if k_scale_frac > 0 else 0
    rows = torch.zeros((B, n), dtype=torch.int64)
    for b in range(B):
        if n:
            rows[b] = torch.randperm(L, generator=g)[:n].sort().values
            k[b, rows[b]] = k[b, rows[b]] * k_scale
    return q, k, v, rows


def workload_inputs(name):
    w = WORKLOADS[name]
    return make_qkv(w["B"], w["L"], w["H"], w["d"], w["seed"], w["k_scale_frac"])


def make_extreme_qkv(B, L, H, d, seed, mode):
    """q, k, v (CPU bf16, [B, L, H, d]) whose scores q.k / sqrt(d) are tens of nats from 0:
      "large"    -- q and k of make_qkv times 4 (exact in bf16): scores ~ N(0, 16^2) nats;
      "negative" -- every key near one random direction u_h per head (k = u + 0.5 n) and
                    every query near -4 u_h (q = -4 (u + 0.1 n)): all scores about -45 nats,
                    spread by a few nats;
      "mixed"    -- like "negative", with a random sign per query token, so half the rows
                    score about +45 nats and half about -45."""
    if mode == "large":
        q, k, v, _ = make_qkv(B, L, H, d, seed)
        return (q.float() * 4).to(torch.bfloat16), (k.float() * 4).to(torch.bfloat16), v
    g = torch.Generator().manual_seed(int(seed))
    u = torch.randn((H, d), generator=g)
    k = u + 0.5 * torch.randn((B, L, H, d), generator=g)
    q = -4.0 * (u + 0.1 * torch.randn((B, L, H, d), generator=g))
    if mode == "mixed":
        sign = torch.randint(0, 2, (B, L, 1, 1), generator=g).float() * 2 - 1
        q = q * sign
    elif mode != "negative":
        raise ValueError(mode)
    v = torch.randn((B, L, H, d), generator=g)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def make_dout(B, L, H, d, seed=7):
    """The output gradient dO [B, L, H, d] bf16 of the backward workloads, N(0, 1)."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn((B, L, H, d), generator=g).to(torch.bfloat16)


def randn_bf16(shape, seed):
    """One bf16 tensor from N(0, 1) with its own seeded generator."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def randn_f32(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn(shape, generator=g, dtype=torch.float32) * scale


def random_ints(n, low, high, seed):
    g = torch.Generator().manual_seed(int(seed))
    return torch.randint(low, high, (n,), generator=g, dtype=torch.int64)


def random_perm(n, seed):
    g = torch.Generator().manual_seed(int(seed))
    return torch.randperm(n, generator=g)


def make_cu_seqlens(L, n_seqs, seed):
    """Boundaries of n_seqs packed sequences over L tokens: n_seqs - 1 distinct cut points
    drawn uniformly from 1..L-1 with a seeded generator (a broad length mix, from a few
    tokens to several times the mean).  Returns an int64 tensor [0, c_1, ..., L]."""
    g = torch.Generator().manual_seed(int(seed))
    cuts = torch.randperm(L - 1, generator=g)[:n_seqs - 1] + 1
    return torch.cat([torch.zeros(1, dtype=torch.int64), cuts.sort().values,
                      torch.full((1,), L, dtype=torch.int64)])
