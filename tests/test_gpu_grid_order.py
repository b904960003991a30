"""The launch order of the query units and key tiles changes nothing but speed.

Causal work grows with position, so the forward and both backward passes run
heavy units first, taking (batch, head) pairs in chunks whose keys and values
fit in L2 together ("From Ring Attention to DeepSpeed Ulysses to USP",
jsqmd.com/news/734632, §3.4 and §4 discuss the causal imbalance this evens
out on one device).  ra_set_launch_chunk_budget sets the chunk budget.  Here it is set so
that the chunks split the pairs unevenly (a partial last chunk), and the results
must be bit-identical to those of the default order -- every unit's arithmetic
is independent of when it runs -- and match the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import assert_attention_close
from oracle.backward import attention_backward
from synthetic_inputs import randn_bf16
from test_gpu_backward import assert_grad_close, run_bwd
from test_gpu_gqa import run_ring_gqa

pytestmark = pytest.mark.gpu


# B, L, H, Hkv, d, N, layout, chunk budget in KB.  Streamed bytes per pair are
# 4 L d / group (forward and dQ pass) and 4 L d group (dK/dV pass): 512 KB per
# head at L = 1024, d = 128.
CASES = [
    (1, 1024, 5, 5, 128, 4, "striped", 1024),     # chunks of 2 + 2 + 1 pairs, every pass
    (1, 1024, 9, 3, 128, 4, "contiguous", 900),   # GQA: query chunks of 5 + 4
    (2, 768, 5, 5, 64, 3, "zigzag", 800),         # B*H = 10 in chunks of 4 + 4 + 2 (192 KB per head)
]


@pytest.mark.parametrize("B,L,H,Hkv,d,N,layout,kb", CASES)
def test_chunked_order_bit_identical(ralib, gpu, B, L, H, Hkv, d, N, layout, kb):
    ra = ralib
    seed = 7000 + L + H
    q, k, v = randn_bf16((B, L, H, d), seed), randn_bf16((B, L, Hkv, d), seed + 1), randn_bf16((B, L, Hkv, d), seed + 2)
    do = randn_bf16((B, L, H, d), seed + 3)
    ra.ra_set_launch_chunk_budget(0)
    o0, lse0 = run_ring_gqa(ra, q, k, v, N, layout, True)
    g0 = run_bwd(ra, q, k, v, do, N, layout, True)
    ra.ra_set_launch_chunk_budget(kb << 10)
    try:
        # the forward's and the dQ pass's chunks split the pairs unevenly
        group = H // Hkv
        c = ra.ra_launch_chunk_pairs(4 * L * d // group, B * H)
        assert 1 < c < B * H and (B * H) % c != 0, c
        o1, lse1 = run_ring_gqa(ra, q, k, v, N, layout, True)
        g1 = run_bwd(ra, q, k, v, do, N, layout, True)
    finally:
        ra.ra_set_launch_chunk_budget(0)
    assert np.array_equal(o0, o1) and np.array_equal(lse0, lse1), "forward depends on the unit order"
    for a, b, name in zip(g0, g1, ("dq", "dk", "dv")):
        assert np.array_equal(a, b), name + " depends on the tile order"
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=True)
    assert_attention_close(o1, o_ref, lse1, lse_ref, "chunked forward")
    for g, r, name in zip(g1, attention_backward(q, k, v, do, causal=True), ("dq", "dk", "dv")):
        assert_grad_close(g, r, name)
