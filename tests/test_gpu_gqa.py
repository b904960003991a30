"""Grouped-query attention on the GPU against the fp64 oracle.

"From Ring Attention to DeepSpeed Ulysses to USP" (jsqmd.com/news/734632), §5.3:
with GQA, K and V carry H_kv < H heads and the Ulysses degree must divide
H_kv, while the ring is not constrained by the head count.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.layouts as ly
from conftest import assert_attention_close
from synthetic_inputs import randn_bf16

pytestmark = pytest.mark.gpu


def _qkv(B, L, H, Hkv, d, seed):
    return (randn_bf16((B, L, H, d), seed), randn_bf16((B, L, Hkv, d), seed + 1),
            randn_bf16((B, L, Hkv, d), seed + 2))


def run_ring_gqa(ra, q, k, v, N, layout, causal, U=1, flags=0):
    dev = torch.device("cuda:0")
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    R, P = N, U * N
    sh = []
    for x, Hx in ((q, H), (k, Hkv), (v, Hkv)):
        y = torch.empty((P, B, L // P, Hx, d), dtype=torch.bfloat16, device=dev)
        ra.ra_shard_permute(x.to(dev), y, ra.RA_SEQ_TO_SHARDS, layout, B, L, Hx, d, R, U)
        if U > 1:
            z = torch.empty((R, U, B, L // R, Hx // U, d), dtype=torch.bfloat16, device=dev)
            ra.ra_shard_permute(y, z, ra.RA_ULYSSES_SEQ_TO_HEAD, layout, B, L, Hx, d, R, U)
            y = z
        sh.append(y)
    Bq, Hq, Hkq = U * B, H // U, Hkv // U
    o = torch.empty(sh[0].shape, dtype=torch.float32, device=dev)
    lse = torch.empty((R, Bq, Hq, L // R), dtype=torch.float32, device=dev)
    ws = ra.new_workspace(ra.ra_ring_attn_workspace_bytes(Bq, L, Hq, d, R, flags))
    ra.ra_ring_attn_fwd_gqa(*sh, o, lse, Bq, L, Hq, Hkq, d, R, layout, causal, flags=flags, workspace=ws)
    if U > 1:
        o2 = torch.empty((P, B, L // P, H, d), dtype=torch.float32, device=dev)
        ra.ra_shard_permute(o, o2, ra.RA_ULYSSES_HEAD_TO_SEQ, layout, B, L, H, d, R, U)
        o = o2
    o_seq = torch.empty((B, L, H, d), dtype=torch.float32, device=dev)
    ra.ra_shard_permute(o, o_seq, ra.RA_SHARDS_TO_SEQ, layout, B, L, H, d, R, U)
    lse_seq = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    ra.ra_lse_to_seq(lse, lse_seq, layout, B, L, H, R, U)
    ra.ra_check_status(ws)
    return o_seq.cpu().numpy(), lse_seq.cpu().numpy()


@pytest.mark.parametrize("B,L,H,Hkv,d,N,layout,causal,U", [
    (1, 1024, 8, 2, 128, 4, "striped", True, 1),
    (1, 1024, 4, 1, 128, 4, "zigzag", True, 1),       # multi-query attention
    (2, 1200, 6, 3, 64, 3, "contiguous", True, 1),   # ragged tiles
    (1, 768, 4, 4, 128, 2, "striped", False, 1),     # H_kv = H
    (1, 2048, 8, 2, 128, 4, "zigzag", True, 2),      # USP: U = 2 divides H_kv = 2
])
@pytest.mark.parametrize("flags", [0, 1], ids=["fused", "stepwise"])
def test_ring_gqa_matches_oracle(ralib, gpu, B, L, H, Hkv, d, N, layout, causal, U, flags):
    q, k, v = _qkv(B, L, H, Hkv, d, seed=L + H + Hkv)
    o, lse = run_ring_gqa(ralib, q, k, v, N, layout, causal, U=U, flags=flags)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=causal)
    assert_attention_close(o, o_ref, lse, lse_ref, "gqa %s H=%d Hkv=%d U=%d" % (layout, H, Hkv, U))


def test_block_gqa_matches_oracle(ralib, gpu):
    B, S, H, Hkv, d, N, layout = 1, 256, 8, 2, 128, 4, "striped"
    q, k, v = _qkv(B, S * N, H, Hkv, d, seed=5)
    u16 = lambda t: t.view(torch.int16).numpy()
    qs = torch.from_numpy(ly.seq_to_shards(u16(q), layout, N)).view(torch.bfloat16)
    ks = torch.from_numpy(ly.seq_to_shards(u16(k), layout, N)).view(torch.bfloat16)
    vs = torch.from_numpy(ly.seq_to_shards(u16(v), layout, N)).view(torch.bfloat16)
    ws = ralib.new_workspace(256)
    for i, j in [(1, 1), (1, 3), (3, 0)]:
        o = torch.empty((B, S, H, d), dtype=torch.float32, device=gpu)
        lse = torch.empty((B, H, S), dtype=torch.float32, device=gpu)
        ralib.ra_block_attn_fwd_gqa(qs[i].cuda(), ks[j].cuda(), vs[j].cuda(), o, lse, B, S, H, Hkv, d, N,
                                    i, j, layout, True, workspace=ws)
        ralib.ra_check_status(ws)
        o_ref, lse_ref = oracle.block_attention(qs[i], ks[j], vs[j], layout, N, i, j, True)
        assert_attention_close(o.cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref, "gqa block (%d,%d)" % (i, j))


def test_gqa_rejects_bad_head_counts(ralib, gpu):
    lib = ralib.lib()
    F = 0x10000
    st = lib.ra_ring_attn_fwd_gqa(F, F, F, F, F, 1, 1024, 8, 3, 128, 4, 0, 1, 0.0, 0, F, 256, None)
    assert st == ralib.RA_ERR_SHAPE
