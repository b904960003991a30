"""Attention on the GPU through the C ABI against the fp64 oracle, at sizes that span
several 128-row tiles and a ragged tail.

Ring sweep: "From Ring Attention to DeepSpeed Ulysses to USP" (jsqmd.com/news/734632),
§3.1-§3.3; causal mask by position, §3.4; layouts §4 / §6.1; USP §7.2.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import assert_attention_close
from synthetic_inputs import make_qkv

pytestmark = pytest.mark.gpu


def run_ring(ra, q, k, v, N, layout, causal, flags=0, U=1, scale=0.0, o_dtype=torch.float32):
    """Full path on the GPU: shard (and Ulysses) permutes, ring sweep, and back."""
    dev = torch.device("cuda:0")
    B, L, H, d = q.shape
    R = N
    P = U * R
    seq_sh = []
    for x in (q, k, v):
        y = torch.empty((P, B, L // P, H, d), dtype=torch.bfloat16, device=dev)
        ra.ra_shard_permute(x.to(dev), y, ra.RA_SEQ_TO_SHARDS, layout, B, L, H, d, R, U)
        if U > 1:
            z = torch.empty((R, U, B, L // R, H // U, d), dtype=torch.bfloat16, device=dev)
            ra.ra_shard_permute(y, z, ra.RA_ULYSSES_SEQ_TO_HEAD, layout, B, L, H, d, R, U)
            y = z
        seq_sh.append(y)
    Bq, Hq = U * B, H // U
    o = torch.empty(seq_sh[0].shape, dtype=o_dtype, device=dev)
    lse = torch.empty((R, Bq, Hq, L // R), dtype=torch.float32, device=dev)
    wflags = flags | (ra.RA_FLAG_O_BF16 if o_dtype == torch.bfloat16 else 0)
    ws = ra.new_workspace(ra.ra_ring_attn_workspace_bytes(Bq, L, Hq, d, R, wflags))
    ra.ra_ring_attn_fwd(*seq_sh, o, lse, Bq, L, Hq, d, R, layout, causal, scale=scale,
                        flags=flags, workspace=ws)
    if U > 1:
        o2 = torch.empty((P, B, L // P, H, d), dtype=o_dtype, device=dev)
        ra.ra_shard_permute(o, o2, ra.RA_ULYSSES_HEAD_TO_SEQ, layout, B, L, H, d, R, U)
        o = o2
    o_seq = torch.empty((B, L, H, d), dtype=o_dtype, device=dev)
    ra.ra_shard_permute(o, o_seq, ra.RA_SHARDS_TO_SEQ, layout, B, L, H, d, R, U)
    lse_seq = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    ra.ra_lse_to_seq(lse, lse_seq, layout, B, L, H, R, U)
    ra.ra_check_status(ws)
    return o_seq.float().cpu().numpy(), lse_seq.cpu().numpy()


RING_CASES = [
    # B, L, H, d, N, layout, causal
    (1, 512, 2, 64, 4, "contiguous", False),
    (1, 1024, 2, 128, 4, "contiguous", True),
    (1, 1024, 2, 128, 4, "striped", True),
    (1, 1024, 2, 128, 4, "zigzag", True),
    (2, 1200, 3, 128, 4, "striped", True),      # S = 300: ragged tiles
    (1, 1200, 2, 64, 3, "zigzag", True),        # chunks of 200 straddle tiles
    (1, 640, 2, 128, 5, "contiguous", True),
    (1, 384, 2, 128, 1, "contiguous", True),    # N = 1: plain causal attention
    (1, 768, 2, 64, 2, "striped", False),
    (1, 200, 2, 128, 2, "striped", True),       # S = 100 < one tile
]


@pytest.mark.parametrize("B,L,H,d,N,layout,causal", RING_CASES)
@pytest.mark.parametrize("flags", [0, 1], ids=["fused", "stepwise"])
def test_ring_matches_oracle(ralib, gpu, B, L, H, d, N, layout, causal, flags):
    q, k, v, _ = make_qkv(B, L, H, d, seed=L + H + d + N)
    o, lse = run_ring(ralib, q, k, v, N, layout, causal, flags=flags)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=causal)
    assert_attention_close(o, o_ref, lse, lse_ref, "%s N=%d causal=%s" % (layout, N, causal))


@pytest.mark.parametrize("flags", [0, 1], ids=["fused", "stepwise"])
def test_ring_bf16_output(ralib, gpu, flags):
    """With RA_FLAG_O_BF16 the output is the fp32 result rounded once to bf16, so it lies
    within the fp32 bar plus half a bf16 ulp of |O| (2^-8 relative) of the exact result."""
    q, k, v, _ = make_qkv(1, 1024, 2, 128, seed=31)
    o, lse = run_ring(ralib, q, k, v, 4, "zigzag", True, flags=flags, o_dtype=torch.bfloat16)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=True)
    half_ulp = np.abs(o_ref) * 2.0 ** -8
    assert np.all(np.abs(o - o_ref) <= 1e-2 + half_ulp)
    assert np.abs(lse - lse_ref).max() <= 1e-3
    # and it is exactly the fp32 path rounded to bf16
    o32, _ = run_ring(ralib, q, k, v, 4, "zigzag", True, flags=flags)
    np.testing.assert_array_equal(o, torch.from_numpy(o32).to(torch.bfloat16).float().numpy())


def test_ring_explicit_scale(ralib, gpu):
    q, k, v, _ = make_qkv(1, 512, 2, 128, seed=77)
    o, lse = run_ring(ralib, q, k, v, 4, "striped", True, scale=0.05)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=True, scale=0.05)
    assert_attention_close(o, o_ref, lse, lse_ref)


def test_ring_with_scaled_keys(ralib, gpu):
    """Large K rows (x4 on 1%) force running-max rescales mid-sweep."""
    q, k, v, _ = make_qkv(1, 2048, 2, 128, seed=5, k_scale_frac=0.01)
    o, lse = run_ring(ralib, q, k, v, 4, "zigzag", True)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=True)
    assert_attention_close(o, o_ref, lse, lse_ref)


@pytest.mark.parametrize("flags", [0, 1], ids=["fused", "stepwise"])
def test_usp_small(ralib, gpu, flags):
    """Ulysses x ring (U=2, R=4, zigzag, causal) composed from the permutes and the sweep."""
    q, k, v, _ = make_qkv(1, 2048, 4, 128, seed=55)
    o, lse = run_ring(ralib, q, k, v, 4, "zigzag", True, flags=flags, U=2)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=True)
    assert_attention_close(o, o_ref, lse, lse_ref)


BLOCK_CASES = [
    # B, S, H, d, N, layout, causal, (q_rank, kv_rank) pairs
    (1, 256, 2, 128, 4, "contiguous", True, [(2, 2), (2, 1), (1, 3), (0, 0)]),
    (1, 256, 2, 128, 4, "striped", True, [(1, 1), (1, 3), (3, 0), (0, 2)]),
    (2, 300, 2, 64, 4, "zigzag", True, [(0, 0), (0, 3), (3, 0), (2, 1)]),
    (1, 384, 3, 128, 2, "contiguous", False, [(0, 1), (1, 0)]),
]


@pytest.mark.parametrize("B,S,H,d,N,layout,causal,pairs", BLOCK_CASES)
def test_block_matches_oracle(ralib, gpu, B, S, H, d, N, layout, causal, pairs):
    L = S * N
    q, k, v, _ = make_qkv(B, L, H, d, seed=S + d)
    import oracle.layouts as ly
    qs = torch.from_numpy(ly.seq_to_shards(q.view(torch.int16).numpy(), layout, N)).view(torch.bfloat16)
    ks = torch.from_numpy(ly.seq_to_shards(k.view(torch.int16).numpy(), layout, N)).view(torch.bfloat16)
    vs = torch.from_numpy(ly.seq_to_shards(v.view(torch.int16).numpy(), layout, N)).view(torch.bfloat16)
    ws = ralib.new_workspace(256)
    for (i, j) in pairs:
        o = torch.empty((B, S, H, d), dtype=torch.float32, device=gpu)
        lse = torch.empty((B, H, S), dtype=torch.float32, device=gpu)
        ralib.ra_block_attn_fwd(qs[i].contiguous().to(gpu), ks[j].contiguous().to(gpu),
                                vs[j].contiguous().to(gpu), o, lse, B, S, H, d, N, i, j, layout,
                                causal, workspace=ws)
        ralib.ra_check_status(ws)
        o_ref, lse_ref = oracle.block_attention(qs[i], ks[j], vs[j], layout, N, i, j, causal)
        assert_attention_close(o.cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref,
                               "%s block (%d, %d)" % (layout, i, j))


def test_block_steps_merge_to_full(ralib, gpu):
    """N block calls folded with ra_lse_merge reproduce the one-shot oracle (§3.3 loop)."""
    B, L, H, d, N, layout = 1, 1024, 2, 128, 4, "striped"
    q, k, v, _ = make_qkv(B, L, H, d, seed=91)
    S = L // N
    dev = gpu
    sh = []
    for x in (q, k, v):
        y = torch.empty((N, B, S, H, d), dtype=torch.bfloat16, device=dev)
        ralib.ra_shard_permute(x.to(dev), y, ralib.RA_SEQ_TO_SHARDS, layout, B, L, H, d, N)
        sh.append(y)
    ws = ralib.new_workspace(256)
    o_seq = np.zeros((B, L, H, d))
    lse_seq = np.zeros((B, H, L))
    import oracle.layouts as ly
    pos = ly.rank_positions(layout, N, L)
    for i in range(N):
        acc_o = torch.empty((B, S, H, d), dtype=torch.float32, device=dev)
        acc_l = torch.empty((B, H, S), dtype=torch.float32, device=dev)
        part_o = torch.empty_like(acc_o)
        part_l = torch.empty_like(acc_l)
        for step in range(N):
            j = (i - step) % N
            dst_o, dst_l = (acc_o, acc_l) if step == 0 else (part_o, part_l)
            ralib.ra_block_attn_fwd(sh[0][i], sh[1][j], sh[2][j], dst_o, dst_l, B, S, H, d, N, i, j,
                                    layout, True, workspace=ws)
            if step:
                ralib.ra_lse_merge_bshd(acc_o, acc_l, part_o, part_l, B, S, H, d)
        o_seq[:, pos[i]] = acc_o.cpu().numpy()
        lse_seq[:, :, pos[i]] = acc_l.cpu().numpy()
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=True)
    assert_attention_close(o_seq, o_ref, lse_seq, lse_ref)


def test_status_word_stays_clear(ralib, gpu):
    ws = ralib.new_workspace(256)
    assert int(ws[:4].view(torch.int32).item()) == 0
    ralib.ra_check_status(ws)
