"""The multi-GPU ring driver on one GPU: N virtual ranks in one process, the KV shift
done by device-to-device copies on a copy stream (LoopbackRing), every step's block
call and merge through the C ABI ("From Ring Attention to DeepSpeed Ulysses to USP",
jsqmd.com/news/734632, §3.3 and §6.2).

The driver launches the same kernels in the same order per rank as the stepwise sweep
(RA_FLAG_STEPWISE), except that steps with no visible pair launch nothing -- and merging
an empty partial leaves the accumulator bit for bit unchanged -- so the results must be
identical to it, and within the parity bar of the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import assert_attention_close
from synthetic_inputs import randn_bf16

pytestmark = pytest.mark.gpu


def stacks(ra, xs, layout, N):
    out = []
    for x in xs:
        B, L, Hx, d = x.shape
        y = torch.empty((N, B, L // N, Hx, d), dtype=torch.bfloat16, device="cuda")
        ra.ra_shard_permute(x.cuda(), y, ra.RA_SEQ_TO_SHARDS, layout, B, L, Hx, d, N)
        out.append(y)
    return out


CASES = [
    # B, L, H, Hkv, d, N, layout, causal
    (1, 2048, 4, 4, 128, 4, "striped", True),
    (1, 2048, 4, 2, 128, 4, "contiguous", True),    # later ranks' shards: no launch
    (2, 1200, 2, 2, 64, 3, "zigzag", True),         # S = 400: ragged tiles
    (1, 1280, 4, 1, 128, 5, "striped", False),
    (1, 8192, 8, 8, 128, 16, "zigzag", True),
]


@pytest.mark.parametrize("B,L,H,Hkv,d,N,layout,causal", CASES)
def test_loopback_ring_matches_stepwise_and_oracle(ralib, gpu, B, L, H, Hkv, d, N, layout, causal):
    from sequence_blockwise_softmax_gb300 import ring
    seed = 4000 + L + N
    q = randn_bf16((B, L, H, d), seed)
    k = randn_bf16((B, L, Hkv, d), seed + 1)
    v = randn_bf16((B, L, Hkv, d), seed + 2)
    qs, ks, vs = stacks(ralib, (q, k, v), layout, N)
    o, lse, launched = ring.ring_attention_fwd_loopback(qs, ks, vs, N, layout, causal)
    S = L // N
    # the stepwise sweep: N block launches and N - 1 merges per rank, all ranks at once
    o_sw = torch.empty((N, B, S, H, d), dtype=torch.float32, device="cuda")
    lse_sw = torch.empty((N, B, H, S), dtype=torch.float32, device="cuda")
    ws = ralib.new_workspace(ralib.ra_ring_attn_workspace_bytes(B, L, H, d, N, ralib.RA_FLAG_STEPWISE))
    ralib.ra_ring_attn_fwd_gqa(qs, ks, vs, o_sw, lse_sw, B, L, H, Hkv, d, N, layout, causal,
                               flags=ralib.RA_FLAG_STEPWISE, workspace=ws)
    ralib.ra_check_status(ws)
    torch.cuda.synchronize()
    assert torch.equal(o, o_sw) and torch.equal(lse, lse_sw)
    active = sum(1 for i in range(N) for s, j, p in ring.ring_schedule(layout, S, N, i, causal) if s == 0 or p)
    assert launched == N + 2 * (active - N)
    o_seq = torch.empty((B, L, H, d), dtype=torch.float32, device="cuda")
    ralib.ra_shard_permute(o.contiguous(), o_seq, ralib.RA_SHARDS_TO_SEQ, layout, B, L, H, d, N)
    lse_seq = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    ralib.ra_lse_to_seq(lse.contiguous(), lse_seq, layout, B, L, H, N)
    kk = k.repeat_interleave(H // Hkv, dim=2)
    vv = v.repeat_interleave(H // Hkv, dim=2)
    o_ref, lse_ref = oracle.full_attention(q, kk, vv, causal=causal)
    assert_attention_close(o_seq.cpu().numpy(), o_ref, lse_seq.cpu().numpy(), lse_ref,
                           "loopback ring %s N=%d" % (layout, N))
