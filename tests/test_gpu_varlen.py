"""Packed variable-length sequences in the ring sweep, against the fp64 oracle.

"From Ring Attention to DeepSpeed Ulysses to USP" (jsqmd.com/news/734632):
§6.2 (a varlen kernel per ring step), §8 (variable lengths as a ring weak
spot).  The layout shards the packed stream by position; a query sees only its
own sequence.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import assert_attention_close
from synthetic_inputs import make_cu_seqlens, randn_bf16

pytestmark = pytest.mark.gpu


def run_varlen(ra, q, k, v, cu, N, layout, causal, flags=0):
    dev = torch.device("cuda:0")
    _, L, H, d = q.shape
    Hkv = k.shape[2]
    sh = []
    for x, hx in ((q, H), (k, Hkv), (v, Hkv)):
        y = torch.empty((N, 1, L // N, hx, d), dtype=torch.bfloat16, device=dev)
        ra.ra_shard_permute(x.to(dev), y, ra.RA_SEQ_TO_SHARDS, layout, 1, L, hx, d, N)
        sh.append(y)
    o = torch.empty(sh[0].shape, dtype=torch.float32, device=dev)
    lse = torch.empty((N, 1, H, L // N), dtype=torch.float32, device=dev)
    ws = ra.new_workspace(ra.ra_ring_attn_workspace_bytes(1, L, H, d, N, flags))
    cu_dev = torch.as_tensor(cu, dtype=torch.int32).to(dev)
    ra.ra_ring_attn_fwd_varlen(*sh, o, lse, cu_dev, L, H, Hkv, d, N, layout, causal, flags=flags,
                               workspace=ws)
    o_seq = torch.empty((1, L, H, d), dtype=torch.float32, device=dev)
    ra.ra_shard_permute(o, o_seq, ra.RA_SHARDS_TO_SEQ, layout, 1, L, H, d, N)
    lse_seq = torch.empty((1, H, L), dtype=torch.float32, device=dev)
    ra.ra_lse_to_seq(lse, lse_seq, layout, 1, L, H, N)
    ra.ra_check_status(ws)
    return o_seq.cpu().numpy(), lse_seq.cpu().numpy()


CASES = [
    # L, H, Hkv, d, N, layout, causal, boundaries
    (1024, 2, 2, 128, 4, "contiguous", True, "random5"),
    (1024, 2, 2, 128, 4, "striped", True, [0, 1, 1, 300, 301, 700, 1024]),   # empty and 1-token
    (1200, 4, 2, 64, 3, "zigzag", True, "random7"),
    (768, 2, 2, 128, 2, "striped", False, "random4"),
    (2048, 2, 1, 128, 4, "zigzag", True, "random33"),
    (1024, 2, 2, 128, 4, "striped", True, [0, 1024]),                          # one sequence
    # many short sequences: each 128-row Q tile of a unit sees only some of
    # the tiles the unit visits, so d = 128 striped / zigzag skip tiles per Q tile
    (8192, 2, 1, 128, 4, "striped", True, "random64"),
    (6144, 2, 2, 128, 3, "zigzag", True, "random48"),
    (4096, 2, 2, 128, 4, "striped", False, "random20"),
    # more ring steps than the skip table holds: every tile is visited
    (9216, 1, 1, 128, 72, "striped", True, "random30"),
]


@pytest.mark.parametrize("L,H,Hkv,d,N,layout,causal,cu", CASES)
@pytest.mark.parametrize("flags", [0, 1], ids=["fused", "stepwise"])
def test_varlen_matches_oracle(ralib, gpu, L, H, Hkv, d, N, layout, causal, cu, flags):
    if isinstance(cu, str):
        cu = make_cu_seqlens(L, int(cu[6:]), seed=L + int(cu[6:])).numpy()
    cu = np.asarray(cu)
    q = randn_bf16((1, L, H, d), L + 1)
    k = randn_bf16((1, L, Hkv, d), L + 2)
    v = randn_bf16((1, L, Hkv, d), L + 3)
    o, lse = run_varlen(ralib, q, k, v, cu, N, layout, causal, flags=flags)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=causal, cu_seqlens=cu)
    assert_attention_close(o, o_ref, lse, lse_ref, "varlen %s %s" % (layout, list(cu)[:6]))
