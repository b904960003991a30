"""The forward of grouped-query attention and of packed sequences at the size
bench.py times them (B=1, H=8, L=131072, d=128, N=16, causal; bench.py
--kv-heads 2 and --varlen 64), through the same calls, against the fp64
oracle on a sample of query rows it computes one by one: every shard's first
and last rows, random rows, and, with packed sequences, the first and last
row of every sequence.

"From Ring Attention to DeepSpeed Ulysses to USP" (jsqmd.com/news/734632):
§5.3 (grouped key/value heads), §6.2 and §8 (variable-length sequences).
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import assert_attention_close
from synthetic_inputs import WORKLOADS, make_cu_seqlens, make_qkv
from test_gpu_workloads import sample_rows

pytestmark = pytest.mark.gpu

WORKLOAD = "striped_B1_H8_L131072_d128_N16"


def ring_fwd_rows(ra, q, k, v, N, layout, causal, rows, cu=None):
    """Shard permutes, fused ring sweep (GQA or packed-sequence entry point),
    inverse permutes; O and LSE of the given sequence rows."""
    dev = torch.device("cuda:0")
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    S = L // N
    sh = []
    for x in (q, k, v):
        xg = x.to(dev)
        y = torch.empty((N, B, S, x.shape[2], d), dtype=torch.bfloat16, device=dev)
        ra.ra_shard_permute(xg, y, ra.RA_SEQ_TO_SHARDS, layout, B, L, x.shape[2], d, N)
        sh.append(y)
        del xg
    o = torch.empty((N, B, S, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((N, B, H, S), dtype=torch.float32, device=dev)
    ws = ra.new_workspace(ra.ra_ring_attn_workspace_bytes(B, L, H, d, N))
    if cu is None:
        ra.ra_ring_attn_fwd_gqa(*sh, o, lse, B, L, H, Hkv, d, N, layout, causal, workspace=ws)
    else:
        cu_dev = torch.as_tensor(np.asarray(cu), dtype=torch.int32).to(dev)
        ra.ra_ring_attn_fwd_varlen(*sh, o, lse, cu_dev, L, H, Hkv, d, N, layout, causal, workspace=ws)
    del sh
    o_seq = torch.empty((B, L, H, d), dtype=torch.float32, device=dev)
    ra.ra_shard_permute(o, o_seq, ra.RA_SHARDS_TO_SEQ, layout, B, L, H, d, N)
    lse_seq = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    ra.ra_lse_to_seq(lse, lse_seq, layout, B, L, H, N)
    ra.ra_check_status(ws)
    idx = torch.as_tensor(rows, device=dev)
    return o_seq[:, idx].cpu().numpy(), lse_seq[:, :, idx].cpu().numpy()


def test_gqa_full_size(ralib, gpu):
    w = WORKLOADS[WORKLOAD]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    Hkv = 2
    q, k, v, _ = make_qkv(B, L, H, d, w["seed"], w["k_scale_frac"])
    k, v = k[:, :, :Hkv].contiguous(), v[:, :, :Hkv].contiguous()
    rows = sample_rows(w, "striped", [], seed=3)
    o, lse = ring_fwd_rows(ralib, q, k, v, N, "striped", True, rows)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=True, rows=rows)
    assert_attention_close(o, o_ref, lse, lse_ref, "GQA H_kv=2 at 128K")


@pytest.mark.parametrize("layout", ["striped", "zigzag", "contiguous"])
def test_packed_sequences_full_size(ralib, gpu, layout):
    w = WORKLOADS[WORKLOAD]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    q, k, v, _ = make_qkv(B, L, H, d, w["seed"], w["k_scale_frac"])
    cu = make_cu_seqlens(L, 64, w["seed"]).numpy()
    bounds = np.concatenate([cu[:-1], cu[1:] - 1])
    rows = np.unique(np.concatenate([sample_rows(w, layout, [], seed=4), bounds[(bounds >= 0) & (bounds < L)]]))
    o, lse = ring_fwd_rows(ralib, q, k, v, N, layout, True, rows, cu=cu)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=True, rows=rows, cu_seqlens=cu)
    assert_attention_close(o, o_ref, lse, lse_ref, "64 packed sequences at 128K, %s" % layout)
