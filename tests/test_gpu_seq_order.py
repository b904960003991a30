"""The fused sweep reading and writing token order (RA_FLAG_SEQ_ORDER) against
the explicit path: shard permutes, the sweep on shard stacks, the inverse
permutes ("From Ring Attention to DeepSpeed Ulysses to USP",
jsqmd.com/news/734632, §3.1, §4, §6.1: the layout assigns token positions to
ranks).  The kernel's arithmetic is the same in both forms, only the tile
addresses differ, so O and LSE must agree bit for bit; small cases are also
compared with the fp64 oracle element by element, and the 128K workload on
sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import assert_attention_close
from synthetic_inputs import WORKLOADS, make_cu_seqlens, make_qkv, randn_bf16
from test_gpu_workloads import sample_rows

pytestmark = pytest.mark.gpu


def explicit_path(ra, q, k, v, N, layout, causal, o_dtype=torch.float32, cu=None):
    dev = q.device
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    S = L // N
    sh = []
    for x in (q, k, v):
        y = torch.empty((N, B, S, x.shape[2], d), dtype=torch.bfloat16, device=dev)
        ra.ra_shard_permute(x, y, ra.RA_SEQ_TO_SHARDS, layout, B, L, x.shape[2], d, N)
        sh.append(y)
    o = torch.empty((N, B, S, H, d), dtype=o_dtype, device=dev)
    lse = torch.empty((N, B, H, S), dtype=torch.float32, device=dev)
    ws = ra.new_workspace(ra.ra_ring_attn_workspace_bytes(B, L, H, d, N))
    if cu is None:
        ra.ra_ring_attn_fwd_gqa(*sh, o, lse, B, L, H, Hkv, d, N, layout, causal, workspace=ws)
    else:
        ra.ra_ring_attn_fwd_varlen(*sh, o, lse, cu, L, H, Hkv, d, N, layout, causal, workspace=ws)
    del sh
    o_seq = torch.empty((B, L, H, d), dtype=o_dtype, device=dev)
    ra.ra_shard_permute(o, o_seq, ra.RA_SHARDS_TO_SEQ, layout, B, L, H, d, N)
    lse_seq = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    ra.ra_lse_to_seq(lse, lse_seq, layout, B, L, H, N)
    ra.ra_check_status(ws)
    return o_seq, lse_seq


def seq_order_path(ra, q, k, v, N, layout, causal, o_dtype=torch.float32, cu=None):
    dev = q.device
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    o = torch.empty((B, L, H, d), dtype=o_dtype, device=dev)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    flags = ra.RA_FLAG_SEQ_ORDER
    ws = ra.new_workspace(ra.ra_ring_attn_workspace_bytes(B, L, H, d, N, flags))
    if cu is None:
        ra.ra_ring_attn_fwd_gqa(q, k, v, o, lse, B, L, H, Hkv, d, N, layout, causal, flags=flags, workspace=ws)
    else:
        ra.ra_ring_attn_fwd_varlen(q, k, v, o, lse, cu, L, H, Hkv, d, N, layout, causal, flags=flags,
                                   workspace=ws)
    ra.ra_check_status(ws)
    return o, lse


CASES = [
    # B, L, H, Hkv, d, N, layout, causal, packed sequences, bf16 O
    (2, 1024, 2, 2, 128, 4, "striped", True, None, False),
    (1, 1200, 4, 2, 64, 4, "contiguous", True, None, False),      # S = 300: ragged tiles
    (1, 1000, 2, 1, 128, 5, "striped", False, None, False),       # S = 200, MQA, non-causal
    (2, 2048, 2, 2, 128, 4, "zigzag", True, None, False),         # zigzag chunk 256
    (1, 3072, 2, 2, 64, 3, "zigzag", True, None, True),           # chunk 512, bf16 O
    (1, 2304, 2, 2, 128, 1, "contiguous", True, None, False),     # one rank
    (1, 4096, 2, 1, 128, 4, "striped", True, 40, False),          # packed: the tile-skipping variant
    (1, 2048, 2, 2, 128, 4, "zigzag", True, 9, False),            # packed
    (1, 1200, 2, 2, 128, 3, "contiguous", True, 7, True),         # packed, S = 400, bf16 O
]


@pytest.mark.parametrize("B,L,H,Hkv,d,N,layout,causal,packed,o_bf16", CASES)
def test_seq_order_matches_explicit_path_and_oracle(ralib, gpu, B, L, H, Hkv, d, N, layout, causal, packed,
                                                    o_bf16):
    dev = torch.device("cuda:0")
    q = randn_bf16((B, L, H, d), L + 31)
    k = randn_bf16((B, L, Hkv, d), L + 32)
    v = randn_bf16((B, L, Hkv, d), L + 33)
    cu = cu_dev = None
    if packed:
        cu = make_cu_seqlens(L, packed, seed=L + packed).numpy()
        cu_dev = torch.as_tensor(cu, dtype=torch.int32, device=dev)
    od = torch.bfloat16 if o_bf16 else torch.float32
    qg, kg, vg = q.to(dev), k.to(dev), v.to(dev)
    o_e, lse_e = explicit_path(ralib, qg, kg, vg, N, layout, causal, od, cu_dev)
    o_s, lse_s = seq_order_path(ralib, qg, kg, vg, N, layout, causal, od, cu_dev)
    assert torch.equal(o_s, o_e) and torch.equal(lse_s, lse_e)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=causal, cu_seqlens=cu)
    o = o_s.float().cpu().numpy()
    lse = lse_s.cpu().numpy()
    if o_bf16:
        # one bf16 rounding of the fp32 result: half an ulp of |O| on top of the bar
        assert np.abs(o - o_ref).max() <= 1e-2 + np.abs(o_ref).max() * 2.0 ** -8
        assert_attention_close(o_ref, o_ref, lse, lse_ref, "%s seq order, LSE" % layout)
    else:
        assert_attention_close(o, o_ref, lse, lse_ref, "%s seq order" % layout)


FULL = [(name, layout) for name, w in WORKLOADS.items() if w.get("U", 1) == 1 and w["L"] >= 8192
        for layout in w["layouts"]]


@pytest.mark.parametrize("name,layout", FULL)
def test_seq_order_full_size(ralib, gpu, name, layout):
    """The workloads bench.py times, both forms on the device, bit for bit; the
    128K one also against the oracle on a stratified row sample."""
    w = WORKLOADS[name]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    q, k, v, scaled = make_qkv(B, L, H, d, w["seed"], w["k_scale_frac"])
    dev = torch.device("cuda:0")
    qg, kg, vg = q.to(dev), k.to(dev), v.to(dev)
    o_e, lse_e = explicit_path(ralib, qg, kg, vg, N, layout, w["causal"])
    o_s, lse_s = seq_order_path(ralib, qg, kg, vg, N, layout, w["causal"])
    assert torch.equal(o_s, o_e) and torch.equal(lse_s, lse_e)
    if L == 131072:
        rows = sample_rows(w, layout, scaled, n_random=24, seed=9)
        idx = torch.as_tensor(rows, device=dev)
        o_ref, lse_ref = oracle.full_attention(q, k, v, causal=w["causal"], rows=rows)
        assert_attention_close(o_s[:, idx].cpu().numpy(), o_ref, lse_s[:, :, idx].cpu().numpy(), lse_ref,
                               "%s/%s seq order" % (name, layout))


def stack_backward(ra, q, k, v, do, N, layout, causal, cu=None):
    """Shard permutes, forward and backward on shard stacks, gradients back to token order."""
    dev = q.device
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    S = L // N

    def shard(x):
        y = torch.empty((N, B, S, x.shape[2], d), dtype=x.dtype, device=dev)
        ra.ra_shard_permute(x, y, ra.RA_SEQ_TO_SHARDS, layout, B, L, x.shape[2], d, N)
        return y

    qs, ks, vs, dos = shard(q), shard(k), shard(v), shard(do)
    o = torch.empty((N, B, S, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((N, B, H, S), dtype=torch.float32, device=dev)
    ws = ra.new_workspace(max(ra.ra_ring_attn_workspace_bytes(B, L, H, d, N),
                              ra.ra_ring_attn_bwd_workspace_bytes(B, L, H, d, N)))
    if cu is None:
        ra.ra_ring_attn_fwd_gqa(qs, ks, vs, o, lse, B, L, H, Hkv, d, N, layout, causal, workspace=ws)
    else:
        ra.ra_ring_attn_fwd_varlen(qs, ks, vs, o, lse, cu, L, H, Hkv, d, N, layout, causal, workspace=ws)
    dq = torch.empty_like(o)
    dk = torch.empty((N, B, S, Hkv, d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    ra.ra_ring_attn_bwd(qs, ks, vs, o, dos, lse, dq, dk, dv, B, L, H, Hkv, d, N, layout, causal,
                        cu_seqlens=cu, workspace=ws)
    ra.ra_check_status(ws)
    out = []
    for x in (dq, dk, dv):
        y = torch.empty((B, L, x.shape[3], d), dtype=torch.float32, device=dev)
        ra.ra_shard_permute(x, y, ra.RA_SHARDS_TO_SEQ, layout, B, L, x.shape[3], d, N)
        out.append(y)
    return out


def seq_order_backward(ra, q, k, v, do, N, layout, causal, cu=None):
    """Forward and backward in token order: no permute at all."""
    dev = q.device
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    flags = ra.RA_FLAG_SEQ_ORDER
    o = torch.empty((B, L, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    ws = ra.new_workspace(max(ra.ra_ring_attn_workspace_bytes(B, L, H, d, N, flags),
                              ra.ra_ring_attn_bwd_workspace_bytes(B, L, H, d, N)))
    if cu is None:
        ra.ra_ring_attn_fwd_gqa(q, k, v, o, lse, B, L, H, Hkv, d, N, layout, causal, flags=flags, workspace=ws)
    else:
        ra.ra_ring_attn_fwd_varlen(q, k, v, o, lse, cu, L, H, Hkv, d, N, layout, causal, flags=flags,
                                   workspace=ws)
    dq = torch.empty_like(o)
    dk = torch.empty((B, L, Hkv, d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    ra.ra_ring_attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, L, H, Hkv, d, N, layout, causal, cu_seqlens=cu,
                        workspace=ws, flags=flags)
    ra.ra_check_status(ws)
    return dq, dk, dv


BWD_CASES = [
    # B, L, H, Hkv, d, N, layout, causal, packed sequences
    (1, 1024, 2, 2, 128, 4, "striped", True, None),
    (2, 2048, 2, 1, 64, 4, "zigzag", True, None),          # zigzag chunk 256, MQA
    (1, 1200, 4, 2, 128, 4, "contiguous", True, None),     # S = 300: ragged tiles
    (1, 1000, 2, 2, 128, 5, "striped", False, None),       # S = 200, non-causal
    (1, 2048, 2, 2, 128, 4, "striped", True, 12),          # packed sequences
]


@pytest.mark.parametrize("B,L,H,Hkv,d,N,layout,causal,packed", BWD_CASES)
def test_backward_seq_order_matches_stack_path_and_oracle(ralib, gpu, B, L, H, Hkv, d, N, layout, causal, packed):
    from oracle.backward import attention_backward
    from test_gpu_backward import assert_grad_close
    dev = torch.device("cuda:0")
    q = randn_bf16((B, L, H, d), L + 41)
    k = randn_bf16((B, L, Hkv, d), L + 42)
    v = randn_bf16((B, L, Hkv, d), L + 43)
    do = randn_bf16((B, L, H, d), L + 44)
    cu = cu_dev = None
    if packed:
        cu = make_cu_seqlens(L, packed, seed=L + packed).numpy()
        cu_dev = torch.as_tensor(cu, dtype=torch.int32, device=dev)
    args = (q.to(dev), k.to(dev), v.to(dev), do.to(dev), N, layout, causal, cu_dev)
    tok = seq_order_backward(ralib, *args)
    stk = stack_backward(ralib, *args)
    for name, a, b in zip(("dq", "dk", "dv"), tok, stk):
        assert torch.equal(a, b), name
    ref = attention_backward(q, k, v, do, causal, cu_seqlens=cu)
    for name, g, r in zip(("dq", "dk", "dv"), tok, ref):
        assert_grad_close(g.cpu().numpy(), r, "%s token order %s" % (name, layout))


def test_backward_seq_order_full_size(ralib, gpu):
    """The backward bench workload (128K striped), both forms on the device, bit for bit."""
    from synthetic_inputs import make_dout
    w = WORKLOADS["striped_B1_H8_L131072_d128_N16"]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    q, k, v, _ = make_qkv(B, L, H, d, w["seed"], w["k_scale_frac"])
    dev = torch.device("cuda:0")
    args = (q.to(dev), k.to(dev), v.to(dev), make_dout(B, L, H, d).to(dev), N, "striped", True, None)
    tok = seq_order_backward(ralib, *args)
    stk = stack_backward(ralib, *args)
    for name, a, b in zip(("dq", "dk", "dv"), tok, stk):
        assert torch.equal(a, b), name
