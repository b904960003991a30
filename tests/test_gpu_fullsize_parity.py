"""Whole-head parity at the full workload sizes, and the per-step calls at the
bench's size.

The stratified row samples of ``test_gpu_workloads`` cover a small fraction of
O; here every row of chosen (batch, head) slices is compared with the fp64
oracle element by element, through the launches bench.py times (the fused
token-order sweep, ``RA_FLAG_SEQ_ORDER``):

  * 128K causal (B=1, H=8, L=131072, d=128, N=16): one whole head, striped and
    contiguous (1/8 of O each);
  * 2 x 32K zigzag with scaled keys (B=2, H=32, N=8): four whole (batch, head)
    slices (4/64 of O);
  * the USP workload (L=262144, U=2 x R=4 zigzag): one head over windows of
    4096 rows on both sides of every zigzag-chunk / Ulysses-piece boundary (the
    two coincide in token order), and the last 4096 rows (61440 of the head's
    262144 rows);
  * 32K with grouped key/value heads and packed sequences: two whole heads,
    striped (the tile-skipping variant) and zigzag;

and the pages' per-step structure at the 128K size ("From Ring Attention to
DeepSpeed Ulysses to USP", jsqmd.com/news/734632, §3.1-§3.3: N rounds of block
attention merged online equal single-device attention, in any block order):

  * ``RA_FLAG_STEPWISE`` (N block launches + N-1 merges) on the oracle's
    stratified row sample and against the fused sweep over the whole output;
  * ``ra_block_attn_fwd`` for diagonal, earlier and later key shards (each a
    whole 8192 x 8192 block, all heads), element by element.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import assert_attention_close
from synthetic_inputs import WORKLOADS, make_qkv
from test_gpu_workloads import gpu_path, sample_rows

pytestmark = pytest.mark.gpu

W4 = "striped_B1_H8_L131072_d128_N16"


def seq_order_sweep(ra, q, k, v, N, layout, causal):
    dev = torch.device("cuda:0")
    B, L, H, d = q.shape
    qg, kg, vg = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty((B, L, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    flags = ra.RA_FLAG_SEQ_ORDER
    ws = ra.new_workspace(ra.ra_ring_attn_workspace_bytes(B, L, H, d, N, flags))
    ra.ra_ring_attn_fwd(qg, kg, vg, o, lse, B, L, H, d, N, layout, causal, flags=flags, workspace=ws)
    ra.ra_check_status(ws)
    return o, lse


def head_slice(x, h):
    return x[:, :, h:h + 1].contiguous()


def test_128k_whole_head_striped_and_contiguous(ralib, gpu):
    w = WORKLOADS[W4]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    q, k, v, _ = make_qkv(B, L, H, d, w["seed"])
    h = 5
    o_ref, lse_ref = oracle.full_attention(head_slice(q, h), head_slice(k, h), head_slice(v, h), causal=True)
    for layout in ("striped", "contiguous"):
        o, lse = seq_order_sweep(ralib, q, k, v, N, layout, True)
        assert_attention_close(o[:, :, h:h + 1].cpu().numpy(), o_ref, lse[:, h:h + 1].cpu().numpy(), lse_ref,
                               "128K %s, head %d, every row" % (layout, h))
        del o, lse


def test_zigzag_32k_four_whole_heads(ralib, gpu):
    name = "zigzag_B2_H32_L32768_d128_N8_kscaled"
    w = WORKLOADS[name]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    q, k, v, _ = make_qkv(B, L, H, d, w["seed"], w["k_scale_frac"])
    o, lse = seq_order_sweep(ralib, q, k, v, N, "zigzag", True)
    for b, h in ((0, 0), (0, 17), (1, 6), (1, 31)):
        sl = lambda x: x[b:b + 1, :, h:h + 1].contiguous()
        o_ref, lse_ref = oracle.full_attention(sl(q), sl(k), sl(v), causal=True)
        assert_attention_close(o[b:b + 1, :, h:h + 1].cpu().numpy(), o_ref, lse[b:b + 1, h:h + 1].cpu().numpy(),
                               lse_ref, "zigzag 32K, batch %d head %d, every row" % (b, h))


def test_usp_boundary_windows_of_one_head(ralib, gpu):
    name = "usp_U2xR4_zigzag_B1_H16_L262144_d128"
    w = WORKLOADS[name]
    B, L, H, d, N, U = w["B"], w["L"], w["H"], w["d"], w["N"], w["U"]
    q, k, v, _ = make_qkv(B, L, H, d, w["seed"])
    C = L // (2 * N)               # zigzag chunk = Ulysses piece (L / (U * R)) here
    assert C == L // (U * N)
    win = 4096
    rows = set(range(L - win, L))
    for c in range(1, 2 * N):
        rows |= set(range(c * C - win, c * C + win))
    rows = np.array(sorted(rows), dtype=np.int64)
    h = 11
    o, lse = gpu_path(ralib, q, k, v, N, "zigzag", True, U=U, rows=rows)
    o_ref, lse_ref = oracle.full_attention(head_slice(q, h), head_slice(k, h), head_slice(v, h), causal=True,
                                           rows=rows)
    assert_attention_close(o[:, :, h:h + 1], o_ref, lse[:, h:h + 1], lse_ref,
                           "USP head %d, %d rows around every chunk boundary" % (h, rows.size))


def stack_inputs(ra, q, k, v, N, layout):
    dev = torch.device("cuda:0")
    B, L, H, d = q.shape
    out = []
    for x in (q, k, v):
        y = torch.empty((N, B, L // N, H, d), dtype=torch.bfloat16, device=dev)
        ra.ra_shard_permute(x.to(dev), y, ra.RA_SEQ_TO_SHARDS, layout, B, L, H, d, N)
        out.append(y)
    return out


@pytest.mark.parametrize("layout", ["striped", "contiguous"])
def test_128k_stepwise_sweep(ralib, gpu, layout):
    """N = 16 block launches of 8192 x 8192 (64 key tiles each) and 15 merges: the oracle's
    stratified row sample, and every element against the fused sweep at the same bar."""
    w = WORKLOADS[W4]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    q, k, v, scaled = make_qkv(B, L, H, d, w["seed"])
    S = L // N
    dev = torch.device("cuda:0")
    qs, ks, vs = stack_inputs(ralib, q, k, v, N, layout)
    o = torch.empty((N, B, S, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((N, B, H, S), dtype=torch.float32, device=dev)
    ws = ralib.new_workspace(ralib.ra_ring_attn_workspace_bytes(B, L, H, d, N, ralib.RA_FLAG_STEPWISE))
    ralib.ra_ring_attn_fwd(qs, ks, vs, o, lse, B, L, H, d, N, layout, True, flags=ralib.RA_FLAG_STEPWISE,
                           workspace=ws)
    o_f = torch.empty_like(o)
    lse_f = torch.empty_like(lse)
    ralib.ra_ring_attn_fwd(qs, ks, vs, o_f, lse_f, B, L, H, d, N, layout, True, workspace=ws)
    ralib.ra_check_status(ws)
    del ws, qs, ks, vs
    # whole output: stepwise against fused (both are within the bar of the exact result)
    assert_attention_close(o.cpu().numpy(), o_f.cpu().numpy(), lse.cpu().numpy(), lse_f.cpu().numpy(),
                           "128K %s stepwise vs fused" % layout)
    del o_f, lse_f
    o_seq = torch.empty((B, L, H, d), dtype=torch.float32, device=dev)
    ralib.ra_shard_permute(o, o_seq, ralib.RA_SHARDS_TO_SEQ, layout, B, L, H, d, N)
    lse_seq = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    ralib.ra_lse_to_seq(lse, lse_seq, layout, B, L, H, N)
    rows = sample_rows(w, layout, scaled, n_random=24, seed=17)
    idx = torch.as_tensor(rows, device=dev)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=True, rows=rows)
    assert_attention_close(o_seq[:, idx].cpu().numpy(), o_ref, lse_seq[:, :, idx].cpu().numpy(), lse_ref,
                           "128K %s stepwise, sampled rows" % layout)


@pytest.mark.parametrize("q_rank,kv_rank", [(15, 15), (9, 2), (2, 9), (0, 15)])
def test_128k_block_calls(ralib, gpu, q_rank, kv_rank):
    """ra_block_attn_fwd at the bench's shard size, striped: the own shard (diagonal), an
    earlier and a later rank's shard (the strict mask, row 0 empty), element by element."""
    w = WORKLOADS[W4]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    q, k, v, _ = make_qkv(B, L, H, d, w["seed"])
    S = L // N
    layout = "striped"
    dev = torch.device("cuda:0")
    qs, ks, vs = stack_inputs(ralib, q, k, v, N, layout)
    o = torch.empty((B, S, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    ws = ralib.new_workspace(256)
    ralib.ra_block_attn_fwd(qs[q_rank], ks[kv_rank], vs[kv_rank], o, lse, B, S, H, d, N, q_rank, kv_rank,
                            layout, True, workspace=ws)
    ralib.ra_check_status(ws)
    cpu = lambda t: t.cpu()
    o_ref, lse_ref = oracle.block_attention(cpu(qs[q_rank]), cpu(ks[kv_rank]), cpu(vs[kv_rank]), layout, N,
                                            q_rank, kv_rank, True)
    assert_attention_close(o.cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref,
                           "128K block q_rank %d kv_rank %d" % (q_rank, kv_rank))


@pytest.mark.parametrize("layout", ["striped", "zigzag"])
def test_32k_gqa_and_packed_whole_heads(ralib, gpu, layout):
    """Grouped key/value heads (H = 8, H_kv = 2) with 48 packed sequences over 32K tokens,
    N = 8, token order: in the striped layout this runs the tile-skipping kernel variant.
    Two whole query heads (of different key/value heads), every row, element by element."""
    B, L, H, Hkv, d, N = 1, 32768, 8, 2, 128, 8
    from synthetic_inputs import make_cu_seqlens, randn_bf16
    q = randn_bf16((B, L, H, d), 8101)
    k = randn_bf16((B, L, Hkv, d), 8102)
    v = randn_bf16((B, L, Hkv, d), 8103)
    cu = make_cu_seqlens(L, 48, seed=8104).numpy()
    dev = torch.device("cuda:0")
    cu_dev = torch.as_tensor(cu, dtype=torch.int32, device=dev)
    o = torch.empty((B, L, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    flags = ralib.RA_FLAG_SEQ_ORDER
    ws = ralib.new_workspace(ralib.ra_ring_attn_workspace_bytes(B, L, H, d, N, flags))
    ralib.ra_ring_attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), o, lse, cu_dev, L, H, Hkv, d, N, layout, True,
                                  flags=flags, workspace=ws)
    ralib.ra_check_status(ws)
    for h in (1, 6):
        kv = h // (H // Hkv)
        o_ref, lse_ref = oracle.full_attention(head_slice(q, h), head_slice(k, kv), head_slice(v, kv), causal=True,
                                               cu_seqlens=cu)
        assert_attention_close(o[:, :, h:h + 1].cpu().numpy(), o_ref, lse[:, h:h + 1].cpu().numpy(), lse_ref,
                               "32K GQA packed %s, head %d, every row" % (layout, h))
