"""Gradients at the size the backward bench times (B=1, H=8, L=131072, d=128,
N=16, striped, causal; MHA and H_kv = 2), through the same calls, against the
fp64 oracle where it can compute them one by one, and two identities over
every key.

- dQ of a sample of query rows in every head (the first and last 32 positions,
  which hold every shard's first and last rows in the striped layout, and 32
  random rows): a row's dQ depends on its own row only.
- dK and dV of the last 256 keys of the first and last key/value head: with the
  causal mask only the last 256 query rows see them.
- Identities of the derivative of "From Ring Attention to DeepSpeed Ulysses to
  USP" (jsqmd.com/news/734632) §2's attention, over all keys: each row of dS
  sums to 0, so sum_k dK = 0, and each row of P sums to 1, so
  sum_k dV = sum_q dO over the query heads of the group.  The kernels round P
  and dS to bf16 (2^-9 relative per element), which leaves sum_k dK at about
  0.6 % of the key-wise norm of dK (measured with the same rounding in fp64 at
  2K-8K keys) and sum_k dV within 1e-4 of sum_q dO; the bounds are 3e-2 and
  1e-3.  A D (rowsum dO * O) off by a few percent breaks the first.
"""
import numpy as np
import pytest
import torch

from oracle.backward import attention_backward_rows
from synthetic_inputs import WORKLOADS, make_dout, make_qkv
from test_gpu_backward import assert_grad_close

pytestmark = pytest.mark.gpu

WORKLOAD = "striped_B1_H8_L131072_d128_N16"
TAIL = 256


def gpu_gradients(ra, q, k, v, do, N, layout, causal):
    """Shard, forward, backward, un-shard; returns dq, dk, dv [B, L, ., d] fp32 on the device."""
    dev = torch.device("cuda:0")
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    S = L // N

    def shard(x):
        xg = x.to(dev)
        y = torch.empty((N, B, S, x.shape[2], d), dtype=torch.bfloat16, device=dev)
        ra.ra_shard_permute(xg, y, ra.RA_SEQ_TO_SHARDS, layout, B, L, x.shape[2], d, N)
        return y

    qs, ks, vs, dos = shard(q), shard(k), shard(v), shard(do)
    o = torch.empty((N, B, S, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((N, B, H, S), dtype=torch.float32, device=dev)
    ws = ra.new_workspace(max(ra.ra_ring_attn_workspace_bytes(B, L, H, d, N),
                              ra.ra_ring_attn_bwd_workspace_bytes(B, L, H, d, N)))
    ra.ra_ring_attn_fwd_gqa(qs, ks, vs, o, lse, B, L, H, Hkv, d, N, layout, causal, workspace=ws)
    dq = torch.empty_like(o)
    dk = torch.empty((N, B, S, Hkv, d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    ra.ra_ring_attn_bwd(qs, ks, vs, o, dos, lse, dq, dk, dv, B, L, H, Hkv, d, N, layout, causal, workspace=ws)
    ra.ra_check_status(ws)
    del qs, ks, vs, dos, o, lse

    def unshard(x):
        y = torch.empty((B, L, x.shape[3], d), dtype=torch.float32, device=dev)
        ra.ra_shard_permute(x, y, ra.RA_SHARDS_TO_SEQ, layout, B, L, x.shape[3], d, N)
        return y

    return unshard(dq), unshard(dk), unshard(dv)


@pytest.mark.parametrize("Hkv", [8, 2], ids=["mha", "gqa4"])
def test_backward_full_size(ralib, gpu, Hkv):
    w = WORKLOADS[WORKLOAD]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    layout, causal = "striped", w["causal"]
    q, k, v, _ = make_qkv(B, L, H, d, w["seed"], w["k_scale_frac"])
    if Hkv != H:
        k, v = k[:, :, :Hkv].contiguous(), v[:, :, :Hkv].contiguous()
    do = make_dout(B, L, H, d)
    dq, dk, dv = gpu_gradients(ralib, q, k, v, do, N, layout, causal)
    assert bool(torch.isfinite(dq).all()) and bool(torch.isfinite(dk).all()) and bool(torch.isfinite(dv).all())
    group = H // Hkv

    # identities over every key (fp64 sums on the device)
    dev = dq.device
    do_sum = do.to(dev).double().sum(dim=1).view(B, Hkv, group, d).sum(dim=2)
    dv_sum = dv.double().sum(dim=1)
    err_v = (dv_sum - do_sum).abs().max().item()
    assert err_v <= 1e-3 * max(1.0, do_sum.abs().max().item()), "sum_k dV - sum_q dO: %g" % err_v
    dk_sum = dk.double().sum(dim=1)
    dk_norm = dk.double().pow(2).sum(dim=1).sqrt()
    ratio = (dk_sum.abs() / dk_norm.clamp_min(1e-30)).max().item()
    assert ratio <= 3e-2, "sum_k dK / |dK| = %g" % ratio

    # sampled query rows of every head: dQ
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.arange(32), np.arange(L - 32, L),
                                     rng.choice(np.arange(32, L - 32), size=32, replace=False)]))
    dq_rows = dq[:, torch.as_tensor(rows, device=dev)].cpu().numpy()
    for b in range(B):
        for h in range(H):
            ref, _, _ = attention_backward_rows(q, k, v, do, causal, b, h, rows)
            assert_grad_close(dq_rows[b, :, h], ref, "dQ rows, head %d" % h)

    # the last TAIL keys of the first and last key/value heads: dK and dV
    k0 = L - TAIL
    tail = np.arange(k0, L)
    dk_tail = dk[:, k0:].cpu().numpy()
    dv_tail = dv[:, k0:].cpu().numpy()
    for b in range(B):
        for kv in sorted({0, Hkv - 1}):
            parts = [attention_backward_rows(q, k, v, do, causal, b, h, tail)
                     for h in range(kv * group, (kv + 1) * group)]
            assert_grad_close(dk_tail[b, :, kv], sum(p[1] for p in parts)[k0:], "dK last keys, kv head %d" % kv)
            assert_grad_close(dv_tail[b, :, kv], sum(p[2] for p in parts)[k0:], "dV last keys, kv head %d" % kv)


def test_backward_zigzag_32k_whole_head(ralib, gpu):
    """Every gradient element of one (batch, head) of the 2 x 32K zigzag workload (H = 32,
    N = 8, 1 % of the key rows scaled x4), through the token-order backward, against the
    fp64 derivative computed over all rows of that head: dQ of every row, and dK and dV of
    every key as the sum of all rows' contributions."""
    w = WORKLOADS["zigzag_B2_H32_L32768_d128_N8_kscaled"]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    q, k, v, _ = make_qkv(B, L, H, d, w["seed"], w["k_scale_frac"])
    do = make_dout(B, L, H, d, seed=11)
    dev = torch.device("cuda:0")
    qg, kg, vg, dog = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    flags = ralib.RA_FLAG_SEQ_ORDER
    o = torch.empty((B, L, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    ws = ralib.new_workspace(max(ralib.ra_ring_attn_workspace_bytes(B, L, H, d, N, flags),
                                 ralib.ra_ring_attn_bwd_workspace_bytes(B, L, H, d, N)))
    ralib.ra_ring_attn_fwd(qg, kg, vg, o, lse, B, L, H, d, N, "zigzag", True, flags=flags, workspace=ws)
    dq = torch.empty_like(o)
    dk = torch.empty_like(o)
    dv = torch.empty_like(o)
    ralib.ra_ring_attn_bwd(qg, kg, vg, o, dog, lse, dq, dk, dv, B, L, H, H, d, N, "zigzag", True, workspace=ws,
                           flags=flags)
    ralib.ra_check_status(ws)
    b, h = 1, 7
    ref_dq, ref_dk, ref_dv = attention_backward_rows(q, k, v, do, True, b, h, np.arange(L), chunk=256)
    assert_grad_close(dq[b, :, h].cpu().numpy(), ref_dq, "dQ, zigzag 32K, every row")
    assert_grad_close(dk[b, :, h].cpu().numpy(), ref_dk, "dK, zigzag 32K, every key")
    assert_grad_close(dv[b, :, h].cpu().numpy(), ref_dv, "dV, zigzag 32K, every key")
