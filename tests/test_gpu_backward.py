"""Gradients of the ring attention on the GPU against the fp64 oracle backward.

Tolerance (derived, the pages fix none for gradients): the kernels round P and
dS to bf16 before the tensor-core products (2^-9 relative per element) and
accumulate in fp32, like the forward's PV product, so the forward's relative
bar is kept: rel-L2 <= 5e-3, and max-abs <= 2e-2 * max(1, max |ref|) since
gradient magnitudes grow with the data (|dK|, |dQ| up to ~10 here).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.backward import attention_backward
from synthetic_inputs import make_cu_seqlens, randn_bf16

pytestmark = pytest.mark.gpu


def assert_grad_close(g, ref, what):
    g = np.asarray(g, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(g)), what
    err = np.abs(g - ref).max()
    rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    bound = 2e-2 * max(1.0, np.abs(ref).max())
    assert err <= bound, "%s: max-abs %g > %g" % (what, err, bound)
    assert rel <= 5e-3, "%s: rel-L2 %g" % (what, rel)


def run_bwd(ra, q, k, v, do, N, layout, causal, cu=None):
    dev = torch.device("cuda:0")
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    S = L // N

    def shard(x):
        y = torch.empty((N, B, S, x.shape[2], d), dtype=x.dtype, device=dev)
        ra.ra_shard_permute(x.to(dev).contiguous(), y, ra.RA_SEQ_TO_SHARDS, layout, B, L, x.shape[2], d, N)
        return y

    qs, ks, vs, dos = shard(q), shard(k), shard(v), shard(do)
    cu_dev = None if cu is None else torch.as_tensor(cu, dtype=torch.int32).to(dev)
    o = torch.empty((N, B, S, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((N, B, H, S), dtype=torch.float32, device=dev)
    ws = ra.new_workspace(max(ra.ra_ring_attn_workspace_bytes(B, L, H, d, N),
                              ra.ra_ring_attn_bwd_workspace_bytes(B, L, H, d, N)))
    if cu is None:
        ra.ra_ring_attn_fwd_gqa(qs, ks, vs, o, lse, B, L, H, Hkv, d, N, layout, causal, workspace=ws)
    else:
        ra.ra_ring_attn_fwd_varlen(qs, ks, vs, o, lse, cu_dev, L, H, Hkv, d, N, layout, causal, workspace=ws)
    dq = torch.empty_like(o)
    dk = torch.empty((N, B, S, Hkv, d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    ra.ra_ring_attn_bwd(qs, ks, vs, o, dos, lse, dq, dk, dv, B, L, H, Hkv, d, N, layout, causal,
                        cu_seqlens=cu_dev, workspace=ws)
    ra.ra_check_status(ws)

    def unshard(x):
        y = torch.empty((B, L, x.shape[3], d), dtype=torch.float32, device=dev)
        ra.ra_shard_permute(x, y, ra.RA_SHARDS_TO_SEQ, layout, B, L, x.shape[3], d, N)
        return y.cpu().numpy()

    return unshard(dq), unshard(dk), unshard(dv)


CASES = [
    # B, L, H, Hkv, d, N, layout, causal, packed
    (1, 512, 2, 2, 128, 4, "contiguous", True, None),
    (1, 1024, 2, 2, 128, 4, "striped", True, None),
    (2, 768, 2, 2, 64, 3, "zigzag", True, None),
    (1, 640, 4, 2, 128, 2, "striped", False, None),
    (1, 1200, 4, 1, 128, 4, "contiguous", True, None),    # MQA, S = 300 ragged
    (1, 1024, 2, 2, 128, 4, "striped", True, 9),          # packed sequences
]


@pytest.mark.parametrize("B,L,H,Hkv,d,N,layout,causal,packed", CASES)
def test_backward_matches_oracle(ralib, gpu, B, L, H, Hkv, d, N, layout, causal, packed):
    q = randn_bf16((B, L, H, d), L + 11)
    k = randn_bf16((B, L, Hkv, d), L + 12)
    v = randn_bf16((B, L, Hkv, d), L + 13)
    do = randn_bf16((B, L, H, d), L + 14)
    cu = None if packed is None else make_cu_seqlens(L, packed, seed=L).numpy()
    dq, dk, dv = run_bwd(ralib, q, k, v, do, N, layout, causal, cu)
    rq, rk, rv = attention_backward(q, k, v, do, causal, cu_seqlens=cu)
    assert_grad_close(dq, rq, "dQ")
    assert_grad_close(dk, rk, "dK")
    assert_grad_close(dv, rv, "dV")
