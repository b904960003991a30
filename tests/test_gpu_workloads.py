"""The five standard workloads at full size, through the same calls bench.py times.

Small workloads are compared with the fp64 oracle element by element.  The large
ones are compared on a stratified sample of query rows (every batch and head; the
first and last rows of every shard, zigzag chunk and Ulysses piece; the rows at
scaled keys; random rows), which the oracle computes one by one, and on a
closed form that holds at any size (Q = 0: O_t is the mean of v_0..v_t and
LSE_t = ln(t + 1)).
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.layouts as ly
from conftest import assert_attention_close
from synthetic_inputs import WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu


def gpu_path(ra, q, k, v, N, layout, causal, U=1, rows=None):
    """Shard / Ulysses permutes, fused ring sweep, inverse permutes; returns O and LSE
    in sequence order (only the given rows when ``rows`` is set)."""
    dev = torch.device("cuda:0")
    B, L, H, d = q.shape
    R, P = N, U * N
    sh = []
    for x in (q, k, v):
        xg = x.to(dev)
        y = torch.empty((P, B, L // P, H, d), dtype=torch.bfloat16, device=dev)
        ra.ra_shard_permute(xg, y, ra.RA_SEQ_TO_SHARDS, layout, B, L, H, d, R, U)
        del xg
        if U > 1:
            z = torch.empty((R, U, B, L // R, H // U, d), dtype=torch.bfloat16, device=dev)
            ra.ra_shard_permute(y, z, ra.RA_ULYSSES_SEQ_TO_HEAD, layout, B, L, H, d, R, U)
            y = z
        sh.append(y)
    Bq, Hq = U * B, H // U
    o = torch.empty(sh[0].shape, dtype=torch.float32, device=dev)
    lse = torch.empty((R, Bq, Hq, L // R), dtype=torch.float32, device=dev)
    ws = ra.new_workspace(ra.ra_ring_attn_workspace_bytes(Bq, L, Hq, d, R))
    ra.ra_ring_attn_fwd(*sh, o, lse, Bq, L, Hq, d, R, layout, causal, workspace=ws)
    del sh
    if U > 1:
        o2 = torch.empty((P, B, L // P, H, d), dtype=torch.float32, device=dev)
        ra.ra_shard_permute(o, o2, ra.RA_ULYSSES_HEAD_TO_SEQ, layout, B, L, H, d, R, U)
        o = o2
    o_seq = torch.empty((B, L, H, d), dtype=torch.float32, device=dev)
    ra.ra_shard_permute(o, o_seq, ra.RA_SHARDS_TO_SEQ, layout, B, L, H, d, R, U)
    lse_seq = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    ra.ra_lse_to_seq(lse, lse_seq, layout, B, L, H, R, U)
    ra.ra_check_status(ws)
    if rows is not None:
        idx = torch.as_tensor(rows, device=dev)
        return o_seq[:, idx].cpu().numpy(), lse_seq[:, :, idx].cpu().numpy()
    return o_seq.cpu().numpy(), lse_seq.cpu().numpy()


def sample_rows(w, layout, scaled_rows, n_random=40, seed=0):
    L, N, U = w["L"], w["N"], w.get("U", 1)
    S = L // N
    local = {0, S - 1}
    if layout == "zigzag":
        local |= {S // 2 - 1, S // 2}
    if U > 1:
        Lp = L // (N * U)
        local |= {u * Lp for u in range(U)} | {u * Lp - 1 for u in range(1, U + 1)}
    rows = set()
    for r in range(N):
        rows |= set(ly.global_position(layout, r, np.array(sorted(local)), N, S).tolist())
    for t in np.asarray(scaled_rows).ravel().tolist()[:24]:
        rows |= {t, min(L - 1, t + 1)}
    rng = np.random.default_rng(seed)
    rows |= set(rng.integers(0, L, n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)


CASES = [(name, layout) for name, w in WORKLOADS.items() for layout in w["layouts"]]


@pytest.mark.parametrize("name,layout", CASES)
def test_workload_parity(ralib, gpu, name, layout):
    w = WORKLOADS[name]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    U = w.get("U", 1)
    q, k, v, scaled = make_qkv(B, L, H, d, w["seed"], w["k_scale_frac"])
    full = B * H * L * L <= 2 ** 31
    rows = None if full else sample_rows(w, layout, scaled)
    o, lse = gpu_path(ralib, q, k, v, N, layout, w["causal"], U=U, rows=rows)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=w["causal"], rows=rows)
    assert_attention_close(o, o_ref, lse, lse_ref, "%s/%s" % (name, layout))


@pytest.mark.parametrize("layout", ["striped", "contiguous"])
def test_zero_queries_closed_form_at_full_size(ralib, gpu, layout):
    """Q = 0 on the 128K workload: every row is the running mean of V."""
    w = WORKLOADS["striped_B1_H8_L131072_d128_N16"]
    B, L, H, d, N = w["B"], w["L"], w["H"], w["d"], w["N"]
    _, k, v, _ = make_qkv(B, L, H, d, w["seed"])
    q = torch.zeros_like(k)
    o, lse = gpu_path(ralib, q, k, v, N, layout, True)
    n = np.arange(1, L + 1, dtype=np.float64)
    mean = np.cumsum(v.double().numpy(), axis=1) / n[None, :, None, None]
    err = np.abs(o - mean).max()
    assert err <= 1e-2, err
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(n), lse.shape), rtol=0, atol=1e-3)
