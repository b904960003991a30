"""Pins of the fp64 attention backward against finite differences and identities."""
import numpy as np
import pytest

from oracle.backward import attention_backward
from synthetic_inputs import randn_bf16


def _forward_plain(q, k, v, causal, seg=None):
    """Attention written out directly (exp / sum, fp64), independent of the backward."""
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    out = np.zeros(q.shape)
    for b in range(B):
        for h in range(H):
            for t in range(L):
                keys = [u for u in range(L) if (not causal or u <= t) and (seg is None or seg[u] == seg[t])]
                w = np.array([np.exp(q[b, t, h] @ k[b, u, h // (H // Hkv)] / np.sqrt(d)) for u in keys])
                out[b, t, h] = (w[:, None] * v[b, keys, h // (H // Hkv)]).sum(0) / w.sum()
    return out


@pytest.mark.parametrize("causal,Hkv,cu", [(False, 2, None), (True, 2, None), (True, 1, [0, 2, 5, 6])])
def test_backward_matches_finite_differences(causal, Hkv, cu):
    B, L, H, d = 1, 6, 2, 4
    rng = np.random.default_rng(7)
    q = rng.standard_normal((B, L, H, d))
    k = rng.standard_normal((B, L, Hkv, d))
    v = rng.standard_normal((B, L, Hkv, d))
    do = rng.standard_normal((B, L, H, d))
    seg = None if cu is None else np.searchsorted(np.array(cu), np.arange(L), side="right") - 1
    dq, dk, dv = attention_backward(q, k, v, do, causal, cu_seqlens=cu)
    eps = 1e-6

    def loss(q_, k_, v_):
        return float((_forward_plain(q_, k_, v_, causal, seg) * do).sum())

    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args_p = [q, k, v]; args_m = [q, k, v]
            which = 0 if x is q else (1 if x is k else 2)
            args_p[which] = xp; args_m[which] = xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-7)


def test_backward_identities():
    """sum_k dK = 0 (each row of dS sums to 0) and sum_k dV = sum_q dO (softmax rows sum to 1)."""
    B, L, H, d = 2, 33, 4, 8
    q, k, v, do = (randn_bf16((B, L, H, d), s) for s in (1, 2, 3, 4))
    for causal in (False, True):
        dq, dk, dv = attention_backward(q, k, v, do, causal)
        np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
        np.testing.assert_allclose(dv.sum(axis=1), do.double().numpy().sum(axis=1), atol=1e-12)


def test_backward_single_key_row():
    """Causal row 0 sees one key: its softmax is constant, so dQ_0 = 0."""
    B, L, H, d = 1, 5, 1, 8
    q, k, v, do = (randn_bf16((B, L, H, d), s) for s in (5, 6, 7, 8))
    dq, _, _ = attention_backward(q, k, v, do, True)
    assert np.abs(dq[0, 0]).max() == 0.0
    assert np.abs(dq[0, 1:]).max() > 0


def test_backward_catches_planted_transpose():
    """Using dS instead of dS^T for dK (a transposed operand) breaks the dK identity."""
    B, L, H, d = 1, 9, 1, 4
    rng = np.random.default_rng(3)
    q, k, v, do = (rng.standard_normal((B, L, H, d)) for _ in range(4))
    dq, dk, dv = attention_backward(q, k, v, do, True)
    s = q[0, :, 0] @ k[0, :, 0].T / 2.0
    s = np.where(np.tril(np.ones((L, L), bool)), s, -np.inf)
    p = np.exp(s - s.max(1, keepdims=True)); p /= p.sum(1, keepdims=True)
    dP = do[0, :, 0] @ v[0, :, 0].T
    dS = p * (dP - (p * dP).sum(1, keepdims=True))
    wrong = dS @ q[0, :, 0] / 2.0
    assert np.abs(wrong - dk[0, :, 0]).max() > 1e-3


@pytest.mark.parametrize("causal,Hkv,cu", [(True, 4, None), (False, 2, None), (True, 1, [0, 17, 18, 40, 70])])
def test_backward_rows_matches_full_backward(causal, Hkv, cu):
    """The row-restricted backward (used at sizes where [L, L] does not fit) against the
    full one, itself pinned by finite differences above: dQ of any rows; with every row
    of every query head of a group passed, dK and dV of the group's key/value head; and
    with causal masking, the exact dK / dV of the last keys from the rows that see them."""
    from oracle.backward import attention_backward_rows
    B, L, H, d = 2, 70, 4, 8
    q, do = (randn_bf16((B, L, H, d), s) for s in (21, 22))
    k, v = (randn_bf16((B, L, Hkv, d), s) for s in (23, 24))
    dq, dk, dv = attention_backward(q, k, v, do, causal, cu_seqlens=cu)
    group = H // Hkv
    rows = np.array([0, 1, 5, 17, 18, 39, 40, 69])
    for b in range(B):
        for h in range(H):
            dq_r, _, _ = attention_backward_rows(q, k, v, do, causal, b, h, rows, cu_seqlens=cu, chunk=3)
            np.testing.assert_allclose(dq_r, dq[b, rows, h], rtol=0, atol=1e-12)
        for kv in range(Hkv):
            heads = range(kv * group, (kv + 1) * group)
            parts = [attention_backward_rows(q, k, v, do, causal, b, h, np.arange(L), cu_seqlens=cu)
                     for h in heads]
            np.testing.assert_allclose(sum(p[1] for p in parts), dk[b, :, kv], rtol=0, atol=1e-12)
            np.testing.assert_allclose(sum(p[2] for p in parts), dv[b, :, kv], rtol=0, atol=1e-12)
            if causal:
                k0 = L - 9
                tail = [attention_backward_rows(q, k, v, do, causal, b, h, np.arange(k0, L), cu_seqlens=cu)
                        for h in heads]
                np.testing.assert_allclose(sum(p[1] for p in tail)[k0:], dk[b, k0:, kv], rtol=0, atol=1e-12)
                np.testing.assert_allclose(sum(p[2] for p in tail)[k0:], dv[b, k0:, kv], rtol=0, atol=1e-12)
