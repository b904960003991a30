"""fp64 gradients of softmax attention -- TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The pages describe the forward pass only; the backward here is the plain
derivative of the attention of "From Ring Attention to DeepSpeed Ulysses to
USP" (jsqmd.com/news/734632), §2, O = softmax(Q K^T * scale) V, under the
same masks as the forward (causal by position, optional packed sequences,
grouped key/value heads).  For one head, with P the row-softmax of the masked
scores and dO the gradient of O:
    dV = P^T dO
    dP = dO V^T
    dS = P * (dP - rowsum(P * dP))          (softmax Jacobian, row by row)
    dQ = dS K * scale,   dK = dS^T Q * scale
With grouped key/value heads, a key/value head's dK and dV add up over the
query heads that read it.  Every step is a numpy fp64 matrix product or an
elementwise operation on the whole [L, L] matrices: no blocking, no online
softmax.
"""
import numpy as np


def _f64(x):
    if isinstance(x, np.ndarray):
        return x.astype(np.float64)
    return x.detach().cpu().double().numpy()


def attention_backward(q, k, v, do, causal, scale=None, cu_seqlens=None):
    """q, do [B, L, H, d]; k, v [B, L, Hkv, d] (bf16 tensors or arrays).

    Returns (dq [B, L, H, d], dk [B, L, Hkv, d], dv [B, L, Hkv, d]) in float64.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    group = H // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    allowed = np.ones((L, L), dtype=bool)
    if causal:
        allowed &= np.tril(np.ones((L, L), dtype=bool))
    if cu_seqlens is not None:
        seg = np.searchsorted(np.asarray(cu_seqlens), np.arange(L), side="right") - 1
        allowed &= seg[:, None] == seg[None, :]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            kv = h // group
            s = (q[b, :, h] @ k[b, :, kv].T) * scale
            s = np.where(allowed, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            m = np.where(np.isfinite(m), m, 0.0)
            e = np.exp(s - m)
            den = e.sum(axis=1, keepdims=True)
            p = np.where(den > 0, e / np.where(den > 0, den, 1.0), 0.0)
            dP = do[b, :, h] @ v[b, :, kv].T
            dS = p * (dP - (p * dP).sum(axis=1, keepdims=True))
            dv[b, :, kv] += p.T @ do[b, :, h]
            dq[b, :, h] = dS @ k[b, :, kv] * scale
            dk[b, :, kv] += dS.T @ q[b, :, h] * scale
    return dq, dk, dv


def attention_backward_rows(q, k, v, do, causal, b, h, rows, scale=None, cu_seqlens=None, chunk=64):
    """The same derivative restricted to the query rows ``rows`` of batch b and
    query head h, for inputs too long for the [L, L] matrices.

    A query row's softmax, dP, dS and dQ depend only on that row and all keys,
    so each row is computed whole (every visible key in one product); rows are
    taken ``chunk`` at a time only to bound memory.  Returns
        dq      [len(rows), d]   exact dQ of those rows,
        dk_part [L, d]           sum over those rows of dS[row, key] * q_row * scale,
        dv_part [L, d]           sum over those rows of P[row, key] * dO_row,
    the rows' contributions to dK and dV of key/value head h // (H / Hkv).  A
    key every one of whose seeing rows (over all query heads of the group) is
    passed gets its exact dK and dV as the sum of those contributions.
    """
    B, L, H, d = q.shape
    Hkv = k.shape[2]
    kv = h // (H // Hkv)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.asarray(rows, dtype=np.int64)
    kk = _f64(k[b, :, kv])
    vv = _f64(v[b, :, kv])
    seg = None
    if cu_seqlens is not None:
        seg = np.searchsorted(np.asarray(cu_seqlens), np.arange(L), side="right") - 1
    keys = np.arange(L)
    dq = np.zeros((len(rows), d))
    dk_part = np.zeros((L, d))
    dv_part = np.zeros((L, d))
    for c0 in range(0, len(rows), chunk):
        r = rows[c0:c0 + chunk]
        qr = _f64(q[b, r, h])
        dor = _f64(do[b, r, h])
        allowed = np.ones((len(r), L), dtype=bool)
        if causal:
            allowed &= keys[None, :] <= r[:, None]
        if seg is not None:
            allowed &= seg[None, :] == seg[r][:, None]
        s = np.where(allowed, (qr @ kk.T) * scale, -np.inf)
        m = s.max(axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.exp(s - m)
        den = e.sum(axis=1, keepdims=True)
        p = np.where(den > 0, e / np.where(den > 0, den, 1.0), 0.0)
        dP = dor @ vv.T
        dS = p * (dP - (p * dP).sum(axis=1, keepdims=True))
        dq[c0:c0 + len(r)] = dS @ kk * scale
        dk_part += dS.T @ qr * scale
        dv_part += p.T @ dor
    return dq, dk_part, dv_part
