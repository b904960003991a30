"""Pins of the fp64 attention oracle against values fixed by the pages and by mathematics.

Definition pinned: "From Ring Attention to DeepSpeed Ulysses to USP"
(jsqmd.com/news/734632), §2 (softmax(QK^T/sqrt(d_k)) V), §3.4 (causal mask),
§6.3 (natural-log LSE).
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from synthetic_inputs import make_qkv, randn_bf16


def _bits(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    return t


def test_hand_2x2(ora):
    q = _bits([[[1.0, 0.0]], [[0.0, 1.0]]])
    k = q.clone()
    v = _bits([[[1.0, 2.0]], [[3.0, 4.0]]])
    rows = read_golden("hand_2x2.txt")
    assert len(rows) == 5
    for case, scale, causal, row, o0, o1, lse in rows:
        o, l = ora.attention(q, k, v, causal=bool(int(causal)), scale=float(scale))
        r = int(row)
        assert o[r, 0, 0] == pytest.approx(float(o0), abs=1e-14)
        assert o[r, 0, 1] == pytest.approx(float(o1), abs=1e-14)
        assert l[r, 0] == pytest.approx(float(lse), abs=1e-14)


def _direct_softmax_mp(q, k, v, scale, causal):
    """Attention by the textbook formula without max-subtraction, in 60-digit arithmetic."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    qf = q.float().numpy().astype(np.float64)
    kf = k.float().numpy().astype(np.float64)
    vf = v.float().numpy().astype(np.float64)
    L, H, d = qf.shape
    O = np.zeros((L, H, d))
    LSE = np.zeros((L, H))
    for t in range(L):
        for h in range(H):
            keys = range(t + 1) if causal else range(L)
            w = []
            for u in keys:
                dot = mpmath.fsum(mpmath.mpf(qf[t, h, e]) * mpmath.mpf(kf[u, h, e]) for e in range(d))
                w.append(mpmath.exp(dot * mpmath.mpf(scale)))
            z = mpmath.fsum(w)
            for e in range(d):
                O[t, h, e] = float(mpmath.fsum(wi * mpmath.mpf(vf[u, h, e]) for wi, u in zip(w, keys)) / z)
            LSE[t, h] = float(mpmath.log(z))
    return O, LSE


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L,H,d,seed", [(5, 1, 4, 11), (12, 2, 8, 12), (16, 2, 6, 13)])
def test_brute_force_direct_softmax(ora, causal, L, H, d, seed):
    q = randn_bf16((L, H, d), seed)
    k = randn_bf16((L, H, d), seed + 100)
    v = randn_bf16((L, H, d), seed + 200)
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = _direct_softmax_mp(q, k, v, scale, causal)
    o, lse = ora.attention(q, k, v, causal=causal)          # default scale 1/sqrt(d)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_closed_form_zero_queries(ora, causal):
    """Q = 0: every allowed score is 0, so O_t is the mean of the allowed v and LSE_t = ln |A(t)|."""
    L, H, d = 37, 3, 16
    q = torch.zeros((L, H, d), dtype=torch.bfloat16)
    k = randn_bf16((L, H, d), 5)
    v = randn_bf16((L, H, d), 6)
    o, lse = ora.attention(q, k, v, causal=causal)
    vf = v.double().numpy()
    for t in range(L):
        n = t + 1 if causal else L
        np.testing.assert_allclose(o[t], vf[:n].mean(axis=0), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[t], np.full(H, math.log(n)), rtol=0, atol=1e-13)


def test_closed_form_constant_values(ora):
    """V rows all equal to c: every output row is c, whatever the scores."""
    L, H, d = 29, 2, 8
    q = randn_bf16((L, H, d), 7)
    k = randn_bf16((L, H, d), 8)
    c = randn_bf16((1, H, d), 9)
    v = c.expand(L, H, d).contiguous()
    for causal in (False, True):
        o, _ = ora.attention(q, k, v, causal=causal)
        np.testing.assert_allclose(o, np.broadcast_to(c.double().numpy(), o.shape), rtol=0, atol=1e-13)


def test_closed_form_first_causal_row(ora):
    """Causal row 0 sees only key 0: O_0 = v_0 and LSE_0 = scale * q_0 . k_0."""
    L, H, d = 9, 2, 32
    q = randn_bf16((L, H, d), 21)
    k = randn_bf16((L, H, d), 22)
    v = randn_bf16((L, H, d), 23)
    o, lse = ora.attention(q, k, v, causal=True)
    np.testing.assert_allclose(o[0], v[0].double().numpy(), rtol=0, atol=1e-15)
    qk = (q[0].double() * k[0].double()).sum(-1).numpy() / math.sqrt(d)
    np.testing.assert_allclose(lse[0], qk, rtol=0, atol=1e-14)


def test_key_order_and_positions(ora):
    """The result depends on the key set and positions only: shuffling the key rows
    together with their positions leaves every output unchanged."""
    L, H, d = 24, 2, 16
    q, k, v, _ = make_qkv(1, L, H, d, seed=31)
    q, k, v = q[0], k[0], v[0]
    perm = torch.randperm(L, generator=torch.Generator().manual_seed(3)).numpy()
    o_a, lse_a = ora.attention(q, k, v, causal=True)
    o_b, lse_b = ora.attention(q, k[perm], v[perm], k_pos=np.arange(L)[perm], causal=True)
    np.testing.assert_allclose(o_a, o_b, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_a, lse_b, rtol=0, atol=1e-13)


def test_fully_masked_row_is_empty(ora):
    q = randn_bf16((2, 1, 4), 1)
    k = randn_bf16((3, 1, 4), 2)
    v = randn_bf16((3, 1, 4), 3)
    o, lse = ora.attention(q, k, v, q_pos=np.array([0, 5]), k_pos=np.array([1, 2, 3]), causal=True)
    assert np.isneginf(lse[0, 0]) and np.all(o[0] == 0)
    assert np.isfinite(lse[1, 0])


# --- sensitivity: a planted mistake in the oracle's inputs must fail a pin ----------------

def test_pins_catch_wrong_scale(ora):
    q = _bits([[[1.0, 0.0]], [[0.0, 1.0]]])
    v = _bits([[[1.0, 2.0]], [[3.0, 4.0]]])
    o, _ = ora.attention(q, q, v, scale=2.0)          # the pin expects scale 1
    assert abs(o[0, 0, 0] - 1.5378828427399902) > 1e-3


def test_pins_catch_swapped_operands(ora):
    L, H, d = 29, 2, 8
    q = randn_bf16((L, H, d), 7)
    k = randn_bf16((L, H, d), 8)
    c = randn_bf16((1, H, d), 9)
    v = c.expand(L, H, d).contiguous()
    o, _ = ora.attention(q, v, k)                      # K and V transposed
    assert np.abs(o - c.double().numpy()).max() > 1e-2


def test_pins_catch_off_by_one_mask(ora):
    L, H, d = 9, 2, 32
    q = randn_bf16((L, H, d), 21)
    k = randn_bf16((L, H, d), 22)
    v = randn_bf16((L, H, d), 23)
    # a mask that also lets row t see key t+1
    o, _ = ora.attention(q, k, v, q_pos=np.arange(L) + 1, causal=True)
    assert np.abs(o[0] - v[0].double().numpy()).max() > 1e-2


# --- grouped-query attention ("From Ring Attention to DeepSpeed Ulysses to USP", §5.3) ---

def test_gqa_hand_case(ora):
    """Two query heads share one key/value head: both rows follow the 2x2 hand case."""
    q = _bits([[[1.0, 0.0], [1.0, 0.0]], [[0.0, 1.0], [0.0, 1.0]]])     # [L=2, H=2, d=2]
    k = _bits([[[1.0, 0.0]], [[0.0, 1.0]]])                              # [L=2, Hkv=1, d=2]
    v = _bits([[[1.0, 2.0]], [[3.0, 4.0]]])
    rows = {r[0] + r[3]: r for r in read_golden("hand_2x2.txt")}
    o, lse = ora.attention(q, k, v, scale=1.0)
    for h in range(2):
        assert o[0, h, 0] == pytest.approx(float(rows["noncausal0"][4]), abs=1e-14)
        assert o[1, h, 1] == pytest.approx(float(rows["noncausal1"][5]), abs=1e-14)
        assert lse[0, h] == pytest.approx(float(rows["noncausal0"][6]), abs=1e-14)


def test_gqa_zero_queries_closed_form(ora):
    """Q = 0 with 4 query heads per key/value head: head h averages v of head h // 4."""
    L, H, Hkv, d = 21, 8, 2, 16
    q = torch.zeros((L, H, d), dtype=torch.bfloat16)
    k = randn_bf16((L, Hkv, d), 41)
    v = randn_bf16((L, Hkv, d), 42)
    o, lse = ora.attention(q, k, v, causal=True)
    vf = v.double().numpy()
    for t in range(L):
        for h in range(H):
            np.testing.assert_allclose(o[t, h], vf[:t + 1, h // 4].mean(axis=0), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[t], np.full(H, math.log(t + 1)), rtol=0, atol=1e-13)


def test_gqa_rejects_bad_head_counts(ora):
    q = randn_bf16((3, 3, 4), 1)
    k = randn_bf16((3, 2, 4), 2)
    with pytest.raises((ValueError, AssertionError)):
        ora.attention(q, k, k)


# --- packed variable-length sequences ---------------------------------------------------

def test_varlen_single_token_sequences(ora):
    """Every token its own sequence: O_t = v_t and LSE_t = scale * q_t . k_t, causal or not."""
    L, H, d = 6, 2, 8
    q, k, v = randn_bf16((1, L, H, d), 61), randn_bf16((1, L, H, d), 62), randn_bf16((1, L, H, d), 63)
    for causal in (False, True):
        o, lse = ora.full_attention(q, k, v, causal=causal, cu_seqlens=np.arange(L + 1))
        np.testing.assert_allclose(o[0], v[0].double().numpy(), rtol=0, atol=1e-15)
        qk = (q[0].double() * k[0].double()).sum(-1).numpy() / math.sqrt(d)
        np.testing.assert_allclose(lse[0], qk.T, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_separate_sequences(ora, causal):
    """Packed attention equals attention run on each sequence on its own, stitched back;
    empty sequences are allowed."""
    L, H, d = 40, 2, 16
    cu = np.array([0, 7, 7, 19, 20, 40])
    q, k, v = randn_bf16((1, L, H, d), 71), randn_bf16((1, L, H, d), 72), randn_bf16((1, L, H, d), 73)
    o, lse = ora.full_attention(q, k, v, causal=causal, cu_seqlens=cu)
    for a, b in zip(cu[:-1], cu[1:]):
        if a == b:
            continue
        o_s, lse_s = ora.full_attention(q[:, a:b], k[:, a:b], v[:, a:b], causal=causal)
        np.testing.assert_allclose(o[:, a:b], o_s, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, a:b], lse_s, rtol=0, atol=1e-13)


def test_varlen_zero_queries_closed_form(ora):
    """Q = 0, causal, packed: O_t is the mean of v over its own sequence up to t."""
    L, H, d = 30, 1, 8
    cu = np.array([0, 11, 12, 30])
    q = torch.zeros((1, L, H, d), dtype=torch.bfloat16)
    k, v = randn_bf16((1, L, H, d), 81), randn_bf16((1, L, H, d), 82)
    o, lse = ora.full_attention(q, k, v, causal=True, cu_seqlens=cu)
    vf = v.double().numpy()[0]
    for t in range(L):
        s0 = cu[np.searchsorted(cu, t, side="right") - 1]
        np.testing.assert_allclose(o[0, t], vf[s0:t + 1].mean(axis=0), rtol=0, atol=1e-13)
        assert lse[0, 0, t] == pytest.approx(math.log(t + 1 - s0), abs=1e-13)
