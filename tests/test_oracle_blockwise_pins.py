"""Pins of the blockwise combination rules against one-shot softmax.

"From Ring Attention to DeepSpeed Ulysses to USP" (jsqmd.com/news/734632),
§3.2: the online (m, l, O) recursion gives the same result for any order and
any split of the KV blocks as one softmax over all keys; §6.3: the LSE merge
of two normalised partial results.
"""
import math

import numpy as np
import pytest

from synthetic_inputs import randn_bf16, random_ints, random_perm


def _scores(q, k, scale, q_pos, k_pos, causal):
    z = (q.double().numpy() @ k.double().numpy().T) * scale
    if causal:
        z = np.where(k_pos[None, :] <= q_pos[:, None], z, -np.inf)
    return z


def _random_splits(nk, nblocks, seed):
    cuts = sorted(set(random_ints(nblocks - 1, 1, nk, seed).tolist()))
    return cuts


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("trial", range(6))
def test_recursion_and_merge_equal_one_shot(ora, causal, trial):
    nq, nk, d = 19, 53, 16
    q = randn_bf16((nq, d), 100 + trial)
    k = randn_bf16((nk, d), 200 + trial)
    v = randn_bf16((nk, d), 300 + trial)
    # queries sit at positions spread over the keys so causal rows have ragged key sets
    q_pos = np.sort(random_ints(nq, 0, nk, 400 + trial).numpy())
    k_pos = np.arange(nk)
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = ora.attention(q[:, None], k[:, None], v[:, None], q_pos=q_pos, k_pos=k_pos,
                                   causal=causal, scale=scale)
    o_ref, lse_ref = o_ref[:, 0], lse_ref[:, 0]
    z = _scores(q, k, scale, q_pos, k_pos, causal)
    vf = v.double().numpy()
    splits = _random_splits(nk, 2 + trial, 500 + trial)
    order = random_perm(len(splits) + 1, 600 + trial).tolist()
    o1, lse1 = ora.blockwise.softmax_blockwise(z, vf, splits, order)
    o2, lse2 = ora.blockwise.lse_merge_blockwise(z, vf, splits, order)
    np.testing.assert_allclose(o1, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse1, lse_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o2, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse_ref, rtol=0, atol=1e-12)


def test_lse_is_m_plus_ln_l():
    import oracle.blockwise as bw
    z = np.array([[0.5, -1.0, 2.0], [3.0, 3.0, -np.inf]])
    v = np.eye(3)
    st = bw.online_update(bw.init_state(2, 3), z, v)
    m, l, _ = st
    np.testing.assert_allclose(m, [2.0, 3.0])
    np.testing.assert_allclose(l, [math.exp(-1.5) + math.exp(-3.0) + 1.0, 2.0], rtol=1e-15)
    np.testing.assert_allclose(bw.state_lse(st), [2.0 + math.log(l[0]), 3.0 + math.log(2.0)], rtol=1e-15)


def test_merge_closed_forms():
    import oracle.blockwise as bw
    oa = np.array([[1.0, 2.0]])
    ob = np.array([[3.0, 6.0]])
    # equal lse: the two halves carry equal weight, lse grows by ln 2
    o, lse = bw.lse_merge(oa, np.array([0.7]), ob, np.array([0.7]))
    np.testing.assert_allclose(o, [[2.0, 4.0]], rtol=1e-15)
    np.testing.assert_allclose(lse, [0.7 + math.log(2.0)], rtol=1e-15)
    # lse_b = lse_a + ln 3: weights 1/4 and 3/4
    o, lse = bw.lse_merge(oa, np.array([0.0]), ob, np.array([math.log(3.0)]))
    np.testing.assert_allclose(o, [[2.5, 5.0]], rtol=1e-14)
    np.testing.assert_allclose(lse, [math.log(4.0)], rtol=1e-15)


def test_empty_blocks_merge_without_nan():
    import oracle.blockwise as bw
    empty_o = np.zeros((1, 2))
    ninf = np.array([-np.inf])
    o, lse = bw.lse_merge(empty_o, ninf, empty_o, ninf)
    assert np.all(o == 0) and np.isneginf(lse[0])
    full_o = np.array([[1.5, -2.0]])
    o, lse = bw.lse_merge(empty_o, ninf, full_o, np.array([0.25]))
    np.testing.assert_array_equal(o, full_o)
    assert lse[0] == 0.25
    o, lse = bw.lse_merge(full_o, np.array([0.25]), empty_o, ninf)
    np.testing.assert_array_equal(o, full_o)
    # a fully masked block in the recursion leaves the state untouched
    st = bw.online_update(bw.init_state(1, 2), np.array([[-np.inf, -np.inf]]), np.ones((2, 2)))
    assert np.isneginf(st[0][0]) and st[1][0] == 0 and np.all(st[2] == 0)


def test_merge_catches_planted_sign_error():
    """A merge with the exponent's sign flipped must fail the one-shot pin."""
    import oracle.blockwise as bw
    z = np.array([[0.1, 1.3, -0.4, 2.2]])
    v = np.arange(8.0).reshape(4, 2)
    p = np.exp(z - z.max())
    o_ref = (p @ v) / p.sum()
    a = bw.online_update(bw.init_state(1, 2), z[:, :2], v[:2])
    b = bw.online_update(bw.init_state(1, 2), z[:, 2:], v[2:])
    la, lb = bw.state_lse(a), bw.state_lse(b)
    lse = np.maximum(la, lb) + np.log1p(np.exp(-abs(la - lb)))
    bad = a[2] * np.exp(lse - la)[:, None] + b[2] * np.exp(lse - lb)[:, None]
    good, _ = bw.lse_merge(a[2], la, b[2], lb)
    np.testing.assert_allclose(good, o_ref, rtol=1e-14)
    assert np.abs(bad - o_ref).max() > 1e-2
