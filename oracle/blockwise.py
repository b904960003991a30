"""Blockwise softmax in fp64: the online (m, l, O) recursion and the LSE merge.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  These are the two
combination rules the ring sweep relies on, written out in the pages' order
and notation with numpy.  They serve the invariance pins of the oracle and
are the oracle of ``ra_lse_merge``.  Nothing here is shared with the CUDA
path.

Source: "From Ring Attention to DeepSpeed Ulysses to USP"
(jsqmd.com/news/734632):
  §3.2 "Online softmax: the mathematical basis" -- for a query x and the
  (j+1)-th KV block with scores z_k = q_x . k_k / sqrt(d):
      m_{j+1} = max(m_j, max_k z_k)
      l_{j+1} = l_j e^{m_j - m_{j+1}} + sum_k e^{z_k - m_{j+1}}
      O_{j+1} = (O_j l_j e^{m_j - m_{j+1}} + sum_k e^{z_k - m_{j+1}} v_k) / l_{j+1}
  §6.3 "LSE merge (numerically stable)":
      lse = max(lse_A, lse_B) + log(1 + e^{-|lse_A - lse_B|})
      O   = O_A e^{lse_A - lse} + O_B e^{lse_B - lse}
  (the article's rendering of the second line is garbled; it is read as the
  weighted sum above, with no division, because both O's are already
  normalised.)

An empty block (every key masked) is the state (m = -inf, l = 0, O = 0),
i.e. lse = -inf; it contributes weight zero and the merge of two empty
states stays empty, with no NaN.
"""
import numpy as np


def init_state(rows, d):
    return (np.full(rows, -np.inf), np.zeros(rows), np.zeros((rows, d)))


def online_update(state, z, v):
    """One step of the (m, l, O) recursion.

    state: (m [rows], l [rows], O [rows, d]); z: [rows, nk] scores of the new
    block (-inf where masked); v: [nk, d] values of the new block.
    """
    m, l, O = state
    z = np.asarray(z, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    block_max = z.max(axis=1) if z.shape[1] else np.full(z.shape[0], -np.inf)
    m_new = np.maximum(m, block_max)
    # reference point for the exponentials; a row that is still empty keeps
    # every weight at exactly zero
    ref = np.where(np.isfinite(m_new), m_new, 0.0)
    carry = np.exp(m - ref)                      # e^{m_j - m_{j+1}}
    p = np.exp(z - ref[:, None])                 # e^{z_k - m_{j+1}}
    l_new = l * carry + p.sum(axis=1)
    num = O * (l * carry)[:, None] + p @ v
    with np.errstate(invalid="ignore", divide="ignore"):
        O_new = np.where(l_new[:, None] > 0, num / np.where(l_new > 0, l_new, 1.0)[:, None], 0.0)
    return m_new, l_new, O_new


def state_lse(state):
    """lse = m + ln l for a recursion state (-inf for an empty row)."""
    m, l, _ = state
    with np.errstate(divide="ignore"):
        return np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)


def lse_merge(o_a, lse_a, o_b, lse_b):
    """Merge two normalised partial results by their log-sum-exp."""
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    hi = np.maximum(lse_a, lse_b)
    with np.errstate(invalid="ignore"):
        gap = np.abs(lse_a - lse_b)
    both_empty = np.isneginf(hi)
    gap = np.where(both_empty, np.inf, gap)      # (-inf) - (-inf) is not a number
    lse = np.where(both_empty, -np.inf, hi + np.log1p(np.exp(-gap)))
    ref = np.where(both_empty, 0.0, lse)
    w_a = np.exp(lse_a - ref)
    w_b = np.exp(lse_b - ref)
    o = o_a * w_a[..., None] + o_b * w_b[..., None]
    return o, lse


def softmax_blockwise(z, v, splits, order):
    """Run the §3.2 recursion over the key blocks given by ``splits`` in ``order``.

    z: [rows, nk] scores (-inf where masked); v: [nk, d];
    splits: sorted cut points in (0, nk); order: permutation of the blocks.
    Returns (O, lse).
    """
    bounds = [0] + list(splits) + [z.shape[1]]
    blocks = [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]
    st = init_state(z.shape[0], v.shape[1])
    for bi in order:
        a, b = blocks[bi]
        st = online_update(st, z[:, a:b], v[a:b])
    return st[2], state_lse(st)


def lse_merge_blockwise(z, v, splits, order):
    """Per block: normalised softmax output and lse; then fold with §6.3's merge."""
    bounds = [0] + list(splits) + [z.shape[1]]
    blocks = [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]
    o = np.zeros((z.shape[0], v.shape[1]))
    lse = np.full(z.shape[0], -np.inf)
    for bi in order:
        a, b = blocks[bi]
        part = online_update(init_state(z.shape[0], v.shape[1]), z[:, a:b], v[a:b])
        o, lse = lse_merge(o, lse, part[2], state_lse(part))
    return o, lse
