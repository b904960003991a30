"""Pins of the token-assignment and Ulysses index formulas against the pages' examples.

"From Ring Attention to DeepSpeed Ulysses to USP" (jsqmd.com/news/734632):
§4 (contiguous vs striped, 16 tokens on 4 GPUs), §5.1 (Ulysses shapes),
§6.1 (zigzag, cp = 4), §7.1 (USP grid), §7.2 (USP-Attn shapes).
"""
import numpy as np
import pytest

from conftest import read_golden
from oracle import layouts as ly


def test_contiguous_and_striped_match_page_example():
    rows = read_golden("contiguous_striped_assignment.txt")
    assert len(rows) == 8
    for layout, gpu, *tokens in rows:
        pos = ly.rank_positions(layout, 4, 16)
        assert pos[int(gpu)].tolist() == [int(t) for t in tokens]


def test_zigzag_matches_page_example():
    rows = read_golden("zigzag_assignment.txt")
    assert len(rows) == 4
    L = 16                      # 2 tokens per chunk, 8 chunks
    for cp, rank, c0, c1 in rows:
        cp, rank = int(cp), int(rank)
        pos = ly.rank_positions("zigzag", cp, L)[rank]
        C = L // (2 * cp)
        want = list(range(int(c0) * C, int(c0) * C + C)) + list(range(int(c1) * C, int(c1) * C + C))
        assert pos.tolist() == want


@pytest.mark.parametrize("layout", ly.LAYOUTS)
@pytest.mark.parametrize("N,L", [(1, 8), (4, 16), (8, 64), (3, 30)])
def test_positions_are_a_permutation_and_round_trip(layout, N, L):
    pos = ly.rank_positions(layout, N, L)
    assert sorted(pos.ravel().tolist()) == list(range(L))
    x = np.arange(2 * L * 3 * 2).reshape(2, L, 3, 2)
    y = ly.seq_to_shards(x, layout, N)
    assert y.shape == (N, 2, L // N, 3, 2)
    np.testing.assert_array_equal(ly.shards_to_seq(y, layout), x)


@pytest.mark.parametrize("layout", ly.LAYOUTS)
def test_positions_increase_within_a_rank(layout):
    # each rank's local order is increasing in global position (the mask reduces to a prefix)
    pos = ly.rank_positions(layout, 8, 128)
    assert np.all(np.diff(pos, axis=1) > 0)


def _causal_pairs_per_rank(layout, N, L):
    pos = ly.rank_positions(layout, N, L)
    return (pos + 1).sum(axis=1)          # token t sees t+1 keys


def test_balance_claims():
    """§3.4: contiguous causal work grows with rank; §4/§6.1: striped and zigzag even it out."""
    N, L = 4, 64
    S = L // N
    c = _causal_pairs_per_rank("contiguous", N, L)
    # exactly (i + 1/2) S^2 + S/2 pairs on rank i
    np.testing.assert_array_equal(c, [(i * S * S) + S * (S + 1) // 2 for i in range(N)])
    z = _causal_pairs_per_rank("zigzag", N, L)
    assert len(set(z.tolist())) == 1
    s = _causal_pairs_per_rank("striped", N, L)
    assert s.max() - s.min() == (N - 1) * S        # rank r pays r extra per local token


def test_usp_grid_matches_page():
    rows = read_golden("usp_grid.txt")
    R = U = 4
    for u, *gpus in rows:
        assert [int(g) for g in gpus] == [int(u) * R + r for r in range(R)]


def test_ulysses_shapes_and_contents():
    """§5.1 with the USP numbering of §7.1/§7.2: before, rank p holds [bs, L/P, H, d];
    after, block (r, u') holds [bs, L/R, H/U, d]: ring shard r's tokens, head slice u'."""
    B, L, H, d, R, U = 2, 48, 4, 3, 3, 2
    x = np.random.default_rng(0).integers(0, 1 << 15, size=(B, L, H, d)).astype(np.uint16)
    seq = ly.usp_seq_to_shards(x, "zigzag", R, U)
    assert seq.shape == (U * R, B, L // (U * R), H, d)
    head = ly.ulysses_seq_to_head(seq, R, U)
    assert head.shape == (R, U, B, L // R, H // U, d)
    ring = ly.seq_to_shards(x, "zigzag", R)          # [R, B, L/R, H, d]
    for r in range(R):
        for up in range(U):
            np.testing.assert_array_equal(head[r, up], ring[r][:, :, up * (H // U):(up + 1) * (H // U)])
    np.testing.assert_array_equal(ly.ulysses_head_to_seq(head, R, U), seq)
    np.testing.assert_array_equal(ly.usp_shards_to_seq(seq, "zigzag", R, U), x)


def test_plain_ulysses_is_page_example():
    """R = 1, U = P: GPU u' after the all-to-all holds the whole sequence, heads u'H/P..(u'+1)H/P."""
    B, L, H, d, P = 1, 16, 8, 2, 4
    x = np.arange(B * L * H * d).reshape(B, L, H, d)
    seq = ly.usp_seq_to_shards(x, "contiguous", 1, P)
    for p in range(P):                             # before: GPU p holds seq p*L/P..(p+1)*L/P, all heads
        np.testing.assert_array_equal(seq[p], x[:, p * (L // P):(p + 1) * (L // P)])
    head = ly.ulysses_seq_to_head(seq, 1, P)
    for up in range(P):
        np.testing.assert_array_equal(head[0, up], x[:, :, up * (H // P):(up + 1) * (H // P)])


@pytest.mark.parametrize("layout", ly.LAYOUTS)
def test_lse_to_seq(layout):
    B, L, H, R, U = 2, 24, 4, 3, 2
    lse = np.random.default_rng(1).standard_normal((B, H, L))
    # build the ring-output order by hand from positions, then undo it
    pos = ly.rank_positions(layout, R, L)
    ring = np.empty((R, U * B, H // U, L // R))
    for r in range(R):
        for u in range(U):
            for b in range(B):
                ring[r, u * B + b] = lse[b, u * (H // U):(u + 1) * (H // U)][:, pos[r]]
    np.testing.assert_array_equal(ly.lse_to_seq(ring, layout, R, U, B), lse)


def test_zigzag_rejects_odd_shards():
    with pytest.raises(ValueError):
        ly.rank_positions("zigzag", 3, 9)
