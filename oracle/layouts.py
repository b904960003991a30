"""Token-to-rank assignments and the Ulysses transpose, as plain index formulas.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Each function builds
an explicit index table with numpy and applies it with fancy indexing, so a
reader can check every formula against the pages by eye.  No code here is
shared with the CUDA path.

Notation: L tokens, N ring ranks, S = L / N tokens per rank, rank r holds
local tokens s = 0..S-1.  Full-sequence tensors are [B, L, H, d] (the pages'
[bs, seq, heads, head_dim]); shard stacks are [N, B, S, H, d].

Sources:
  * contiguous and striped -- "From Ring Attention to DeepSpeed Ulysses to USP"
    (jsqmd.com/news/734632), §4 "Striped Attention": with 16 tokens on 4 GPUs
    contiguous gives GPU r the tokens 4r..4r+3 and striped gives GPU r the
    tokens r, r+4, r+8, r+12.
  * zigzag -- same article, §6.1 "Zigzag load-balanced split": the sequence is
    cut into 2N equal chunks and rank k holds chunks k and 2N-1-k, in that
    order.
  * Ulysses -- same article, §5.1: before the all-to-all each rank holds
    [bs, L/P, H, d] (its sequence slice, all heads); after it each rank holds
    [bs, L, H/P, d] (the whole sequence, one head slice); §7.2 (USP-Attn):
    the all-to-all scatters the head dimension and gathers the sequence
    dimension inside each Ulysses group, giving [bs, L/N_ring, H/N_ulysses, d].
"""
import numpy as np

LAYOUTS = ("contiguous", "striped", "zigzag")


def global_position(layout, r, s, N, S):
    """Global token index of local token ``s`` (array or int) on ring rank ``r``."""
    s = np.asarray(s, dtype=np.int64)
    if layout == "contiguous":
        return r * S + s
    if layout == "striped":
        return s * N + r
    if layout == "zigzag":
        if S % 2:
            raise ValueError("zigzag needs an even shard length")
        C = S // 2
        return np.where(s < C, r * C + s, (2 * N - 1 - r) * C + (s - C))
    raise ValueError(layout)


def rank_positions(layout, N, L):
    """[N, S] table: positions[r, s] = global token of local token s on rank r."""
    if L % N:
        raise ValueError("N must divide L")
    S = L // N
    s = np.arange(S, dtype=np.int64)
    return np.stack([global_position(layout, r, s, N, S) for r in range(N)])


def seq_to_shards(x, layout, N):
    """[B, L, ...] -> [N, B, S, ...]: shard r, local token s is token positions[r, s]."""
    x = np.asarray(x)
    pos = rank_positions(layout, N, x.shape[1])
    return np.stack([x[:, pos[r]] for r in range(N)])


def shards_to_seq(y, layout):
    """Inverse of seq_to_shards: [N, B, S, ...] -> [B, L, ...]."""
    y = np.asarray(y)
    N, S = y.shape[0], y.shape[2]
    pos = rank_positions(layout, N, N * S)
    out = np.empty((y.shape[1], N * S) + y.shape[3:], dtype=y.dtype)
    for r in range(N):
        out[:, pos[r]] = y[r]
    return out


def usp_seq_to_shards(x, layout, R, U):
    """USP sequence-sharded state: [B, L, H, d] -> [U*R, B, L/(U*R), H, d].

    Global rank p = u*R + r sits in row u, column r of the USP process grid
    (same article, §7.1: Ulysses along the columns, the ring along the rows).
    Ring rank r owns the ``layout`` token list of length L/R; Ulysses member u
    of that column holds the u-th contiguous piece of it.
    """
    ring = seq_to_shards(x, layout, R)               # [R, B, L/R, H, d]
    B, LR = ring.shape[1], ring.shape[2]
    if LR % U:
        raise ValueError("U must divide L/R")
    Lp = LR // U
    out = np.empty((U * R, B, Lp) + ring.shape[3:], dtype=ring.dtype)
    for u in range(U):
        for r in range(R):
            out[u * R + r] = ring[r][:, u * Lp:(u + 1) * Lp]
    return out


def usp_shards_to_seq(y, layout, R, U):
    """Inverse of usp_seq_to_shards."""
    y = np.asarray(y)
    P, B, Lp = y.shape[0], y.shape[1], y.shape[2]
    assert P == U * R
    ring = np.empty((R, B, U * Lp) + y.shape[3:], dtype=y.dtype)
    for u in range(U):
        for r in range(R):
            ring[r][:, u * Lp:(u + 1) * Lp] = y[u * R + r]
    return shards_to_seq(ring, layout)


def ulysses_seq_to_head(x, R, U):
    """All-to-all inside each Ulysses group, as a local gather.

    in : [U*R, B, Lp, H, d]      rank p = u*R + r holds Lp tokens, all H heads
    out: [R, U, B, U*Lp, H/U, d] block (r, u') holds, for the U members of
         column r in order u = 0..U-1, their tokens, heads u'*H/U..(u'+1)*H/U.
    out[r, u', b, u*Lp + s, hh] = in[u*R + r, b, s, u'*(H/U) + hh]
    """
    x = np.asarray(x)
    P, B, Lp, H = x.shape[:4]
    if H % U:
        raise ValueError("U must divide H")
    Hu = H // U
    out = np.empty((R, U, B, U * Lp, Hu) + x.shape[4:], dtype=x.dtype)
    for r in range(R):
        for up in range(U):
            for u in range(U):
                out[r, up, :, u * Lp:(u + 1) * Lp] = x[u * R + r, :, :, up * Hu:(up + 1) * Hu]
    return out


def ulysses_head_to_seq(y, R, U):
    """Inverse all-to-all: [R, U, B, U*Lp, H/U, d] -> [U*R, B, Lp, H, d]."""
    y = np.asarray(y)
    B, LR, Hu = y.shape[2], y.shape[3], y.shape[4]
    Lp = LR // U
    out = np.empty((U * R, B, Lp, Hu * U) + y.shape[5:], dtype=y.dtype)
    for r in range(R):
        for up in range(U):
            for u in range(U):
                out[u * R + r, :, :, up * Hu:(up + 1) * Hu] = y[r, up, :, u * Lp:(u + 1) * Lp]
    return out


def lse_to_seq(lse, layout, R, U, B):
    """Ring-output LSE [R, U*B, H/U, L/R] -> [B, H, L] in original token order.

    Block (r, u*B + b) is the ring shard r of Ulysses head group u, batch b
    (U = 1 is the plain [N, B, H, S] -> [B, H, L] case).
    """
    lse = np.asarray(lse)
    Rr, UB, Hu, LR = lse.shape
    assert Rr == R and UB == U * B
    pos = rank_positions(layout, R, R * LR)
    out = np.empty((B, Hu * U, R * LR), dtype=lse.dtype)
    for r in range(R):
        for u in range(U):
            for b in range(B):
                out[b, u * Hu:(u + 1) * Hu][:, pos[r]] = lse[r, u * B + b]
    return out
