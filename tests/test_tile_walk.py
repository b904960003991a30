"""The attention kernels' own tile walks, counted on the host.

``tests/walk_probe.cu`` runs the unit decode and the key-tile walks of
``ra_positions.cuh`` -- the code the forward kernel and both backward passes run
-- on the CPU and records, for every query row and key/value shard, the keys its
visited tiles let through after the in-tile mask.  Here that is compared with
what the token positions allow ("From Ring Attention to DeepSpeed Ulysses to
USP", jsqmd.com/news/734632: §3.4 a query sees the keys at positions not after
its own; §4 and §6.1 the contiguous, striped and zigzag positions, taken from
``oracle.layouts``; packed sequences, §6.2 and §8: only keys of the query's own
sequence, from ``oracle.segment_ids``):

  * every query row meets every allowed key exactly once over the whole sweep
    (fused, stepwise in N one-step launches, or as N block calls), and no
    disallowed key: the union of visited (query, key) pairs is A(t), with no
    pair twice and none missing;
  * the per-step tile counts the forward's issuers loop over (TileWalk::step_tiles,
    summed one ring step per lane) equal the number of tiles the walk visits;
  * the dK / dV pass reaches every allowed query of every key exactly once, for
    each query head of a key/value group;
  * the launch grid hands out every unit exactly once.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import oracle.layouts as ly
from conftest import ROOT
from synthetic_inputs import make_cu_seqlens

CSRC = os.path.join(ROOT, "sequence_blockwise_softmax_gb300", "csrc")
LAYOUT_IDS = {"contiguous": 0, "striped": 1, "zigzag": 2}
_P, _I = ctypes.c_void_p, ctypes.c_int


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("walk") / "walk_probe.so")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-shared", "-Xcompiler", "-fPIC", "-I",
                    os.path.join(ROOT, "include"), "-I", CSRC, os.path.join(ROOT, "tests", "walk_probe.cu"),
                    "-o", out], check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    lib.ra_test_forward_walk.argtypes = [_I, _I, _I, _I, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]
    lib.ra_test_key_walk.argtypes = [_I, _I, _I, _I, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]
    return lib


def allowed_intervals(layout, N, S, causal, cu, rows_are_queries=True):
    """For every (rank i, local row a, shard j): the local index interval [lo, hi) of
    shard j's tokens that row a's token is paired with.  For queries, the keys at
    positions <= its own (causal) inside its sequence; for keys (rows_are_queries
    False), the queries at positions >= its own inside its sequence.  Local order
    increases with position in every layout, so the allowed set is an interval;
    that it is exactly this interval is checked too."""
    L = N * S
    pos = ly.rank_positions(layout, N, L)                     # [N, S]
    assert np.all(np.diff(pos, axis=1) > 0)
    seg = (oracle.segment_ids(cu, np.arange(L)) if cu is not None else np.zeros(L, dtype=np.int64))
    cu_arr = np.asarray(cu if cu is not None else [0, L], dtype=np.int64)
    t = pos.reshape(-1)                                       # rows in (i, a) order
    start, end = cu_arr[seg[t]], cu_arr[seg[t] + 1]
    lo = np.empty((N * S, N), dtype=np.int64)
    hi = np.empty_like(lo)
    for j in range(N):
        pj = pos[j]
        if rows_are_queries:
            lo[:, j] = np.searchsorted(pj, start, side="left")
            hi[:, j] = np.searchsorted(pj, t if causal else end - 1, side="right")
        else:
            lo[:, j] = np.searchsorted(pj, t if causal else start, side="left")
            hi[:, j] = np.searchsorted(pj, end - 1, side="right")
    hi = np.maximum(hi, lo)
    # brute force on a few rows: the interval holds exactly the allowed tokens
    rng = np.random.default_rng(N * 1000 + S)
    for r in rng.integers(0, N * S, 8):
        for j in range(N):
            pj = pos[j]
            if rows_are_queries:
                ok = (seg[pj] == seg[t[r]]) & ((pj <= t[r]) if causal else True)
            else:
                ok = (seg[pj] == seg[t[r]]) & ((pj >= t[r]) if causal else True)
            idx = np.nonzero(ok)[0]
            assert idx.size == hi[r, j] - lo[r, j]
            if idx.size:
                assert idx[0] == lo[r, j] and idx[-1] == hi[r, j] - 1
    return lo.reshape(N, S, N), hi.reshape(N, S, N)


def run_forward(probe, layout, N, S, causal, cu=None, mode=0, unit_rows=256, skip=0, B=2, H=3, bh_chunk=2):
    lo = np.empty((N, S, N), dtype=np.int32)
    hi = np.empty_like(lo)
    cnt = np.zeros_like(lo)
    n_units = -(-S // unit_rows)
    cov = np.empty(B * H * N * n_units, dtype=np.int32)
    dup = np.zeros(1, dtype=np.int32)
    cu32 = None if cu is None else np.ascontiguousarray(cu, dtype=np.int32)
    rc = probe.ra_test_forward_walk(LAYOUT_IDS[layout], N, S, int(causal),
                                    None if cu32 is None else cu32.ctypes.data,
                                    0 if cu is None else len(cu) - 1, mode, unit_rows, skip, B, H, bh_chunk,
                                    lo.ctypes.data, hi.ctypes.data, cnt.ctypes.data, cov.ctypes.data,
                                    dup.ctypes.data)
    assert rc == 0
    return lo, hi, cnt, cov, int(dup[0])


def check_forward(probe, layout, N, S, causal, cu=None, **kw):
    lo, hi, cnt, cov, dup = run_forward(probe, layout, N, S, causal, cu, **kw)
    elo, ehi = allowed_intervals(layout, N, S, causal, cu)
    assert np.all(cov == 1), "a unit handed out %s times" % sorted(set(cov.tolist()))
    assert dup != 1, "a (row, shard, key tile) visited twice"
    assert dup != 2, "the per-step tile counts (TileWalk::step_tiles) disagree with the walk"
    want = ehi - elo
    # every allowed key of every shard reached once, nothing else
    np.testing.assert_array_equal(cnt, want)
    seen = want > 0
    np.testing.assert_array_equal(lo[seen], elo[seen])
    np.testing.assert_array_equal(hi[seen], ehi[seen])
    L = N * S
    if cu is None:
        assert int(cnt.sum(dtype=np.int64)) == (L * (L + 1) // 2 if causal else L * L)
    else:
        lens = np.diff(np.asarray(cu, dtype=np.int64))
        assert int(cnt.sum(dtype=np.int64)) == int((lens * (lens + 1) // 2 if causal else lens * lens).sum())


SMALL = [("contiguous", 1, 300), ("contiguous", 3, 300), ("contiguous", 4, 256), ("striped", 1, 256),
         ("striped", 3, 200), ("striped", 4, 300), ("striped", 16, 512), ("zigzag", 1, 256),
         ("zigzag", 3, 300), ("zigzag", 4, 512), ("zigzag", 16, 512)]


@pytest.mark.parametrize("layout,N,S", SMALL)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_forward_walk_small(probe, layout, N, S, causal, mode):
    check_forward(probe, layout, N, S, causal, mode=mode)


# the sizes the bench and the parity tests run: 128K over 16 ranks, 2 x 32K over 8 (zigzag),
# the USP ring part (4 ranks of 64K), and 8K over 4
BIG = [("striped", 16, 8192), ("contiguous", 16, 8192), ("zigzag", 16, 8192), ("zigzag", 8, 4096),
       ("zigzag", 4, 65536), ("striped", 4, 2048), ("contiguous", 4, 2048)]


@pytest.mark.parametrize("layout,N,S", BIG)
def test_forward_walk_full_size(probe, layout, N, S):
    check_forward(probe, layout, N, S, True, B=1, H=8, bh_chunk=1)


@pytest.mark.parametrize("layout", ["striped", "contiguous"])
def test_stepwise_walk_full_size(probe, layout):
    """RA_FLAG_STEPWISE: N launches, step s visiting shard (i - s) mod N, partition the sweep."""
    check_forward(probe, layout, 16, 8192, True, mode=1, B=1, H=1, bh_chunk=1)


PACKED = [("striped", 4, 1024, 40, 1), ("striped", 16, 8192, 64, 1), ("striped", 3, 400, 9, 1),
          ("striped", 72, 128, 30, 1),     # 72 steps: past the 64-step table, every tile visited
          ("contiguous", 4, 1024, 40, 0), ("zigzag", 4, 1024, 40, 0), ("zigzag", 16, 8192, 64, 0),
          ("contiguous", 3, 400, 7, 0)]


@pytest.mark.parametrize("layout,N,S,n_seqs,skip", PACKED)
@pytest.mark.parametrize("causal", [True, False])
def test_forward_walk_packed_sequences(probe, layout, N, S, n_seqs, skip, causal):
    """Packed sequences: same-sequence pairs only, with the striped layout's per-Q-tile
    tile skipping (skip = 1) exactly as the kernel variant runs it."""
    cu = make_cu_seqlens(N * S, n_seqs, seed=N * S + n_seqs).numpy()
    check_forward(probe, layout, N, S, causal, cu, skip=skip)


@pytest.mark.parametrize("layout,N,S", [("striped", 4, 300), ("zigzag", 4, 512), ("contiguous", 3, 300),
                                        ("striped", 16, 8192)])
def test_dq_pass_walk(probe, layout, N, S):
    """The dQ pass walks the same keys with 128-row units."""
    check_forward(probe, layout, N, S, True, unit_rows=128, B=1, H=2, bh_chunk=1)


def run_key_walk(probe, layout, N, S, causal, cu, heads, B=2, Hkv=3, bh_chunk=2):
    lo = np.empty((heads, N, S, N), dtype=np.int32)
    hi = np.empty_like(lo)
    cnt = np.zeros_like(lo)
    cov = np.empty(B * Hkv * N * -(-S // 128), dtype=np.int32)
    dup = np.zeros(1, dtype=np.int32)
    cu32 = None if cu is None else np.ascontiguousarray(cu, dtype=np.int32)
    rc = probe.ra_test_key_walk(LAYOUT_IDS[layout], N, S, int(causal), None if cu32 is None else cu32.ctypes.data,
                                0 if cu is None else len(cu) - 1, heads, B, Hkv, bh_chunk, lo.ctypes.data,
                                hi.ctypes.data, cnt.ctypes.data, cov.ctypes.data, dup.ctypes.data)
    assert rc == 0
    return lo, hi, cnt, cov, int(dup[0])


@pytest.mark.parametrize("layout,N,S,causal,n_seqs,heads", [
    ("contiguous", 4, 300, True, None, 1), ("striped", 4, 300, True, None, 2), ("zigzag", 4, 512, True, None, 1),
    ("striped", 3, 200, False, None, 1), ("zigzag", 3, 300, True, 9, 2), ("striped", 4, 1024, True, 40, 1),
    ("striped", 16, 8192, True, None, 1), ("zigzag", 16, 8192, True, None, 1),
])
def test_dkv_pass_walk(probe, layout, N, S, causal, n_seqs, heads):
    """The dK / dV pass: every key meets every query that sees it, once per query head."""
    cu = None if n_seqs is None else make_cu_seqlens(N * S, n_seqs, seed=7 * S + n_seqs).numpy()
    lo, hi, cnt, cov, dup = run_key_walk(probe, layout, N, S, causal, cu, heads)
    elo, ehi = allowed_intervals(layout, N, S, causal, cu, rows_are_queries=False)
    assert np.all(cov == 1) and dup == 0
    for hd in range(heads):
        np.testing.assert_array_equal(cnt[hd], ehi - elo)
        seen = ehi > elo
        np.testing.assert_array_equal(lo[hd][seen], elo[seen])
        np.testing.assert_array_equal(hi[hd][seen], ehi[seen])


def test_a_planted_walk_error_is_caught(probe):
    """The comparison is sharp: the allowed intervals shifted by one key (an off-by-one
    in the causal prefix) or the strict striped mask read as inclusive both fail it."""
    lo, hi, cnt, cov, dup = run_forward(probe, "striped", 4, 300, True)
    elo, ehi = allowed_intervals("striped", 4, 300, True, None)
    assert np.array_equal(cnt, ehi - elo)
    assert not np.array_equal(cnt, np.minimum(ehi + 1, 300) - elo)
    pos = ly.rank_positions("striped", 4, 1200)
    inclusive = np.stack([np.searchsorted(pos[j], pos.reshape(-1) + 1, side="right") for j in range(4)], axis=1)
    assert not np.array_equal(cnt.reshape(-1, 4), inclusive)
