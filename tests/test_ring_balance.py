"""The bench's per-step balance table ("From Ring Attention to DeepSpeed Ulysses to USP",
§3.4 load imbalance, §4 striped, §6.1 zigzag) against brute-force counting over the
oracle's token positions, and the config-4 critical paths of the three layouts."""
import numpy as np
import pytest

import bench
import oracle.layouts as ly


def _brute_counts(layout, N, L, causal):
    pos = ly.rank_positions(layout, N, L)              # [N, S] global token of (rank, local)
    c = np.zeros((N, N), dtype=np.int64)
    for i in range(N):
        for s in range(N):
            j = (i - s) % N
            if causal:
                c[i, s] = int((pos[j][None, :] <= pos[i][:, None]).sum())
            else:
                c[i, s] = pos[i].size * pos[j].size
    return c


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N,L", [(1, 8), (2, 8), (4, 32), (5, 60), (8, 64)])
def test_counts_match_positions(layout, causal, N, L):
    np.testing.assert_array_equal(bench.ring_pair_counts(layout, N, L // N, causal),
                                  _brute_counts(layout, N, L, causal))


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
def test_every_causal_pair_once(layout):
    """The steps together cover the causal triangle exactly: L(L+1)/2 pairs."""
    N, L = 16, 131072
    t = bench.balance_table(layout, N, L // N, True)
    assert t["pairs_total"] == L * (L + 1) // 2


def test_config4_critical_paths():
    """128K tokens over 16 ranks: contiguous is bound by the last rank (S^2/2 + 15 S^2 pairs),
    striped and zigzag stay within a hair of the ideal total / N."""
    N, L = 16, 131072
    S = L // N
    con = bench.balance_table("contiguous", N, S, True)
    st = bench.balance_table("striped", N, S, True)
    zz = bench.balance_table("zigzag", N, S, True)
    assert con["pairs_critical_path"] == S * (S + 1) // 2 + 15 * S * S == 1040191488
    assert st["pairs_critical_path"] == N * S * (S + 1) // 2 == 536936448
    assert zz["pairs_critical_path"] == S * S // 2 + S // 2 + 15 * S * S // 2
    assert 1.93 < con["pairs_ratio"] < 1.95
    assert st["pairs_ratio"] < 1.0002 and zz["pairs_ratio"] < 1.0002


def test_kernel_hash_ignores_comments_only():
    """The DRAM-traffic figure is tied to the kernel's code: comments and
    whitespace do not move the hash, code and string literals do."""
    code = bench._code_only
    a = "int a = 1; // one\n/* block\n comment */ const char *s = \"x // y\";\n"
    b = "int a=1;\nconst char *s = \"x // y\"; // another comment\n"
    assert code(a) == code(b)
    assert code(a) != code(a.replace("a = 1", "a = 2"))
    assert code(a) != code(a.replace("x // y", "x / y"))
