"""The token-order tile addressing of the attention kernels, on the host: every
row of every rank's shard is reached at its token's offset in [B, L, cols] (the
layouts of "From Ring Attention to DeepSpeed Ulysses to USP",
jsqmd.com/news/734632, §4 and §6.1, as the oracle writes them), and the rows
past a shard's end in its last 128-row tile fall outside the view, which is
what makes TMA read zeros there and skip the stores."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle.layouts as ly
from conftest import ROOT

CSRC = os.path.join(ROOT, "sequence_blockwise_softmax_gb300", "csrc")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("addr") / "addr_probe.so")
    subprocess.run([nvcc, "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
                    "-I", CSRC, os.path.join(ROOT, "tests", "addr_probe.cu"), "-o", out],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    lib.ra_test_token_offsets.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    return lib


LAYOUT_IDS = {"contiguous": 0, "striped": 1, "zigzag": 2}


@pytest.mark.parametrize("layout,N,S", [
    ("contiguous", 4, 300), ("contiguous", 1, 256), ("striped", 4, 300), ("striped", 5, 200),
    ("striped", 16, 512), ("zigzag", 4, 256), ("zigzag", 3, 512), ("zigzag", 8, 1024),
])
def test_token_order_addresses(probe, layout, N, S):
    B, cols = 2, 256
    S_pad = (S + 127) // 128 * 128
    off = np.zeros(N * B * S_pad, dtype=np.int64)
    inside = np.zeros(N * B * S_pad, dtype=np.uint8)
    probe.ra_test_token_offsets(LAYOUT_IDS[layout], N, S, B, cols, off.ctypes.data, inside.ctypes.data)
    off = off.reshape(N, B, S_pad)
    inside = inside.reshape(N, B, S_pad).astype(bool)
    L = N * S
    for r in range(N):
        pos = ly.global_position(layout, r, np.arange(S), N, S)
        for b in range(B):
            np.testing.assert_array_equal(off[r, b, :S], (b * L + pos) * cols)
            assert inside[r, b, :S].all()
            assert not inside[r, b, S:].any()
    # every token of the sequence is some rank's row, exactly once
    hits = np.sort(off[:, :, :S].reshape(-1))
    np.testing.assert_array_equal(hits, np.arange(B * L) * cols)
