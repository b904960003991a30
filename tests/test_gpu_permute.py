"""ra_shard_permute / ra_lse_to_seq on the GPU, bit-exact against the oracle's index formulas."""
import numpy as np
import pytest
import torch

import oracle.layouts as ly
from synthetic_inputs import WORKLOADS, randn_bf16, randn_f32

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("layout", ly.LAYOUTS)
@pytest.mark.parametrize("B,L,H,d,R,U", [
    (1, 16, 2, 64, 4, 1),       # the pages' 16-token example
    (2, 48, 4, 64, 3, 1),       # odd ring degree
    (1, 96, 4, 128, 4, 2),      # USP numbering
    (2, 240, 6, 64, 2, 3),
    (1, 64, 8, 8, 8, 1),        # 16-byte tokens
])
def test_seq_to_shards_and_back(ralib, gpu, layout, B, L, H, d, R, U):
    x = randn_bf16((B, L, H, d), 5)
    xg = x.to(gpu)
    P = U * R
    y = torch.empty((P, B, L // P, H, d), dtype=torch.bfloat16, device=gpu)
    ralib.ra_shard_permute(xg, y, ralib.RA_SEQ_TO_SHARDS, layout, B, L, H, d, R, U)
    want = ly.usp_seq_to_shards(_u16(x), layout, R, U)
    np.testing.assert_array_equal(_u16(y), want)
    back = torch.empty_like(xg)
    ralib.ra_shard_permute(y, back, ralib.RA_SHARDS_TO_SEQ, layout, B, L, H, d, R, U)
    np.testing.assert_array_equal(_u16(back), _u16(x))


@pytest.mark.parametrize("B,L,H,d,R,U", [(1, 96, 4, 128, 4, 2), (2, 48, 6, 64, 2, 3), (1, 32, 4, 64, 1, 4)])
def test_ulysses_round_trip(ralib, gpu, B, L, H, d, R, U):
    P = U * R
    x = randn_bf16((P, B, L // P, H, d), 9)
    xg = x.to(gpu)
    y = torch.empty((R, U, B, L // R, H // U, d), dtype=torch.bfloat16, device=gpu)
    ralib.ra_shard_permute(xg, y, ralib.RA_ULYSSES_SEQ_TO_HEAD, "contiguous", B, L, H, d, R, U)
    np.testing.assert_array_equal(_u16(y), ly.ulysses_seq_to_head(_u16(x), R, U))
    back = torch.empty_like(xg)
    ralib.ra_shard_permute(y, back, ralib.RA_ULYSSES_HEAD_TO_SEQ, "contiguous", B, L, H, d, R, U)
    np.testing.assert_array_equal(_u16(back), _u16(x))


def test_fp32_elements(ralib, gpu):
    B, L, H, d, R = 1, 64, 2, 4, 4
    x = randn_f32((B, L, H, d), 3)
    y = torch.empty((R, B, L // R, H, d), dtype=torch.float32, device=gpu)
    ralib.ra_shard_permute(x.to(gpu), y, ralib.RA_SEQ_TO_SHARDS, "zigzag", B, L, H, d, R)
    np.testing.assert_array_equal(y.cpu().numpy(), ly.seq_to_shards(x.numpy(), "zigzag", R))


@pytest.mark.parametrize("layout", ly.LAYOUTS)
@pytest.mark.parametrize("B,L,H,R,U", [(2, 24, 4, 3, 2), (1, 64, 2, 4, 1), (1, 32, 4, 2, 2)])
def test_lse_to_seq(ralib, gpu, layout, B, L, H, R, U):
    src = randn_f32((R, U * B, H // U, L // R), 4)
    dst = torch.empty((B, H, L), dtype=torch.float32, device=gpu)
    ralib.ra_lse_to_seq(src.to(gpu), dst, layout, B, L, H, R, U)
    np.testing.assert_array_equal(dst.cpu().numpy(), ly.lse_to_seq(src.numpy(), layout, R, U, B))


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_permutes_bit_exact(ralib, gpu, name):
    """Full-size shard permutes of every standard workload (one tensor each)."""
    w = WORKLOADS[name]
    B, L, H, d = w["B"], w["L"], w["H"], w["d"]
    U = w.get("U", 1)
    R = w["N"]
    layout = w["layouts"][0]
    x = randn_bf16((B, L, H, d), w["seed"])
    xg = x.to(gpu)
    P = U * R
    y = torch.empty((P, B, L // P, H, d), dtype=torch.bfloat16, device=gpu)
    ralib.ra_shard_permute(xg, y, ralib.RA_SEQ_TO_SHARDS, layout, B, L, H, d, R, U)
    want = ly.usp_seq_to_shards(_u16(x), layout, R, U)
    np.testing.assert_array_equal(_u16(y), want)
    if U > 1:
        z = torch.empty((R, U, B, L // R, H // U, d), dtype=torch.bfloat16, device=gpu)
        ralib.ra_shard_permute(y, z, ralib.RA_ULYSSES_SEQ_TO_HEAD, layout, B, L, H, d, R, U)
        np.testing.assert_array_equal(_u16(z), ly.ulysses_seq_to_head(want, R, U))
    back = torch.empty_like(xg)
    ralib.ra_shard_permute(y, back, ralib.RA_SHARDS_TO_SEQ, layout, B, L, H, d, R, U)
    assert torch.equal(back, xg)
