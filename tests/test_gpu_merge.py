"""ra_lse_merge (strided rows) and ra_lse_merge_bshd on the GPU against the oracle's LSE
merge ("From Ring Attention to DeepSpeed Ulysses to USP", §6.3), including empty (-inf)
partials."""
import numpy as np
import pytest
import torch

import oracle.blockwise as bw
from synthetic_inputs import randn_f32, random_ints

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,S,H,d", [(1, 100, 3, 64), (2, 257, 2, 128), (1, 31, 1, 4), (1, 64, 4, 256)])
def test_merge_matches_oracle(ralib, gpu, B, S, H, d):
    o_a = randn_f32((B, S, H, d), 1)
    o_b = randn_f32((B, S, H, d), 2)
    lse_a = randn_f32((B, H, S), 3, scale=5.0)
    lse_b = randn_f32((B, H, S), 4, scale=5.0)
    # empty partials: some rows empty on one side, some on both
    ea = random_ints(max(1, S // 5), 0, S, 5)
    eb = random_ints(max(1, S // 5), 0, S, 6)
    lse_a[:, :, ea] = -float("inf")
    lse_b[:, :, eb] = -float("inf")
    for b in range(B):
        for h in range(H):
            o_a[b, lse_a[b, h] == -float("inf"), h] = 0
            o_b[b, lse_b[b, h] == -float("inf"), h] = 0
    o_acc, l_acc = o_a.to(gpu), lse_a.to(gpu)
    ralib.ra_lse_merge_bshd(o_acc, l_acc, o_b.to(gpu), lse_b.to(gpu), B, S, H, d)
    # oracle works on rows [B, H, S, d]
    oa = o_a.double().numpy().transpose(0, 2, 1, 3)
    ob = o_b.double().numpy().transpose(0, 2, 1, 3)
    o_ref, lse_ref = bw.lse_merge(oa, lse_a.double().numpy(), ob, lse_b.double().numpy())
    got = o_acc.cpu().double().numpy().transpose(0, 2, 1, 3)
    np.testing.assert_allclose(got, o_ref, rtol=2e-6, atol=2e-6)
    lg = l_acc.cpu().double().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    fin = ~np.isneginf(lse_ref)
    np.testing.assert_allclose(lg[fin], lse_ref[fin], rtol=1e-6, atol=2e-6)
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("rows,d,Ha,Hb", [(300, 128, 4, 1), (33, 64, 3, 2), (1000, 4, 1, 5)])
def test_strided_merge_into_one_head_of_a_wider_buffer(ralib, gpu, rows, d, Ha, Hb):
    """The accumulator is head 1 of an [rows, Ha, d] buffer (row stride Ha*d) and b is head 0
    of an [rows, Hb, d] one: only those rows change, and they match the oracle."""
    acc = randn_f32((rows, Ha, d), 11)
    part = randn_f32((rows, Hb, d), 12)
    la = randn_f32((rows,), 13, scale=4.0)
    lb = randn_f32((rows,), 14, scale=4.0)
    la[random_ints(max(1, rows // 7), 0, rows, 15)] = -float("inf")
    lb[random_ints(max(1, rows // 7), 0, rows, 16)] = -float("inf")
    ha = 1 if Ha > 1 else 0
    acc[la == -float("inf"), ha] = 0
    part[lb == -float("inf"), 0] = 0
    acc_g, part_g = acc.to(gpu), part.to(gpu)
    la_g, lb_g = la.to(gpu), lb.to(gpu)
    ralib.ra_lse_merge(acc_g[:, ha], la_g, part_g[:, 0], lb_g)
    o_ref, lse_ref = bw.lse_merge(acc[:, ha].double().numpy(), la.double().numpy(),
                                  part[:, 0].double().numpy(), lb.double().numpy())
    got = acc_g.cpu()
    np.testing.assert_allclose(got[:, ha].double().numpy(), o_ref, rtol=2e-6, atol=2e-6)
    for h in range(Ha):                       # the other heads are untouched
        if h != ha:
            assert torch.equal(got[:, h], acc[:, h])
    assert torch.equal(part_g.cpu(), part)
    lg = la_g.cpu().double().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    fin = ~np.isneginf(lse_ref)
    np.testing.assert_allclose(lg[fin], lse_ref[fin], rtol=1e-6, atol=2e-6)
