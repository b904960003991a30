"""The bounded-wait path on the GPU, without a fault: the test hook
RA_FLAG_INJECT_STALL makes one CTA's producer withhold a key tile, so the
waits that depend on it run out.  The kernel must record RA_ERR_TIMEOUT in the
status word and exit; the host reads it with ra_check_status, and the context
stays usable for the next call."""
import time

import numpy as np
import pytest
import torch

import oracle
from conftest import assert_attention_close
from synthetic_inputs import make_qkv

pytestmark = pytest.mark.gpu


def _shards(ra, x, N):
    B, L, H, d = x.shape
    y = torch.empty((N, B, L // N, H, d), dtype=torch.bfloat16, device="cuda")
    ra.ra_shard_permute(x.cuda(), y, ra.RA_SEQ_TO_SHARDS, "contiguous", B, L, H, d, N)
    return y


# d = 128 runs two MMA issuers (S and PV), d = 64 one: both wind down on a timeout
@pytest.mark.parametrize("d", [128, 64])
def test_withheld_tile_times_out_and_context_survives(ralib, gpu, d):
    B, L, H, N = 1, 1024, 2, 2
    q, k, v, _ = make_qkv(B, L, H, d, seed=71)
    qs, ks, vs = (_shards(ralib, x, N) for x in (q, k, v))
    S = L // N
    o = torch.zeros((N, B, S, H, d), dtype=torch.float32, device="cuda")
    lse = torch.zeros((N, B, H, S), dtype=torch.float32, device="cuda")
    ws = ralib.new_workspace(256)
    t0 = time.time()
    ralib.ra_ring_attn_fwd(qs, ks, vs, o, lse, B, L, H, d, N, "contiguous", False,
                           flags=ralib.RA_FLAG_INJECT_STALL, workspace=ws)
    with pytest.raises(ralib.RAError) as exc:
        ralib.ra_check_status(ws)
    assert exc.value.status == ralib.RA_ERR_TIMEOUT
    assert time.time() - t0 < 60
    # the status word was cleared by the check; a normal call still works
    ralib.ra_ring_attn_fwd(qs, ks, vs, o, lse, B, L, H, d, N, "contiguous", False, workspace=ws)
    ralib.ra_check_status(ws)
    o_seq = torch.empty((B, L, H, d), dtype=torch.float32, device="cuda")
    ralib.ra_shard_permute(o, o_seq, ralib.RA_SHARDS_TO_SEQ, "contiguous", B, L, H, d, N)
    lse_seq = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    ralib.ra_lse_to_seq(lse, lse_seq, "contiguous", B, L, H, N)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=False)
    assert_attention_close(o_seq.cpu().numpy(), o_ref, lse_seq.cpu().numpy(), lse_ref)
