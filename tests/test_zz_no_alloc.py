"""The allocation-free stepwise sweep against the workspace entry point.

ra_ring_attn_fwd_stepwise_noalloc serves callers that cannot allocate device
memory or pass a workspace (code inside another framework's memory pool or
allocator callback, plugins given only their buffers, paths where cudaMalloc
would synchronise the device).  Its scratch is a fixed array owned by the
library.  This file is collected last so that a run stopping at its first
failure has already run every other test; it also passes on its own in a
fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from conftest import assert_attention_close
from synthetic_inputs import make_qkv

pytestmark = pytest.mark.gpu


def _shards(ra, x, layout, N):
    B, L, H, d = x.shape
    y = torch.empty((N, B, L // N, H, d), dtype=torch.bfloat16, device="cuda")
    ra.ra_shard_permute(x.cuda(), y, ra.RA_SEQ_TO_SHARDS, layout, B, L, H, d, N)
    return y


def _call_noalloc(ra, q, k, v, o, lse, B, L, H, d, N, layout, causal):
    """Through the C ABI directly (ctypes), as a C caller would."""
    lib = ra.lib()
    st = lib.ra_ring_attn_fwd_stepwise_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, L, H, d, N,
        ra.LAYOUTS[layout], int(causal), ctypes.c_float(0.0),
        torch.cuda.current_stream().cuda_stream)
    assert st == ra.RA_OK, lib.ra_last_error().decode()


CASES = [  # two calls in a row, different shapes and layouts, sharing the scratch array
    dict(B=1, L=2048, H=4, d=128, N=4, layout="striped", causal=True, seed=301),
    dict(B=2, L=1200, H=2, d=64, N=3, layout="zigzag", causal=True, seed=302),
]


def test_noalloc_matches_workspace_entry_point_on_two_calls(ralib, gpu):
    for c in CASES:
        B, L, H, d, N, layout, causal = (c[k] for k in ("B", "L", "H", "d", "N", "layout", "causal"))
        q, k, v, _ = make_qkv(B, L, H, d, c["seed"])
        qs, ks, vs = (_shards(ralib, x, layout, N) for x in (q, k, v))
        S = L // N
        o_ref = torch.empty((N, B, S, H, d), dtype=torch.float32, device="cuda")
        lse_ref = torch.empty((N, B, H, S), dtype=torch.float32, device="cuda")
        ws = ralib.new_workspace(ralib.ra_ring_attn_workspace_bytes(B, L, H, d, N, ralib.RA_FLAG_STEPWISE))
        ralib.ra_ring_attn_fwd(qs, ks, vs, o_ref, lse_ref, B, L, H, d, N, layout, causal,
                               flags=ralib.RA_FLAG_STEPWISE, workspace=ws)
        ralib.ra_check_status(ws)
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        _call_noalloc(ralib, qs, ks, vs, o, lse, B, L, H, d, N, layout, causal)
        torch.cuda.synchronize()
        assert_attention_close(o.cpu().numpy(), o_ref.cpu().numpy(), lse.cpu().numpy(),
                               lse_ref.cpu().numpy(), "noalloc %s" % layout)


def test_noalloc_rejects_problems_beyond_its_scratch(ralib, gpu):
    # B*L*H*(d+1)*4 bytes of scratch: 1*65536*16*129*4 > 64 MiB
    lib = ralib.lib()
    st = lib.ra_ring_attn_fwd_stepwise_noalloc(16, 16, 16, 16, 16, 1, 65536, 16, 128, 4, 0, 1,
                                               ctypes.c_float(0.0), None)
    assert st == ralib.RA_ERR_UNSUPPORTED
    assert "64 MiB" in lib.ra_last_error().decode()
