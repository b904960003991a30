"""The allocation-free stepwise sweep against the workspace entry point and the oracle.

ra_ring_attn_fwd_stepwise_noalloc serves callers that cannot allocate device
memory or pass a workspace (code inside another framework's memory pool or
allocator callback, plugins given only their buffers, paths where cudaMalloc
would synchronise the device).  Its scratch is a fixed array owned by the
library.  It runs the same kernels in the same order as the workspace
stepwise sweep, so the two must agree bit for bit; one case is also compared
with the fp64 oracle, a problem at exactly the size limit runs, and a stalled
call is reported by ra_noalloc_check_status.  This file is collected last so
that a run stopping at its first failure has already run every other test; it
also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from conftest import assert_attention_close
from synthetic_inputs import make_qkv

pytestmark = pytest.mark.gpu


def _shards(ra, x, layout, N):
    B, L, H, d = x.shape
    y = torch.empty((N, B, L // N, H, d), dtype=torch.bfloat16, device="cuda")
    ra.ra_shard_permute(x.cuda(), y, ra.RA_SEQ_TO_SHARDS, layout, B, L, H, d, N)
    return y


def _call_noalloc(ra, q, k, v, o, lse, B, L, H, d, N, layout, causal, flags=0):
    """Through the C ABI directly (ctypes), as a C caller would."""
    lib = ra.lib()
    st = lib.ra_ring_attn_fwd_stepwise_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, L, H, d, N,
        ra.LAYOUTS[layout], int(causal), ctypes.c_float(0.0), flags,
        torch.cuda.current_stream().cuda_stream)
    assert st == ra.RA_OK, lib.ra_last_error().decode()


def _check_status(ra):
    return ra.lib().ra_noalloc_check_status(torch.cuda.current_stream().cuda_stream)


def _workspace_stepwise(ra, qs, ks, vs, B, L, H, d, N, layout, causal):
    S = L // N
    o = torch.empty((N, B, S, H, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((N, B, H, S), dtype=torch.float32, device="cuda")
    ws = ra.new_workspace(ra.ra_ring_attn_workspace_bytes(B, L, H, d, N, ra.RA_FLAG_STEPWISE))
    ra.ra_ring_attn_fwd(qs, ks, vs, o, lse, B, L, H, d, N, layout, causal, flags=ra.RA_FLAG_STEPWISE,
                        workspace=ws)
    ra.ra_check_status(ws)
    return o, lse


CASES = [  # calls in a row, different shapes and layouts, sharing the scratch array
    dict(B=1, L=2048, H=4, d=128, N=4, layout="striped", causal=True, seed=301),
    dict(B=2, L=1200, H=2, d=64, N=3, layout="zigzag", causal=True, seed=302),
    dict(B=1, L=1000, H=3, d=128, N=5, layout="contiguous", causal=False, seed=303),
]


def test_noalloc_matches_workspace_entry_point_bit_for_bit(ralib, gpu):
    assert _check_status(ralib) == ralib.RA_OK
    for c in CASES:
        B, L, H, d, N, layout, causal = (c[k] for k in ("B", "L", "H", "d", "N", "layout", "causal"))
        q, k, v, _ = make_qkv(B, L, H, d, c["seed"])
        qs, ks, vs = (_shards(ralib, x, layout, N) for x in (q, k, v))
        o_ref, lse_ref = _workspace_stepwise(ralib, qs, ks, vs, B, L, H, d, N, layout, causal)
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        _call_noalloc(ralib, qs, ks, vs, o, lse, B, L, H, d, N, layout, causal)
        assert _check_status(ralib) == ralib.RA_OK
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), "noalloc %s" % layout


def test_noalloc_matches_the_oracle(ralib, gpu):
    B, L, H, d, N, layout = 1, 1536, 2, 128, 3, "striped"
    q, k, v, _ = make_qkv(B, L, H, d, 304)
    qs, ks, vs = (_shards(ralib, x, layout, N) for x in (q, k, v))
    S = L // N
    o = torch.empty((N, B, S, H, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((N, B, H, S), dtype=torch.float32, device="cuda")
    _call_noalloc(ralib, qs, ks, vs, o, lse, B, L, H, d, N, layout, True)
    assert _check_status(ralib) == ralib.RA_OK
    o_seq = torch.empty((B, L, H, d), dtype=torch.float32, device="cuda")
    ralib.ra_shard_permute(o, o_seq, ralib.RA_SHARDS_TO_SEQ, layout, B, L, H, d, N)
    lse_seq = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    ralib.ra_lse_to_seq(lse, lse_seq, layout, B, L, H, N)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=True)
    assert_attention_close(o_seq.cpu().numpy(), o_ref, lse_seq.cpu().numpy(), lse_ref, "noalloc vs oracle")


def test_noalloc_runs_a_problem_at_exactly_the_limit(ralib, gpu):
    """256 + round256(B*L*H*d*4) + round256(B*L*H*4) = 64 MiB exactly for B=1, L=26011, H=5,
    d=128: accepted, and equal to the workspace path; one token more is rejected."""
    B, L, H, d, N, layout = 1, 26011, 5, 128, 1, "contiguous"
    q, k, v, _ = make_qkv(B, L, H, d, 305)
    qs, ks, vs = (_shards(ralib, x, layout, N) for x in (q, k, v))
    o_ref, lse_ref = _workspace_stepwise(ralib, qs, ks, vs, B, L, H, d, N, layout, True)
    o, lse = torch.empty_like(o_ref), torch.empty_like(lse_ref)
    _call_noalloc(ralib, qs, ks, vs, o, lse, B, L, H, d, N, layout, True)
    assert _check_status(ralib) == ralib.RA_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    lib = ralib.lib()
    st = lib.ra_ring_attn_fwd_stepwise_noalloc(16, 16, 16, 16, 16, B, L + 1, H, d, N, 0, 1, ctypes.c_float(0.0), 0,
                                               None)
    assert st == ralib.RA_ERR_UNSUPPORTED and "64 MiB" in lib.ra_last_error().decode()


def test_noalloc_reports_a_timeout_and_recovers(ralib, gpu):
    """With the stall hook the first step's first CTA withholds a key tile: its bounded waits
    run out (about two seconds), the status word records it, ra_noalloc_check_status reports
    RA_ERR_TIMEOUT once and clears it, and the next call is correct again."""
    B, L, H, d, N, layout = 1, 1024, 2, 128, 4, "striped"
    q, k, v, _ = make_qkv(B, L, H, d, 306)
    qs, ks, vs = (_shards(ralib, x, layout, N) for x in (q, k, v))
    o_ref, lse_ref = _workspace_stepwise(ralib, qs, ks, vs, B, L, H, d, N, layout, True)
    o, lse = torch.empty_like(o_ref), torch.empty_like(lse_ref)
    _call_noalloc(ralib, qs, ks, vs, o, lse, B, L, H, d, N, layout, True, flags=ralib.RA_FLAG_INJECT_STALL)
    assert _check_status(ralib) == ralib.RA_ERR_TIMEOUT
    assert "bounded wait" in ralib.lib().ra_last_error().decode()
    assert _check_status(ralib) == ralib.RA_OK            # cleared by the read
    _call_noalloc(ralib, qs, ks, vs, o, lse, B, L, H, d, N, layout, True)
    assert _check_status(ralib) == ralib.RA_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_noalloc_rejects_problems_beyond_its_scratch(ralib, gpu):
    # 256 + round256(B*L*H*d*4) + round256(B*L*H*4) bytes: 1*65536*16 rows of 129 floats > 64 MiB
    lib = ralib.lib()
    st = lib.ra_ring_attn_fwd_stepwise_noalloc(16, 16, 16, 16, 16, 1, 65536, 16, 128, 4, 0, 1,
                                               ctypes.c_float(0.0), 0, None)
    assert st == ralib.RA_ERR_UNSUPPORTED
    assert "64 MiB" in lib.ra_last_error().decode()
