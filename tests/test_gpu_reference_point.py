"""The online softmax's reference point under scores far from zero.

"From Ring Attention to DeepSpeed Ulysses to USP" (jsqmd.com/news/734632), §3.2: the
running (m, l, O) state.  The kernel keeps m as a reference point that moves only when
the row's running denominator would leave [2^-32, 2^32]; these inputs force that move
(P overflowing against the first reference, or every P of a row underflowing to zero)
on the fused sweep and on the per-step block + merge path, and the result must still be
the exact attention of the fp64 oracle within the usual bar.
"""
import numpy as np
import pytest

import oracle
from conftest import assert_attention_close
from synthetic_inputs import make_extreme_qkv
from test_gpu_attention import run_ring

pytestmark = pytest.mark.gpu

CASES = [
    # mode, B, L, H, d, N, layout, causal
    ("large", 1, 1024, 2, 128, 4, "striped", True),
    ("large", 1, 1200, 2, 128, 4, "contiguous", False),
    ("negative", 1, 1024, 2, 128, 4, "striped", True),
    ("negative", 1, 1024, 2, 128, 4, "zigzag", False),
    ("mixed", 2, 1200, 2, 128, 4, "striped", True),
    ("mixed", 1, 1024, 2, 64, 4, "contiguous", True),
]


@pytest.mark.parametrize("mode,B,L,H,d,N,layout,causal", CASES)
@pytest.mark.parametrize("flags", [0, 1], ids=["fused", "stepwise"])
def test_reference_point_moves(ralib, gpu, mode, B, L, H, d, N, layout, causal, flags):
    q, k, v = make_extreme_qkv(B, L, H, d, seed=L + d + N, mode=mode)
    o_ref, lse_ref = oracle.full_attention(q, k, v, causal=causal)
    # the inputs do reach the regime: rows tens of nats from zero
    if mode == "large":
        assert lse_ref.max() > 25.0
    elif mode == "negative":
        assert lse_ref.max() < -25.0
    else:
        assert lse_ref.max() > 25.0 and lse_ref.min() < -20.0
    o, lse = run_ring(ralib, q, k, v, N, layout, causal, flags=flags)
    assert_attention_close(o, o_ref, lse, lse_ref, "%s %s N=%d causal=%s" % (mode, layout, N, causal))
