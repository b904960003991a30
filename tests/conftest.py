import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Rows of a golden text fixture: comment lines (#) and blank lines dropped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def ora():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def ralib():
    """The built C-ABI library (built here if stale)."""
    from sequence_blockwise_softmax_gb300 import build as b
    b.build()
    import sequence_blockwise_softmax_gb300 as ra
    ra.lib()
    return ra


@pytest.fixture(scope="session")
def gpu(ralib):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test on a machine without CUDA")
    return torch.device("cuda:0")


# Parity bar for bf16 inputs with fp32 accumulation, against the fp64 oracle.
O_MAX_ABS = 1e-2
O_REL_L2 = 5e-3
LSE_MAX_ABS = 1e-3


def assert_attention_close(o, o_ref, lse, lse_ref, what=""):
    """O within max-abs 1e-2 and rel-L2 5e-3, LSE within abs 1e-3 (same -inf pattern)."""
    import numpy as np
    o = np.asarray(o, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    lse_ref = np.asarray(lse_ref, dtype=np.float64)
    assert o.shape == o_ref.shape and lse.shape == lse_ref.shape, what
    assert np.all(np.isfinite(o)), what + ": non-finite O"
    err = np.abs(o - o_ref).max() if o.size else 0.0
    denom = np.linalg.norm(o_ref)
    rel = np.linalg.norm(o - o_ref) / denom if denom > 0 else np.linalg.norm(o - o_ref)
    ninf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), ninf), what + ": -inf pattern of LSE differs"
    lerr = np.abs(lse[~ninf] - lse_ref[~ninf]).max() if (~ninf).any() else 0.0
    assert err <= O_MAX_ABS, "%s: O max-abs %g" % (what, err)
    assert rel <= O_REL_L2, "%s: O rel-L2 %g" % (what, rel)
    assert lerr <= LSE_MAX_ABS, "%s: LSE max-abs %g" % (what, lerr)
    return err, rel, lerr
