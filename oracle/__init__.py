"""CPU oracle for the ring-attention path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (``bench.py``'s ``cpu_baseline`` and ``--impl reference``) may import it.
The library (``sequence_blockwise_softmax_gb300``) never imports, links or
runs anything here, and nothing here imports the library: the two share no
code, only the seeded inputs of ``synthetic_inputs``.

Parts and what pins each (all pins live in ``tests/test_oracle_*.py``):
  * ``attention`` (``attention_fp64.c``): full-softmax attention in fp64 --
    pinned by hand-computed 2x2 cases (``tests/golden/hand_2x2.txt``), by a
    direct softmax without max-subtraction in arbitrary precision on tiny
    inputs, and by closed forms (Q = 0, constant V, the first causal row).
  * ``layouts``: token assignments and the Ulysses transpose -- pinned by the
    pages' worked examples (``tests/golden/*_assignment.txt``) and by exact
    round trips.
  * ``blockwise``: the online (m, l, O) recursion and the LSE merge -- pinned
    against one-shot attention under random block splits and orders, and by
    lse = m + ln l.
  * ``backward``: fp64 gradients of attention -- pinned by central finite
    differences of a separately written forward, and by the identities
    sum_k dK = 0 and sum_k dV = sum_q dO (``tests/test_oracle_backward_pins.py``).
"""
import ctypes
import os
import subprocess

import numpy as np

from . import backward, blockwise, layouts  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_fp64.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_fp64.so")
_lib = None


def build(force=False):
    """Compile the C part of the oracle with gcc (OpenMP) if it is stale."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c99", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_attention_fp64.argtypes = [
            P, I64, P, I64, P, P, I64, P, I64, P, P,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, P, P, ctypes.c_int]
        lib.oracle_attention_fp64.restype = ctypes.c_int
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads():
    return _load().oracle_num_threads()


def _bf16_bits(x):
    """uint16 numpy view of a bf16 torch tensor (or pass a uint16 array through)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def segment_ids(cu_seqlens, positions):
    """Sequence id of each global position for packed sequences with boundaries cu_seqlens."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return np.searchsorted(cu, np.asarray(positions, dtype=np.int64), side="right") - 1


def attention(q, k, v, q_pos=None, k_pos=None, causal=False, scale=None, nthreads=0,
              q_seg=None, k_seg=None):
    """fp64 attention of the query rows ``q`` [nq, H, d] against keys ``k``, ``v`` [nk, Hkv, d].

    With Hkv < H (grouped-query attention) query head h reads key/value head
    h // (H // Hkv).  With ``q_seg`` / ``k_seg`` (sequence ids of packed
    sequences) a key is allowed only within the query's own sequence.

    Inputs are bf16 (torch bf16 tensors or uint16 bit arrays).  ``q_pos`` /
    ``k_pos`` are the rows' global token positions (default 0..n-1); with
    ``causal`` a key is allowed when k_pos <= q_pos.  ``scale`` defaults to
    1/sqrt(d).  Returns (O [nq, H, d] float64, LSE [nq, H] float64).
    """
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    nq, H, d = qb.shape
    nk, Hkv = kb.shape[0], kb.shape[1]
    assert kb.shape == (nk, Hkv, d) and vb.shape == (nk, Hkv, d) and H % Hkv == 0
    q_pos = np.arange(nq, dtype=np.int64) if q_pos is None else np.ascontiguousarray(q_pos, dtype=np.int64)
    k_pos = np.arange(nk, dtype=np.int64) if k_pos is None else np.ascontiguousarray(k_pos, dtype=np.int64)
    assert q_pos.shape == (nq,) and k_pos.shape == (nk,)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if (q_seg is None) != (k_seg is None):
        raise ValueError("give both q_seg and k_seg, or neither")
    if q_seg is not None:
        q_seg = np.ascontiguousarray(q_seg, dtype=np.int64)
        k_seg = np.ascontiguousarray(k_seg, dtype=np.int64)
        assert q_seg.shape == (nq,) and k_seg.shape == (nk,)
    o = np.empty((nq, H, d), dtype=np.float64)
    lse = np.empty((nq, H), dtype=np.float64)
    rc = _load().oracle_attention_fp64(
        qb.ctypes.data, H * d, q_pos.ctypes.data, nq,
        kb.ctypes.data, vb.ctypes.data, Hkv * d, k_pos.ctypes.data, nk,
        None if q_seg is None else q_seg.ctypes.data, None if k_seg is None else k_seg.ctypes.data,
        H, Hkv, d, float(scale), int(bool(causal)), o.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc == -2:
        raise ValueError("the key/value head count must divide the query head count")
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return o, lse


def full_attention(q, k, v, causal, scale=None, rows=None, nthreads=0, cu_seqlens=None):
    """Attention over a whole sequence, [B, L, H, d] inputs.

    ``cu_seqlens``: optional boundaries of packed sequences (0 = c_0 <= ... <= c_n = L);
    a query then attends only within its own sequence.

    ``rows``: optional int array of query positions to evaluate (all if None).
    Returns (O [B, nrows, H, d], LSE [B, H, nrows]) in float64.
    """
    B, L = q.shape[0], q.shape[1]
    idx = np.arange(L, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    seg_all = None if cu_seqlens is None else segment_ids(cu_seqlens, np.arange(L))
    outs, lses = [], []
    for b in range(B):
        o, lse = attention(qb[b][idx], kb[b], vb[b], q_pos=idx, k_pos=None,
                           causal=causal, scale=scale, nthreads=nthreads,
                           q_seg=None if seg_all is None else seg_all[idx], k_seg=seg_all)
        outs.append(o)
        lses.append(lse.T)
    return np.stack(outs), np.stack(lses)


def block_attention(q_shard, k_shard, v_shard, layout, N, q_rank, kv_rank, causal,
                    scale=None, nthreads=0):
    """Partial attention of one Q shard against one KV shard, [B, S, H, d] inputs.

    The mask follows the global positions the layout gives both shards.
    Returns (O [B, S, H, d], LSE [B, H, S]) in float64, with O = 0 and
    LSE = -inf on rows that see no key of this shard.
    """
    B, S = q_shard.shape[0], q_shard.shape[1]
    qp = layouts.global_position(layout, q_rank, np.arange(S), N, S)
    kp = layouts.global_position(layout, kv_rank, np.arange(S), N, S)
    qb, kb, vb = _bf16_bits(q_shard), _bf16_bits(k_shard), _bf16_bits(v_shard)
    outs, lses = [], []
    for b in range(B):
        o, lse = attention(qb[b], kb[b], vb[b], q_pos=qp, k_pos=kp, causal=causal,
                           scale=scale, nthreads=nthreads)
        outs.append(o)
        lses.append(lse.T)
    return np.stack(outs), np.stack(lses)


__all__ = ["attention", "full_attention", "block_attention", "backward", "blockwise", "layouts",
           "build", "num_threads"]
