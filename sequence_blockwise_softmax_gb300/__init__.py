"""Python binding of the GB300 ring-attention library (``libra_gb300.so``).

Argument marshalling only: every function here checks that it was given CUDA
tensors, takes their device pointers and the current CUDA stream, and calls
the C entry point of the same name declared in ``include/ra.h``.  All work
runs in the library's kernels; there is no fallback of any kind -- if the
library is missing, the first call raises.

Layouts (see ``include/ra.h``): full sequences are ``[B, L, H, d]``; shard
stacks ``[N, B, S, H, d]``; LSE ``[.., H, S]`` fp32 in natural log.
"""
import ctypes
import os

import torch

from . import build as _build

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_SHAPE, RA_ERR_UNSUPPORTED, RA_ERR_ALIGNMENT, RA_ERR_CUDA, \
    RA_ERR_TIMEOUT = range(7)
RA_CONTIGUOUS, RA_STRIPED, RA_ZIGZAG = range(3)
RA_SEQ_TO_SHARDS, RA_SHARDS_TO_SEQ, RA_ULYSSES_SEQ_TO_HEAD, RA_ULYSSES_HEAD_TO_SEQ = range(4)
RA_FLAG_STEPWISE = 1
RA_FLAG_O_BF16 = 2
RA_FLAG_SEQ_ORDER = 4
RA_FLAG_INJECT_STALL = 0x80000000
RA_WORKSPACE_MIN_BYTES = 256
LAYOUTS = {"contiguous": RA_CONTIGUOUS, "striped": RA_STRIPED, "zigzag": RA_ZIGZAG}

# every exported symbol of include/ra.h with its ctypes signature
_P, _I, _I64, _U, _F, _SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint,
                             ctypes.c_float, ctypes.c_size_t)
SIGNATURES = {
    "ra_shard_permute": (_I, [_P, _P, _I, _I, _I64, _I64, _I64, _I64, _I, _I, _I, _P]),
    "ra_lse_to_seq": (_I, [_P, _P, _I, _I64, _I64, _I64, _I, _I, _P]),
    "ra_block_attn_fwd": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _I, _I, _I, _F,
                               _P, _SZ, _P]),
    "ra_lse_merge": (_I, [_P, _P, _P, _P, _I64, _I, _I64, _I64, _P]),
    "ra_lse_merge_bshd": (_I, [_P, _P, _P, _P, _I64, _I64, _I64, _I, _P]),
    "ra_ring_attn_fwd": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _I, _F, _U, _P,
                              _SZ, _P]),
    "ra_ring_attn_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I, _I, _U]),
    "ra_block_attn_fwd_gqa": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I, _I, _I, _I, _I, _I,
                                   _F, _P, _SZ, _P]),
    "ra_ring_attn_fwd_gqa": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I, _I, _I, _I, _F, _U,
                                  _P, _SZ, _P]),
    "ra_ring_attn_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _I, _I, _I, _F,
                                     _U, _P, _SZ, _P]),
    "ra_ring_attn_fwd_stepwise_noalloc": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _I,
                                               _F, _U, _P]),
    "ra_noalloc_check_status": (_I, [_P]),
    "ra_ring_attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I64, _I, _I,
                              _I, _I, _F, _U, _P, _SZ, _P]),
    "ra_ring_attn_bwd_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I, _I]),
    "ra_check_status": (_I, [_P, _P]),
    "ra_last_error": (ctypes.c_char_p, []),
    "ra_version": (ctypes.c_char_p, []),
    "ra_ring_step_pairs": (_I64, [_I, _I64, _I, _I, _I, _I]),
    "ra_set_launch_chunk_budget": (_I64, [_I64]),
    "ra_launch_chunk_pairs": (_I64, [_I64, _I64]),
}

_lib = None


class RAError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("ra status %d: %s" % (status, msg))
        self.status = status


def library_path():
    return _build.LIB


def lib():
    """Load libra_gb300.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError("libra_gb300.so is not built (%s); run __graft_entry__.build()" % path)
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(st):
    if st != RA_OK:
        raise RAError(st, lib().ra_last_error().decode())


def _ptr(t, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _layout(layout):
    return LAYOUTS[layout] if isinstance(layout, str) else int(layout)


def ra_shard_permute(src, dst, op, layout, B, L, H, d, R, U=1, stream=None):
    assert src.dtype == dst.dtype
    _check(lib().ra_shard_permute(_ptr(src, "src"), _ptr(dst, "dst"), int(op), _layout(layout),
                                  B, L, H, d, R, U, src.element_size(), _stream(stream)))


def ra_lse_to_seq(src, dst, layout, B, L, H, R, U=1, stream=None):
    assert src.dtype == torch.float32 and dst.dtype == torch.float32
    _check(lib().ra_lse_to_seq(_ptr(src, "src"), _ptr(dst, "dst"), _layout(layout), B, L, H, R, U,
                               _stream(stream)))


def ra_block_attn_fwd(q, k, v, o, lse, B, S, H, d, N, q_rank, kv_rank, layout, causal,
                      scale=0.0, workspace=None, stream=None):
    for t in (q, k, v):
        assert t.dtype == torch.bfloat16
    assert o.dtype == torch.float32 and lse.dtype == torch.float32
    _check(lib().ra_block_attn_fwd(_ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(o, "o"),
                                   _ptr(lse, "lse"), B, S, H, d, N, q_rank, kv_rank,
                                   _layout(layout), int(bool(causal)), float(scale),
                                   _ptr(workspace, "workspace"),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))


def _ptr_view(t, name):
    """Device pointer of a CUDA tensor that may be a strided view (the C call takes strides)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    return t.data_ptr()


def ra_lse_merge(o_acc, lse_acc, o_b, lse_b, stream=None):
    """Strided merge: o_acc, o_b are [rows, d] fp32 views whose rows may be strided (unit
    stride along d); lse_acc, lse_b are contiguous [rows] fp32."""
    for t in (o_acc, o_b):
        assert t.dtype == torch.float32 and t.dim() == 2 and t.stride(1) == 1
    for t in (lse_acc, lse_b):
        assert t.dtype == torch.float32 and t.dim() == 1 and t.is_contiguous()
    rows, d = o_acc.shape
    assert o_b.shape == (rows, d) and lse_acc.numel() == rows and lse_b.numel() == rows
    _check(lib().ra_lse_merge(_ptr_view(o_acc, "o_acc"), _ptr(lse_acc, "lse_acc"), _ptr_view(o_b, "o_b"),
                              _ptr(lse_b, "lse_b"), rows, d, o_acc.stride(0), o_b.stride(0),
                              _stream(stream)))


def ra_lse_merge_bshd(o_acc, lse_acc, o_b, lse_b, B, S, H, d, stream=None):
    _check(lib().ra_lse_merge_bshd(_ptr(o_acc, "o_acc"), _ptr(lse_acc, "lse_acc"), _ptr(o_b, "o_b"),
                                   _ptr(lse_b, "lse_b"), B, S, H, d, _stream(stream)))


def ra_ring_attn_workspace_bytes(B, L, H, d, N, flags=0):
    return int(lib().ra_ring_attn_workspace_bytes(B, L, H, d, N, flags))


def ra_ring_attn_fwd(q, k, v, o, lse, B, L, H, d, N, layout, causal, scale=0.0, flags=0,
                     workspace=None, stream=None):
    """O may be fp32 (default) or bf16; a bf16 ``o`` sets RA_FLAG_O_BF16."""
    for t in (q, k, v):
        assert t.dtype == torch.bfloat16
    assert o.dtype in (torch.float32, torch.bfloat16) and lse.dtype == torch.float32
    if o.dtype == torch.bfloat16:
        flags |= RA_FLAG_O_BF16
    _check(lib().ra_ring_attn_fwd(_ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(o, "o"),
                                  _ptr(lse, "lse"), B, L, H, d, N, _layout(layout),
                                  int(bool(causal)), float(scale), int(flags),
                                  _ptr(workspace, "workspace"),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def ra_ring_attn_fwd_stepwise_noalloc(q, k, v, o, lse, B, L, H, d, N, layout, causal, scale=0.0,
                                      flags=0, stream=None):
    """Stepwise sweep with the library's own fixed scratch array; O is fp32."""
    for t in (q, k, v):
        assert t.dtype == torch.bfloat16
    assert o.dtype == torch.float32 and lse.dtype == torch.float32
    _check(lib().ra_ring_attn_fwd_stepwise_noalloc(_ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"),
                                                   _ptr(o, "o"), _ptr(lse, "lse"), B, L, H, d, N,
                                                   _layout(layout), int(bool(causal)), float(scale),
                                                   int(flags), _stream(stream)))


def ra_noalloc_check_status(stream=None):
    _check(lib().ra_noalloc_check_status(_stream(stream)))


def ra_block_attn_fwd_gqa(q, k, v, o, lse, B, S, H, H_kv, d, N, q_rank, kv_rank, layout, causal,
                          scale=0.0, workspace=None, stream=None):
    """ra_block_attn_fwd with H_kv key/value heads (k, v are [B, S, H_kv, d])."""
    for t in (q, k, v):
        assert t.dtype == torch.bfloat16
    assert o.dtype == torch.float32 and lse.dtype == torch.float32
    _check(lib().ra_block_attn_fwd_gqa(_ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(o, "o"),
                                       _ptr(lse, "lse"), B, S, H, H_kv, d, N, q_rank, kv_rank,
                                       _layout(layout), int(bool(causal)), float(scale),
                                       _ptr(workspace, "workspace"),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))


def ra_ring_attn_fwd_gqa(q, k, v, o, lse, B, L, H, H_kv, d, N, layout, causal, scale=0.0, flags=0,
                         workspace=None, stream=None):
    """ra_ring_attn_fwd with H_kv key/value heads (k, v are [N, B, S, H_kv, d])."""
    for t in (q, k, v):
        assert t.dtype == torch.bfloat16
    assert o.dtype in (torch.float32, torch.bfloat16) and lse.dtype == torch.float32
    if o.dtype == torch.bfloat16:
        flags |= RA_FLAG_O_BF16
    _check(lib().ra_ring_attn_fwd_gqa(_ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(o, "o"),
                                      _ptr(lse, "lse"), B, L, H, H_kv, d, N, _layout(layout),
                                      int(bool(causal)), float(scale), int(flags),
                                      _ptr(workspace, "workspace"),
                                      workspace.numel() * workspace.element_size(), _stream(stream)))


def ra_ring_attn_fwd_varlen(q, k, v, o, lse, cu_seqlens, L, H, H_kv, d, N, layout, causal, scale=0.0,
                            flags=0, workspace=None, stream=None):
    """Ring sweep over packed sequences; ``cu_seqlens`` is an int32 CUDA tensor of n_seqs + 1
    boundaries (B = 1)."""
    for t in (q, k, v):
        assert t.dtype == torch.bfloat16
    assert o.dtype in (torch.float32, torch.bfloat16) and lse.dtype == torch.float32
    assert cu_seqlens.dtype == torch.int32
    if o.dtype == torch.bfloat16:
        flags |= RA_FLAG_O_BF16
    _check(lib().ra_ring_attn_fwd_varlen(_ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(o, "o"),
                                         _ptr(lse, "lse"), _ptr(cu_seqlens, "cu_seqlens"),
                                         cu_seqlens.numel() - 1, L, H, H_kv, d, N, _layout(layout),
                                         int(bool(causal)), float(scale), int(flags),
                                         _ptr(workspace, "workspace"),
                                         workspace.numel() * workspace.element_size(), _stream(stream)))


def ra_ring_attn_bwd_workspace_bytes(B, L, H, d, N):
    return int(lib().ra_ring_attn_bwd_workspace_bytes(B, L, H, d, N))


def ra_ring_attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, L, H, H_kv, d, N, layout, causal,
                     scale=0.0, cu_seqlens=None, workspace=None, stream=None, flags=0):
    """Gradients of the ring attention; o fp32, dout bf16; dq / dk / dv fp32 outputs."""
    for t in (q, k, v, dout):
        assert t.dtype == torch.bfloat16
    for t in (o, lse, dq, dk, dv):
        assert t.dtype == torch.float32
    n_seqs = 0
    if cu_seqlens is not None:
        assert cu_seqlens.dtype == torch.int32
        n_seqs = cu_seqlens.numel() - 1
    _check(lib().ra_ring_attn_bwd(_ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(o, "o"),
                                  _ptr(dout, "dout"), _ptr(lse, "lse"), _ptr(dq, "dq"), _ptr(dk, "dk"),
                                  _ptr(dv, "dv"), _ptr(cu_seqlens, "cu_seqlens"), n_seqs, B, L, H, H_kv,
                                  d, N, _layout(layout), int(bool(causal)), float(scale), int(flags),
                                  _ptr(workspace, "workspace"),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def ra_check_status(workspace, stream=None):
    _check(lib().ra_check_status(_ptr(workspace, "workspace"), _stream(stream)))


def ra_version():
    return lib().ra_version().decode()


def ra_ring_step_pairs(layout, S, N, q_rank, kv_rank, causal):
    """Visible (query, key) pairs of query shard q_rank against key/value shard kv_rank."""
    n = int(lib().ra_ring_step_pairs(_layout(layout), int(S), int(N), int(q_rank), int(kv_rank),
                                     int(bool(causal))))
    if n < 0:
        raise RAError(RA_ERR_INVALID_ARG, "bad arguments to ra_ring_step_pairs")
    return n


def ra_set_launch_chunk_budget(nbytes):
    """Set the launch-order chunk budget (<= 0: the default); returns the previous one."""
    return int(lib().ra_set_launch_chunk_budget(int(nbytes)))


def ra_launch_chunk_pairs(per_pair_bytes, pairs):
    return int(lib().ra_launch_chunk_pairs(int(per_pair_bytes), int(pairs)))


def new_workspace(nbytes, device="cuda"):
    """A zero-filled device workspace of at least ``nbytes`` bytes (16-byte aligned)."""
    n = max(int(nbytes), RA_WORKSPACE_MIN_BYTES)
    return torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device=device)
