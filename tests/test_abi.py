"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "ra.h")


def declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^RA_API\s+[\w\s\*]*?\b(ra_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_four_calls():
    syms = declared_symbols()
    for name in ("ra_shard_permute", "ra_block_attn_fwd", "ra_lse_merge", "ra_ring_attn_fwd"):
        assert name in syms


def test_library_exports_every_declared_symbol(ralib):
    lib = ctypes.CDLL(ralib.library_path())
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(ralib.SIGNATURES)


def test_version(ralib):
    assert "sm_103a" in ralib.ra_version()


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails its checks first


def _ring(ralib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, L=1024, H=2, d=128, N=4, layout=0,
             causal=1, scale=0.0, flags=0, ws=FAKE, wsb=256, stream=None)
    a.update(kw)
    return ralib.lib().ra_ring_attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["L"],
                                        a["H"], a["d"], a["N"], a["layout"], a["causal"], a["scale"],
                                        a["flags"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(L=1022), 2),                         # N does not divide L
    (dict(layout=2, L=1028), 2),               # zigzag needs 2N | L
    (dict(d=96), 3),                           # unsupported head dim
    (dict(N=0), 2),
    (dict(layout=7), 1),
    (dict(flags=8), 1),
    (dict(flags=0x80000001), 1),               # the stall hook is fused-sweep only
    (dict(scale=float("nan")), 1),
    (dict(q=0), 1),                            # null pointer
    (dict(o=FAKE + 8), 4),                     # misaligned
    (dict(wsb=16), 1),                         # workspace too small
    (dict(flags=1, wsb=256), 1),               # stepwise needs the big workspace
    (dict(flags=5), 1),                        # sequence order is fused-sweep only
    (dict(flags=4, layout=2, L=1280), 3),      # sequence-order zigzag: chunk 160 is not a multiple of 128
])
def test_ring_rejects_bad_arguments(ralib, kw, status):
    assert _ring(ralib, **kw) == status
    assert ralib.lib().ra_last_error().decode()


def test_empty_inputs_are_no_ops(ralib):
    assert _ring(ralib, B=0, q=0, k=0, v=0, o=0, lse=0, ws=0) == 0
    assert _ring(ralib, L=0, q=0, k=0, v=0, o=0, lse=0, ws=0) == 0
    lib = ralib.lib()
    assert lib.ra_shard_permute(None, None, 0, 0, 0, 16, 2, 64, 4, 1, 2, None) == 0
    assert lib.ra_lse_merge_bshd(None, None, None, None, 1, 0, 2, 64, None) == 0
    assert lib.ra_lse_merge(None, None, None, None, 0, 64, 64, 64, None) == 0


def test_permute_rejects_bad_arguments(ralib):
    lib = ralib.lib()
    P = lambda *a: lib.ra_shard_permute(FAKE, FAKE + 4096, *a, None)
    assert P(9, 0, 1, 16, 2, 64, 4, 1, 2) == 1          # op
    assert P(0, 5, 1, 16, 2, 64, 4, 1, 2) == 1          # layout
    assert P(0, 0, 1, 18, 2, 64, 4, 1, 2) == 2          # 4 does not divide 18
    assert P(0, 2, 1, 25, 2, 64, 5, 1, 2) == 2          # zigzag needs 2R | L
    assert P(2, 0, 1, 16, 3, 64, 2, 2, 2) == 2          # U does not divide H
    assert P(0, 0, 1, 16, 1, 3, 4, 1, 2) == 4           # 6-byte tokens
    assert P(0, 0, 1, 16, 2, 64, 4, 1, 3) == 1          # elem_bytes
    assert lib.ra_shard_permute(FAKE + 2, FAKE, 0, 0, 1, 16, 2, 64, 4, 1, 2, None) == 4


def test_block_rejects_bad_ranks(ralib):
    lib = ralib.lib()
    st = lib.ra_block_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 4, 0, 0, 1, 0.0,
                               FAKE, 256, None)
    assert st == 1


def test_gqa_rejects_bad_head_counts_on_host(ralib):
    lib = ralib.lib()
    for hkv in (3, 0, 16):
        st = lib.ra_ring_attn_fwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1024, 8, hkv, 128, 4, 0, 1, 0.0, 0,
                                      FAKE, 256, None)
        assert st == 2
    st = lib.ra_block_attn_fwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 8, 3, 128, 4, 0, 0, 0, 1, 0.0,
                                   FAKE, 256, None)
    assert st == 2


def test_varlen_rejects_bad_arguments(ralib):
    lib = ralib.lib()
    V = lambda cu, n: lib.ra_ring_attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, cu, n, 1024, 2, 2, 128, 4,
                                                  0, 1, 0.0, 0, FAKE, 256, None)
    assert V(FAKE, 0) == 2          # no sequences
    assert V(0, 3) == 1             # no boundaries
    assert V(FAKE + 2, 3) == 1      # misaligned boundaries


def test_cu_seqlens_recipe():
    from synthetic_inputs import make_cu_seqlens
    cu = make_cu_seqlens(1000, 17, seed=3)
    assert cu[0] == 0 and cu[-1] == 1000 and len(cu) == 18
    assert bool((cu[1:] > cu[:-1]).all())


def test_workspace_sizes(ralib):
    assert ralib.ra_ring_attn_workspace_bytes(1, 1024, 2, 128, 4, 0) == 256
    n = 1 * 1024 * 2 * 128
    # stepwise, fp32 O: one fp32 partial (O and LSE); the caller's O accumulates
    assert ralib.ra_ring_attn_workspace_bytes(1, 1024, 2, 128, 4, 1) == 256 + n * 4 + 1024 * 2 * 4
    # stepwise, bf16 O: an fp32 accumulator as well
    assert ralib.ra_ring_attn_workspace_bytes(1, 1024, 2, 128, 4, 3) == 256 + 2 * n * 4 + 1024 * 2 * 4
    assert ralib.ra_ring_attn_workspace_bytes(1, 1024, 2, 128, 4, 4) == 256    # sequence order
    assert ralib.ra_ring_attn_workspace_bytes(1, 1024, 2, 128, 4, 5) == 0      # ... not stepwise
    assert ralib.ra_ring_attn_workspace_bytes(1, 1024, 2, 128, 4, 8) == 0      # unknown flag
    assert ralib.ra_ring_attn_workspace_bytes(1, 1024, 2, 96, 4, 0) == 0


def test_launch_chunk_pairs(ralib):
    """The launch-order chunk: all pairs when they stream at most 5/3 of the
    budget together, else the fewest near-equal chunks of at most the budget
    (48 MiB, or what ra_set_launch_chunk_budget set), clamped to [1, pairs]."""
    MiB = 1 << 20
    assert ralib.ra_set_launch_chunk_budget(0) == 48 * MiB     # the default, and it is restored
    assert ralib.ra_launch_chunk_pairs(4 * MiB, 16) == 16      # config 2: 64 MiB in all, one chunk
    assert ralib.ra_launch_chunk_pairs(6 * MiB, 16) == 8       # 96 MiB > 5/3 budget: 8 fit, so 8 + 8
    assert ralib.ra_launch_chunk_pairs(16 * MiB, 64) == 3      # config 3: 3 per chunk
    assert ralib.ra_launch_chunk_pairs(16 * MiB, 8) == 3       # 3 + 3 + 2
    assert ralib.ra_launch_chunk_pairs(64 * MiB, 8) == 1       # a 128K head: one pair per chunk
    assert ralib.ra_launch_chunk_pairs(1 * MiB, 8) == 8
    assert ralib.ra_launch_chunk_pairs(0, 8) == 1
    assert ralib.ra_launch_chunk_pairs(MiB, 0) == 0
    try:
        assert ralib.ra_set_launch_chunk_budget(MiB) == 48 * MiB
        assert ralib.ra_launch_chunk_pairs(512 * 1024, 5) == 2     # 2 + 2 + 1
        assert ralib.ra_launch_chunk_pairs(512 * 1024, 3) == 3     # 1.5 MiB <= 5/3 MiB: one chunk
        for bad in (0, -5):                                        # back to the default
            assert ralib.ra_set_launch_chunk_budget(bad) in (MiB, 48 * MiB)
            assert ralib.ra_launch_chunk_pairs(16 * MiB, 8) == 3, bad
    finally:
        ralib.ra_set_launch_chunk_budget(0)


def test_no_environment_knob(ralib, monkeypatch):
    """The launch order reads nothing from the environment."""
    MiB = 1 << 20
    monkeypatch.setenv("RA_L2_CHUNK_KB", "1024")
    assert ralib.ra_launch_chunk_pairs(16 * MiB, 8) == 3


def test_merge_rejects_bad_arguments(ralib):
    lib = ralib.lib()
    M = lambda rows, d, sa, sb, oa=FAKE, la=FAKE: lib.ra_lse_merge(oa, la, FAKE + 4096, FAKE + 8192, rows, d,
                                                                   sa, sb, None)
    assert M(10, 6, 8, 8) == 3              # d not a multiple of 4
    assert M(10, 260, 260, 260) == 3        # d above 256
    assert M(10, 64, 60, 64) == 2           # rows would overlap
    assert M(10, 64, 66, 64) == 4           # stride not a multiple of 4 floats
    assert M(10, 64, 64, 64, oa=0) == 1     # null
    assert M(10, 64, 64, 64, oa=FAKE + 4) == 4
    assert M(10, 64, 64, 64, la=FAKE + 2) == 4
    assert M(-1, 64, 64, 64) == 2
    assert lib.ra_lse_merge_bshd(FAKE, FAKE + 4, FAKE, FAKE, 1, 8, 2, 64, None) == 4


NOALLOC_CAP = 64 << 20


def _noalloc_need(B, L, H, d):
    r256 = lambda x: (x + 255) // 256 * 256
    return 256 + r256(B * L * H * d * 4) + r256(B * L * H * 4)


def test_noalloc_limit_at_the_boundary(ralib):
    """The stated limit 256 + round256(B*L*H*d*4) + round256(B*L*H*4) <= 64 MiB: a problem
    needing exactly 64 MiB passes the size check (here, without a GPU, it then fails at the
    device lookup), one token more is rejected as too large."""
    lib = ralib.lib()
    assert _noalloc_need(1, 26011, 5, 128) == NOALLOC_CAP
    assert _noalloc_need(1, 26012, 5, 128) > NOALLOC_CAP
    call = lambda L, flags=0: lib.ra_ring_attn_fwd_stepwise_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, L, 5, 128, 1,
                                                                    0, 1, 0.0, flags, None)
    import torch
    if not torch.cuda.is_available():
        assert call(26011) == 5                      # past the checks: no device to look up
    assert call(26012) == 3
    assert "64 MiB" in lib.ra_last_error().decode()
    assert call(26011, flags=1) == 1                 # only the stall hook is a valid flag


def test_noalloc_applies_the_range_checks(ralib):
    """Sizes whose products would wrap around are rejected by the same range checks as
    ra_ring_attn_fwd before any scratch arithmetic."""
    lib = ralib.lib()
    big = lambda B, L, H: lib.ra_ring_attn_fwd_stepwise_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, B, L, H, 128, 1,
                                                                 0, 1, 0.0, 0, None)
    assert big(1 << 21, 1 << 20, 1 << 21) == 3     # B*L*H = 2^62: would wrap the byte count to 0
    assert big(1, 1 << 20, 1 << 21) == 3
    assert big(1 << 21, 16, 1) == 3


def _bwd(ralib, **kw):
    a = dict(B=1, L=1024, H=2, Hkv=2, d=128, N=4, layout=0, causal=1, scale=0.0, flags=0)
    a.update(kw)
    return ralib.lib().ra_ring_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0,
                                        a["B"], a["L"], a["H"], a["Hkv"], a["d"], a["N"], a["layout"],
                                        a["causal"], a["scale"], a["flags"], FAKE, 16, None)


@pytest.mark.parametrize("kw,status", [
    (dict(flags=1), 1),                        # only RA_FLAG_SEQ_ORDER applies to the backward
    (dict(flags=4, layout=2, L=1280), 3),      # token-order zigzag: chunk 160 is not a multiple of 128
    (dict(flags=4), 1),                        # then the small workspace is rejected
    (dict(d=96), 3),
])
def test_backward_rejects_bad_arguments(ralib, kw, status):
    assert _bwd(ralib, **kw) == status
    assert ralib.lib().ra_last_error().decode()


def _ctype_of(decl):
    """ctypes class of one C parameter or return declaration of include/ra.h."""
    decl = " ".join(decl.replace("const", " ").split())
    if decl.startswith("char *") or decl == "char *":
        return ctypes.c_char_p
    if "*" in decl:
        return ctypes.c_void_p
    base = decl.split()[0]
    return {"int64_t": ctypes.c_int64, "int": ctypes.c_int, "unsigned": ctypes.c_uint,
            "float": ctypes.c_float, "size_t": ctypes.c_size_t, "ra_status": ctypes.c_int}[base]


def test_binding_signatures_match_the_header(ralib):
    """Every prototype's return and parameter types, as the Python binding declares them to
    ctypes: a parameter added to a C call without its ctypes slot would shift every argument
    after it."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = re.findall(r"^RA_API\s+([\w\s\*]*?)\b(ra_\w+)\s*\(([^)]*)\)\s*;", src, flags=re.M)
    assert len(protos) == len(ralib.SIGNATURES)
    for ret, name, params in protos:
        params = params.strip()
        args = [] if params in ("", "void") else [_ctype_of(p.rsplit(None, 1)[0] if "*" not in p.split()[-1]
                                                           else p[:p.rfind("*") + 1]) for p in params.split(",")]
        want_ret, want_args = ralib.SIGNATURES[name]
        assert _ctype_of(ret.strip()) is want_ret, name
        assert args == list(want_args), name
