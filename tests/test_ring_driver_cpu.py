"""The multi-GPU ring driver's schedule and exchange, with real process groups on the CPU.

``sequence_blockwise_softmax_gb300.ring`` runs the pages' per-rank loop ("From Ring
Attention to DeepSpeed Ulysses to USP", jsqmd.com/news/734632, §3.3: at step s rank i
holds the KV shard of rank (i - s) mod N, passes it to i + 1 and receives the next one
from i - 1; §6.3: partials folded by their LSE).  Here 2 and 4 gloo ranks (spawned
processes, CPU tensors) run it with the oracle's block attention and LSE merge put in
place of the kernels, so that what is tested is the driver alone:

  * at every step the K and V a rank computes with are exactly shard (i - s) mod N
    (the right shard arrived, in the buffer the step reads, not overwritten);
  * steps with no visible pair (contiguous, causal, a later rank's shard) launch
    nothing, and every other step launches one block call and, after step 0, one merge;
  * the folded result equals the oracle's full attention for the rank's queries.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, layout, causal, Hkv, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import oracle.blockwise as bw
        import oracle.layouts as ly
        from sequence_blockwise_softmax_gb300 import ring
        from synthetic_inputs import make_qkv

        B, L, H, d = 1, 96 * world, 4, 16
        N, S = world, 96
        q, k, v, _ = make_qkv(B, L, H, d, seed=900 + world)
        k, v = k[:, :, :Hkv].contiguous(), v[:, :, :Hkv].contiguous()
        shards = [ly.seq_to_shards(x.float().numpy(), layout, N) for x in (q, k, v)]
        mine = [torch.from_numpy(np.ascontiguousarray(x[rank])).to(torch.bfloat16) for x in shards]
        seen = []

        def block_fn(qs, ks, vs, o, lse, q_rank, kv_rank):
            # the shard in the buffer must be rank kv_rank's
            assert torch.equal(ks, torch.from_numpy(shards[1][kv_rank]).to(torch.bfloat16))
            assert torch.equal(vs, torch.from_numpy(shards[2][kv_rank]).to(torch.bfloat16))
            kk = ks.repeat_interleave(H // Hkv, dim=2)
            vv = vs.repeat_interleave(H // Hkv, dim=2)
            ob, lb = oracle.block_attention(qs, kk, vv, layout, N, q_rank, kv_rank, causal)
            o.copy_(torch.from_numpy(ob))
            lse.copy_(torch.from_numpy(lb))
            seen.append(kv_rank)

        def merge_fn(o, lse, o_part, lse_part):
            om, lm = bw.lse_merge(o.double().numpy().transpose(0, 2, 1, 3), lse.double().numpy(),
                                  o_part.double().numpy().transpose(0, 2, 1, 3), lse_part.double().numpy())
            o.copy_(torch.from_numpy(om.transpose(0, 2, 1, 3)))
            lse.copy_(torch.from_numpy(lm))

        me = ring.RingRank(*mine, rank, N, layout, causal, block_fn=block_fn, merge_fn=merge_fn)
        ring.run_ring([me], ring.ProcessGroupRing())
        pos = ly.global_position(layout, rank, np.arange(S), N, S)
        o_ref, lse_ref = oracle.full_attention(q, k.repeat_interleave(H // Hkv, dim=2),
                                               v.repeat_interleave(H // Hkv, dim=2), causal, rows=pos)
        out[rank] = dict(seen=seen, launched=me.launched, schedule=me.schedule,
                         err_o=float(np.abs(me.o.double().numpy() - o_ref).max()),
                         err_l=float(np.abs(me.lse.double().numpy() - lse_ref).max()))
    finally:
        dist.destroy_process_group()


def _run(world, layout, causal, Hkv=4):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, layout, causal, Hkv, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(240)
            assert p.exitcode == 0
        return dict(out)


@pytest.mark.parametrize("world,layout,causal,Hkv", [
    (2, "striped", True, 4), (2, "contiguous", True, 2), (4, "contiguous", True, 4),
    (4, "zigzag", True, 1), (4, "striped", False, 4),
])
def test_ring_driver_on_gloo_ranks(ralib, world, layout, causal, Hkv):
    res = _run(world, layout, causal, Hkv)
    for i in range(world):
        r = res[i]
        ring_order = [(i - s) % world for s in range(world)]
        active = [j for s, j, pairs in r["schedule"] if s == 0 or pairs > 0]
        assert [j for _, j, _ in r["schedule"]] == ring_order
        # the block calls saw exactly the active shards, in ring order
        assert r["seen"] == active
        assert r["launched"] == 1 + 2 * (len(active) - 1)
        if layout == "contiguous" and causal:
            assert active == [j for j in ring_order if j <= i]
        else:
            assert active == ring_order
        assert r["err_o"] <= 1e-5 and r["err_l"] <= 1e-5, r


def test_schedule_pairs_match_the_pair_table(ralib):
    """ra_ring_step_pairs (the kernels' position code, on the host) against the pair counts
    taken from the layouts' token positions (bench.ring_pair_counts, itself pinned by brute
    force over the oracle's positions)."""
    import bench
    from sequence_blockwise_softmax_gb300 import ring
    for layout in ("contiguous", "striped", "zigzag"):
        for N, S in ((4, 96), (5, 64), (16, 128)):
            table = bench.ring_pair_counts(layout, N, S, True)
            for i in range(N):
                sched = ring.ring_schedule(layout, S, N, i, True)
                assert [p for _, _, p in sched] == table[i].tolist()
            assert ring.ring_schedule(layout, S, N, 0, False)[1][2] == S * S


def test_bytes_per_step():
    from sequence_blockwise_softmax_gb300 import ring
    # the 128K workload over 16 ranks: K and V of one 8192-token shard, 8 heads of 128, bf16
    assert ring.ring_bytes_per_step(1, 8192, 8, 128) == 2 * 8192 * 8 * 128 * 2
