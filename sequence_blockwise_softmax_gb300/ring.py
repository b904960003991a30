"""The ring over real ranks: each rank's KV shard travels round the ring while
the block kernel works on the one that is already there.

"From Ring Attention to DeepSpeed Ulysses to USP" (jsqmd.com/news/734632),
§3.3: at step s rank i holds the key/value shard of rank (i - s) mod N, sends
it to rank i + 1 and receives the next one from rank i - 1 while it computes
its block; §3.2 / §6.3: the partial results are folded with the LSE merge;
§6.2: compute and communication run on two streams so the transfer hides
behind the block kernel.

GB300 form of that loop, per rank:

  * Step 0 computes on the caller's own K and V shards; from step 1 on, the
    shards arrive in two local buffer pairs (K and V, bf16, 2 * B * S * H_kv *
    d * 2 bytes per step): step s computes on pair s % 2 while pair
    (s + 1) % 2 receives the next shard into LOCAL memory, so every kernel (TMA
    included) reads only this GPU's HBM; no peer memory is mapped and nothing
    multicasts.
  * The transfer of step s starts once step s - 1's kernels, which read the
    receiving buffer, are done (an event on the compute stream), runs on its
    own stream, and the compute stream waits for it only before step s + 1.
  * Step 0 (the rank's own shard, which always holds its diagonal) writes O
    and LSE directly; every later step that has any visible pair runs
    ra_block_attn_fwd into a partial and ra_lse_merge_bshd folds it in.  A step
    with no visible pair (contiguous layout, causal, a later rank's shard:
    ra_ring_step_pairs() = 0) launches nothing, but the shard still moves on.

Two transports share that loop:

  * ProcessGroupRing -- one process per GPU, torch.distributed point-to-point
    (NCCL on GPUs; gloo on CPU tensors for the host-side tests): the send to
    i + 1 and the receive from i - 1 of a step form one batch, so no rank's send
    waits behind its own receive;
  * LoopbackRing -- all N ranks in one process on one GPU: the shift is one
    device-to-device copy per rank on a copy stream.  Same buffers, same
    order of kernels, so a single GPU checks the whole driver.

Everything the method computes runs in the library's kernels; this module only
orders launches and transfers.
"""
import torch

from . import (RA_WORKSPACE_MIN_BYTES, _layout, new_workspace, ra_block_attn_fwd_gqa, ra_lse_merge_bshd,
               ra_ring_step_pairs)


def ring_schedule(layout, S, N, rank, causal):
    """[(step, key/value rank, visible pairs)] for query rank ``rank`` over the N steps."""
    out = []
    for s in range(N):
        j = (rank - s) % N
        out.append((s, j, ra_ring_step_pairs(layout, S, N, rank, j, causal)))
    return out


def ring_bytes_per_step(B, S, Hkv, d, elem_bytes=2):
    """Bytes one rank sends (and receives) per ring step: its K and V shard."""
    return 2 * B * S * Hkv * d * elem_bytes


class RingRank:
    """One rank of the ring: its query and own K/V shards, the two receive buffers,
    O / LSE and the partial.  run_ring() may run it any number of times."""

    def __init__(self, q, k, v, rank, N, layout, causal, scale=0.0, block_fn=None, merge_fn=None, o=None,
                 lse=None):
        B, S, H, d = q.shape
        Hkv = k.shape[2]
        assert k.shape == (B, S, Hkv, d) and v.shape == k.shape
        assert q.is_contiguous() and k.is_contiguous() and v.is_contiguous()
        self.q, self.k0, self.v0 = q, k, v
        self.rank, self.N, self.layout, self.causal, self.scale = rank, N, layout, causal, scale
        self.B, self.S, self.H, self.Hkv, self.d = B, S, H, Hkv, d
        dev = q.device
        # receive buffers: pair s % 2 holds the shard of step s >= 1
        self.kb = [torch.empty_like(k) for _ in range(2)] if N > 1 else []
        self.vb = [torch.empty_like(v) for _ in range(2)] if N > 1 else []
        # outputs: the caller's (contiguous fp32 [B, S, H, d] and [B, H, S]) or new tensors
        self.o = o if o is not None else torch.empty((B, S, H, d), dtype=torch.float32, device=dev)
        self.lse = lse if lse is not None else torch.empty((B, H, S), dtype=torch.float32, device=dev)
        assert self.o.shape == (B, S, H, d) and self.lse.shape == (B, H, S)
        assert self.o.is_contiguous() and self.lse.is_contiguous()
        self.o_part = torch.empty_like(self.o)
        self.lse_part = torch.empty_like(self.lse)
        self.schedule = ring_schedule(_layout(layout), S, N, rank, causal)
        self.ws = new_workspace(RA_WORKSPACE_MIN_BYTES, device=dev) if dev.type == "cuda" else None
        self.block_fn = block_fn or self._block
        self.merge_fn = merge_fn or self._merge
        self.launched = 0          # library launches issued by the last run (block calls and merges)

    def kv(self, s):
        """The K and V shards step s computes on (and passes on)."""
        return (self.k0, self.v0) if s == 0 else (self.kb[s % 2], self.vb[s % 2])

    def recv_buffers(self, s):
        """Where the shard of step s + 1 arrives."""
        return self.kb[(s + 1) % 2], self.vb[(s + 1) % 2]

    def _block(self, q, k, v, o, lse, q_rank, kv_rank):
        ra_block_attn_fwd_gqa(q, k, v, o, lse, self.B, self.S, self.H, self.Hkv, self.d, self.N, q_rank, kv_rank,
                              self.layout, self.causal, self.scale, workspace=self.ws)

    def _merge(self, o, lse, o_part, lse_part):
        ra_lse_merge_bshd(o, lse, o_part, lse_part, self.B, self.S, self.H, self.d)

    def compute(self, s):
        """Step s on the shard it holds."""
        step, j, pairs = self.schedule[s]
        if step != 0 and pairs == 0:
            return
        k, v = self.kv(s)
        if step == 0:
            self.block_fn(self.q, k, v, self.o, self.lse, self.rank, j)
            self.launched += 1
        else:
            self.block_fn(self.q, k, v, self.o_part, self.lse_part, self.rank, j)
            self.merge_fn(self.o, self.lse, self.o_part, self.lse_part)
            self.launched += 2


class LoopbackRing:
    """All N ranks in this process (one GPU): the shard rank r holds at step s is copied
    into rank (r + 1)'s receive buffers for step s + 1."""

    def shift(self, ranks, s):
        n = len(ranks)
        for r in ranks:
            dk, dv = ranks[(r.rank + 1) % n].recv_buffers(s)
            k, v = r.kv(s)
            dk.copy_(k, non_blocking=True)
            dv.copy_(v, non_blocking=True)
        return None

    def wait(self, handle):
        pass


class ProcessGroupRing:
    """One rank per process: at step s, send the K and V shards the rank holds to rank + 1
    and receive those of step s + 1 from rank - 1, as one batch of point-to-point
    operations."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist, self.group = dist, group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def _global(self, r):
        return r if self.group is None else self.dist.get_global_rank(self.group, r)

    def shift(self, ranks, s):
        (me,) = ranks
        dist = self.dist
        nxt, prv = self._global((self.rank + 1) % self.world), self._global((self.rank - 1) % self.world)
        (k, v), (rk, rv) = me.kv(s), me.recv_buffers(s)
        ops = [dist.P2POp(dist.isend, k, nxt, self.group), dist.P2POp(dist.isend, v, nxt, self.group),
               dist.P2POp(dist.irecv, rk, prv, self.group), dist.P2POp(dist.irecv, rv, prv, self.group)]
        return dist.batch_isend_irecv(ops)

    def wait(self, handle):
        for req in handle:
            req.wait()


def run_ring(ranks, ring, comm_stream=None):
    """Run the N steps for ``ranks`` (one per process, or all N with LoopbackRing).

    On CUDA tensors the transfers run on ``comm_stream`` (a new stream if None) and the
    kernels on the current stream; the call returns once everything is enqueued."""
    N = ranks[0].N
    cuda = ranks[0].q.is_cuda
    for r in ranks:
        r.launched = 0
    compute = torch.cuda.current_stream() if cuda else None
    if cuda and comm_stream is None:
        comm_stream = torch.cuda.Stream()
    for s in range(N):
        handle = None
        if s + 1 < N:
            if cuda:
                # the receiving buffer was read by step s - 1's kernels
                ready = torch.cuda.Event()
                ready.record(compute)
                comm_stream.wait_event(ready)
                with torch.cuda.stream(comm_stream):
                    handle = ring.shift(ranks, s)
                    done = torch.cuda.Event()
                    done.record(comm_stream)
            else:
                handle = ring.shift(ranks, s)
        for r in ranks:
            r.compute(s)
        if s + 1 < N:
            ring.wait(handle)                  # NCCL: the current (compute) stream waits
            if cuda:
                compute.wait_event(done)       # the copy stream's work (loopback) and NCCL's
    return ranks


def ring_attention_fwd(q, k, v, rank, N, layout, causal, scale=0.0, group=None, comm_stream=None):
    """One rank's part of the ring, one process per GPU: q, k, v are this rank's shards
    [B, S, H(_kv), d] bf16 in ``layout`` over N ranks (N = the group's size).  Returns
    (O [B, S, H, d] fp32, LSE [B, H, S] fp32) of this rank's queries over the whole sequence."""
    ring = ProcessGroupRing(group)
    assert ring.world == N and ring.rank == rank
    me = RingRank(q, k, v, rank, N, layout, causal, scale)
    run_ring([me], ring, comm_stream)
    return me.o, me.lse


def ring_attention_fwd_loopback(q, k, v, N, layout, causal, scale=0.0, comm_stream=None):
    """All N ranks on this GPU through the same driver: q, k, v are shard stacks
    [N, B, S, H(_kv), d].  Returns O [N, B, S, H, d] and LSE [N, B, H, S] (fp32) and the
    number of library launches."""
    ranks = loopback_ranks(q, k, v, N, layout, causal, scale)
    run_ring(ranks, LoopbackRing(), comm_stream)
    return (torch.stack([r.o for r in ranks]), torch.stack([r.lse for r in ranks]),
            sum(r.launched for r in ranks))


def loopback_ranks(q, k, v, N, layout, causal, scale=0.0, o=None, lse=None):
    """The N RingRank objects of shard stacks [N, B, S, H(_kv), d] on one GPU, for repeated
    run_ring(ranks, LoopbackRing()) calls; with ``o`` [N, B, S, H, d] and ``lse``
    [N, B, H, S] (fp32) the ranks write their results there."""
    return [RingRank(q[i], k[i], v[i], i, N, layout, causal, scale,
                     o=None if o is None else o[i], lse=None if lse is None else lse[i]) for i in range(N)]
