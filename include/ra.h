/*
 * ra.h -- C ABI of the GB300 ring-attention library (libra_gb300.so).
 *
 * Exact blockwise attention, softmax(Q K^T / sqrt(d)) V, over a sequence
 * split into N shards ("virtual ranks") that all live on ONE GPU.  Each query
 * shard is swept over the key/value shards in ring order and the partial
 * results are combined with the online-softmax merge; the causal mask is
 * decided from global token positions.  Sources (page title, section):
 *   [USP]  "From Ring Attention to DeepSpeed Ulysses to USP"
 *          (jsqmd.com/news/734632): §2 attention, §3.1 ring order,
 *          §3.2 online softmax, §3.4 causal imbalance, §4 striped,
 *          §5.1 Ulysses, §6.1 zigzag, §6.3 LSE merge, §7.1-7.2 USP.
 *   [SPQ]  "What problem does sequence parallelism solve?"
 *          (model.playoffer.cn, sequence-parallelism): engineering notes
 *          (the ring decides the causal mask by position).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates device memory and keeps no pointer after a call returns.
 *   - Every pointer must be 16-byte aligned (RA_ERR_ALIGNMENT otherwise),
 *     unless its call states a weaker rule.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous and stream-ordered.
 *   - Arguments are checked on the host before anything is launched; a failed
 *     check returns a status and launches nothing.  ra_last_error() then gives
 *     a message (per host thread).
 *   - A launch failure returns RA_ERR_CUDA.
 *   - Every wait inside the attention kernels is bounded (about two seconds);
 *     a kernel that gives up records RA_ERR_TIMEOUT in the status word at the
 *     start of `workspace`, releases what it holds and exits.
 *     ra_check_status() reports and clears it.
 *   - Tensors are row-major.  Full-sequence tensors are [B, L, H, d] (the
 *     pages' [bs, seq, heads, head_dim]); a stack of N shards is
 *     [N, B, S, H, d] with S = L / N; LSE tensors are fp32 [.., H, S] in
 *     natural log.
 */
#ifndef RA_GB300_H
#define RA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RA_API __attribute__((visibility("default")))
#else
#define RA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = 1,  /* null pointer, bad enum, bad flag, bad scale        */
    RA_ERR_SHAPE = 2,        /* sizes that do not divide as the layout needs       */
    RA_ERR_UNSUPPORTED = 3,  /* a valid request this build does not implement      */
    RA_ERR_ALIGNMENT = 4,    /* a pointer or row that is not 16-byte aligned       */
    RA_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed               */
    RA_ERR_TIMEOUT = 6       /* a kernel gave up on a bounded wait                 */
} ra_status;

/* Token -> rank assignment.  Rank r, local token s holds global token:
 *   RA_CONTIGUOUS  r*S + s                                   ([USP] §3.1, §4)
 *   RA_STRIPED     s*N + r                                   ([USP] §4)
 *   RA_ZIGZAG      2N chunks of C = S/2 tokens; rank r holds chunks r and
 *                  2N-1-r in that order: s < C -> r*C + s,
 *                  s >= C -> (2N-1-r)*C + (s - C)            ([USP] §6.1)   */
typedef enum { RA_CONTIGUOUS = 0, RA_STRIPED = 1, RA_ZIGZAG = 2 } ra_layout;

typedef enum {
    RA_SEQ_TO_SHARDS = 0,        /* [B, L, H, d] -> [U*R, B, L/(U*R), H, d]        */
    RA_SHARDS_TO_SEQ = 1,        /* inverse of RA_SEQ_TO_SHARDS                     */
    RA_ULYSSES_SEQ_TO_HEAD = 2,  /* [U*R, B, L/(U*R), H, d] -> [R, U, B, L/R, H/U, d] */
    RA_ULYSSES_HEAD_TO_SEQ = 3   /* inverse of RA_ULYSSES_SEQ_TO_HEAD               */
} ra_perm_op;

/* Launch order.  Causal work grows with position, so the attention kernels
 * (forward and both backward passes) run heavy units first.  They take
 * (batch, head) pairs in chunks whose streamed keys and values (queries and dO
 * in the dK/dV pass) fit in L2 together, 48 MiB per chunk by default (all
 * pairs at once when they fit in 5/3 of that), and interleave the units of a
 * chunk's pairs heaviest first.  ra_set_launch_chunk_budget() changes the
 * budget for the whole process (the one setting this library keeps besides
 * the error text); nothing is read from the environment.  The order never
 * changes a result: every unit's arithmetic is independent of when it runs. */

/* ra_ring_attn_fwd flags */
#define RA_FLAG_STEPWISE 1u  /* run the sweep as N x (block attention + LSE merge) */
#define RA_FLAG_O_BF16 2u    /* write O as bf16 (rounded once, to nearest even)
                                instead of the default fp32 accumulator         */
/* Sequence order: q, k, v and o are the full-sequence tensors [B, L, H, d]
 * ([B, L, H_kv, d] for k and v) in token order and lse is [B, H, L], instead
 * of shard stacks.  The fused sweep reads each rank's shard and writes its
 * result straight from and to token order, the layout ([USP] §4, §6.1) being
 * the tiles' addresses, so no permute runs: the same results as
 * ra_shard_permute(RA_SEQ_TO_SHARDS) + the sweep + RA_SHARDS_TO_SEQ and
 * ra_lse_to_seq, bit for bit.  Fused sweep only (not with RA_FLAG_STEPWISE);
 * zigzag needs its chunk L / 2N to be a multiple of 128 (RA_ERR_UNSUPPORTED
 * otherwise).  There is no Ulysses split in this form (U = 1).            */
#define RA_FLAG_SEQ_ORDER 4u
/* Test hook for the timeout path: the first CTA of the fused sweep (or of
 * the first step of ra_ring_attn_fwd_stepwise_noalloc) never loads one key tile, so the waits that depend on it run out after about two
 * seconds; the kernel records RA_ERR_TIMEOUT in the status word, releases what
 * it holds and exits, and the outputs of that CTA are left unwritten.  Nothing
 * faults and the context stays usable.  Not for production use.              */
#define RA_FLAG_INJECT_STALL 0x80000000u

/* Smallest workspace any attention call accepts (the status word and padding). */
#define RA_WORKSPACE_MIN_BYTES 256u

/*
 * ra_shard_permute -- move tokens between the full sequence and the shard
 * stacks, and between the sequence-sharded and head-sharded Ulysses states.
 * Every op is a pure copy (bit-exact), one contiguous run of bytes per token.
 *
 * R ring ranks, U Ulysses ranks, P = U*R virtual ranks; global rank
 * p = u*R + r (row u, column r of the USP grid, [USP] §7.1).  U = 1 gives a
 * plain ring.
 *   RA_SEQ_TO_SHARDS: dst[u*R + r][b][s] = src[b][pos(r, u*L/P + s)], where
 *       pos is `layout` over R ranks of L/R tokens: ring rank r's token list,
 *       cut into U contiguous pieces ([USP] §7.2 input state [bs, L/N, H, d]).
 *   RA_ULYSSES_SEQ_TO_HEAD: the all-to-all of [USP] §5.1/§7.2 inside each
 *       Ulysses group (column r), as a local gather:
 *       dst[r][u'][b][u*Lp + s][hh] = src[u*R + r][b][s][u'*H/U + hh],
 *       Lp = L/P.  Block (r, u') is [B, L/R, H/U, d]: ring shard r of head
 *       group u', so dst viewed as [R, U*B, L/R, H/U, d] is a ring stack that
 *       one ra_ring_attn_fwd call sweeps.
 *   The _TO_SEQ / _HEAD_TO_SEQ ops are the exact inverses.
 * src, dst: device, non-overlapping; element size elem_bytes (1, 2, 4 or 8;
 * 2 for bf16, 4 for fp32).  Requires P | L, and for zigzag 2R | L; U | H for the Ulysses ops;
 * (H*d*elem_bytes) and ((H/U)*d*elem_bytes) multiples of 16.
 */
RA_API ra_status ra_shard_permute(const void *src, void *dst, int op, int layout,
                           int64_t B, int64_t L, int64_t H, int64_t d,
                           int R, int U, int elem_bytes, void *stream);

/*
 * ra_lse_to_seq -- put a ring call's LSE back in token order.
 * src: fp32 [R, U*B, H/U, L/R] (the LSE of a ring call on a head-sharded
 * stack; U = 1 is the plain [N, B, H, S]); dst: fp32 [B, H, L] with
 * dst[b][u*H/U + hh][pos(r, s)] = src[r][u*B + b][hh][s].  Bit-exact copy.
 */
RA_API ra_status ra_lse_to_seq(const float *src, float *dst, int layout, int64_t B, int64_t L,
                        int64_t H, int R, int U, void *stream);

/*
 * ra_block_attn_fwd -- one ring step: query shard q_rank against key/value
 * shard kv_rank ([USP] §3.3 "flash_attn_block", §6.2).
 * q, k, v: bf16 [B, S, H, d], the two ranks' shards.  Token positions come
 * from `layout` over N ranks of S tokens; with `causal` a query at position t
 * sees the keys at positions <= t ([USP] §3.4, [SPQ] engineering notes).
 * o: fp32 [B, S, H, d], the partial output normalised over the keys this
 * shard contributes; lse: fp32 [B, H, S], ln of the sum of exp(score) over
 * them.  A row that sees no key of this shard gets o = 0, lse = -inf.
 * scale <= 0 selects 1/sqrt(d).  d is 64 or 128; workspace: device, at least
 * RA_WORKSPACE_MIN_BYTES, zero-filled before its first use (status word).
 */
RA_API ra_status ra_block_attn_fwd(const void *q, const void *k, const void *v, float *o, float *lse,
                            int64_t B, int64_t S, int64_t H, int d, int N, int q_rank,
                            int kv_rank, int layout, int causal, float scale,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * ra_lse_merge -- fold partial result b into accumulator acc, in place
 * ([USP] §6.3):  lse = max(lse_a, lse_b) + ln(1 + exp(-|lse_a - lse_b|)),
 *                O   = O_a exp(lse_a - lse) + O_b exp(lse_b - lse).
 * `rows` rows of d fp32 values: row r of the accumulator's O starts at
 * o_acc + r * acc_row_stride and row r of b's at o_b + r * b_row_stride
 * (strides in floats, multiples of 4 and at least d, so O may be a strided
 * view, e.g. one head of a [.., S, H, d] tensor with stride H * d); their
 * LSEs are lse_acc[r] and lse_b[r] (fp32, contiguous).  O pointers 16-byte
 * aligned, LSE pointers 4-byte aligned.  -inf marks an empty partial: it gets
 * weight 0, and two empty partials stay (O = 0, lse = -inf).  d is a multiple
 * of 4, at most 256.  Rows must not overlap between acc and b.
 */
RA_API ra_status ra_lse_merge(float *o_acc, float *lse_acc, const float *o_b, const float *lse_b,
                              int64_t rows, int d, int64_t acc_row_stride, int64_t b_row_stride,
                              void *stream);

/*
 * ra_lse_merge_bshd -- the same merge over whole ring-call tensors:
 * o_acc, o_b fp32 [B, S, H, d]; lse_acc, lse_b fp32 [B, H, S] (the layouts
 * ra_block_attn_fwd writes).  Equivalent to B * H strided ra_lse_merge calls
 * (rows = S, strides H * d), in one launch.  Every pointer 16-byte aligned.
 */
RA_API ra_status ra_lse_merge_bshd(float *o_acc, float *lse_acc, const float *o_b, const float *lse_b,
                                   int64_t B, int64_t S, int64_t H, int d, void *stream);

/*
 * ra_ring_attn_fwd -- the whole ring sweep ([USP] §3.1-§3.3): for every rank
 * i and step s = 0..N-1, query shard i meets key/value shard (i - s) mod N
 * and the results are merged online ([USP] §3.2).  All N ranks run at once.
 * q, k, v: bf16 [N, B, S, H, d] shard stacks (S = L / N) in `layout`;
 * o: [N, B, S, H, d], fp32 by default (the fp32 accumulator itself), bf16
 * with RA_FLAG_O_BF16; lse: fp32 [N, B, H, S] (natural log).
 * Requires N | L, 2N | L for zigzag, d in {64, 128}.  scale <= 0 selects
 * 1/sqrt(d).  flags: any of RA_FLAG_STEPWISE, RA_FLAG_O_BF16, RA_FLAG_SEQ_ORDER
 * (which changes the q/k/v/o/lse layouts to token order, see there; and the
 * test hook RA_FLAG_INJECT_STALL, fused sweep only).  workspace:
 * device, ra_ring_attn_workspace_bytes() bytes, zero-filled before its first
 * use.
 */
RA_API ra_status ra_ring_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                           int64_t B, int64_t L, int64_t H, int d, int N, int layout,
                           int causal, float scale, unsigned flags,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * Grouped-query attention ([USP] §5.3: K and V carry fewer heads than Q).
 * The same calls with H_kv key/value heads: k and v are [.., H_kv, d]
 * instead of [.., H, d], and query head h attends with key/value head
 * h / (H / H_kv).  H_kv must divide H; H_kv = H is the plain call.  Every
 * other argument, layout and behaviour is that of ra_block_attn_fwd /
 * ra_ring_attn_fwd (the workspace size does not depend on H_kv).  For the
 * Ulysses permutes of K and V pass H_kv as H (U must divide H_kv).
 */
RA_API ra_status ra_block_attn_fwd_gqa(const void *q, const void *k, const void *v, float *o,
                                       float *lse, int64_t B, int64_t S, int64_t H, int64_t H_kv,
                                       int d, int N, int q_rank, int kv_rank, int layout,
                                       int causal, float scale, void *workspace,
                                       size_t workspace_bytes, void *stream);
RA_API ra_status ra_ring_attn_fwd_gqa(const void *q, const void *k, const void *v, void *o,
                                      float *lse, int64_t B, int64_t L, int64_t H, int64_t H_kv,
                                      int d, int N, int layout, int causal, float scale,
                                      unsigned flags, void *workspace, size_t workspace_bytes,
                                      void *stream);

/*
 * ra_ring_attn_fwd_varlen -- the ring sweep over packed variable-length
 * sequences ([USP] §6.2 runs a varlen kernel per ring step; §8 names variable
 * lengths as harder for the ring).  The n_seqs sequences are packed into one
 * stream of L tokens (B = 1): cu_seqlens (device, int32, n_seqs + 1 entries)
 * holds their boundaries, 0 = c_0 <= c_1 <= ... <= c_n = L (empty sequences
 * allowed).  The layout shards the packed stream by global position; a query
 * sees only keys of its own sequence (and, causal, not after it).  Boundaries
 * that break these rules give wrong masks but never an out-of-range access.
 * q [N, 1, S, H, d], k and v [N, 1, S, H_kv, d] (with RA_FLAG_SEQ_ORDER the
 * packed stream itself, [1, L, H, d] and [1, L, H_kv, d]); the rest as
 * ra_ring_attn_fwd_gqa.
 */
RA_API ra_status ra_ring_attn_fwd_varlen(const void *q, const void *k, const void *v, void *o,
                                         float *lse, const int32_t *cu_seqlens, int n_seqs,
                                         int64_t L, int64_t H, int64_t H_kv, int d, int N,
                                         int layout, int causal, float scale, unsigned flags,
                                         void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes ra_ring_attn_fwd needs for these arguments (0 on bad ones). */
RA_API size_t ra_ring_attn_workspace_bytes(int64_t B, int64_t L, int64_t H, int d, int N,
                                    unsigned flags);

/*
 * ra_ring_attn_fwd_stepwise_noalloc -- the RA_FLAG_STEPWISE sweep of
 * ra_ring_attn_fwd (fp32 O), for callers that cannot allocate device memory.
 * The pages have no counterpart: it exists for code that may not call
 * cudaMalloc or pass a workspace -- code running inside another framework's
 * memory pool or allocator callback, plugins handed only their inputs and
 * outputs, paths where cudaMalloc / cudaFree would synchronise the device.
 * Its scratch (one fp32 partial O and LSE plus a status word) is a fixed
 * 64 MiB array owned by the library, held on every GPU that loads this code
 * until the process exits.  A problem is accepted when
 *     256 + round256(B*L*H*d*4) + round256(B*L*H*4) <= 64 MiB
 * (round256: up to a multiple of 256 bytes), else RA_ERR_UNSUPPORTED.
 * Arguments, checks and layouts are those of ra_ring_attn_fwd with flags =
 * RA_FLAG_STEPWISE; o is fp32.  flags: 0, or the test hook
 * RA_FLAG_INJECT_STALL (the first step's launch withholds one key tile, so its
 * waits run out as described there).  It allocates nothing.  The first call
 * on each device looks up the array's device address (which loads this part
 * of the library on that device); make that first call before any stream
 * capture.  Every call on a device uses the same array: calls that may
 * overlap on the GPU (other streams, other threads) race on it and must be
 * serialised by the caller.  A wait that runs out is recorded in the array's
 * status word, which keeps it across calls until ra_noalloc_check_status()
 * reports and clears it.
 */
RA_API ra_status ra_ring_attn_fwd_stepwise_noalloc(const void *q, const void *k, const void *v,
                                                   float *o, float *lse, int64_t B, int64_t L,
                                                   int64_t H, int d, int N, int layout,
                                                   int causal, float scale, unsigned flags,
                                                   void *stream);

/*
 * ra_noalloc_check_status -- synchronise `stream`, read the status word of
 * the current device's scratch array, clear it, and return RA_ERR_TIMEOUT if
 * a kernel of ra_ring_attn_fwd_stepwise_noalloc gave up on a bounded wait
 * since the last check (its outputs are then incomplete), RA_ERR_ALIGNMENT
 * if one found its shared memory base unaligned, RA_OK otherwise.  It
 * allocates nothing.
 */
RA_API ra_status ra_noalloc_check_status(void *stream);

/*
 * ra_ring_attn_bwd -- gradients of ra_ring_attn_fwd.  The pages describe the
 * forward only; this is the plain derivative of softmax(Q K^T * scale) V
 * under the same masks (causal by position, optional packed sequences,
 * grouped key/value heads):
 *   dV = P^T dO,  dS = P * (dO V^T - D),  D = rowsum(dO * O),
 *   dQ = dS K * scale,  dK = dS^T Q * scale,
 * with P rebuilt from the forward's LSE.  Deterministic (no atomics): one
 * pass over key tiles for dK and dV, one over query tiles for dQ.
 * q: bf16 [N, B, S, H, d]; k, v: bf16 [N, B, S, H_kv, d]; o: fp32 forward
 * output [N, B, S, H, d]; dout: bf16 gradient of O, like q; lse: fp32
 * [N, B, H, S] from the forward.  dq: fp32 like q; dk, dv: fp32 like k.
 * cu_seqlens / n_seqs: packed sequences as in ra_ring_attn_fwd_varlen (B = 1),
 * or NULL / 0.  d in {64, 128}.  flags: 0 or RA_FLAG_SEQ_ORDER, with which
 * every tensor is in token order as in the forward of that flag (q, dout, o,
 * dq [B, L, H, d]; k, v, dk, dv [B, L, H_kv, d]; lse [B, H, L]), with the
 * same zigzag condition; the results equal the shard-stack call's, bit for
 * bit, in token order.  workspace: ra_ring_attn_bwd_workspace_bytes() bytes
 * (status word, D, and in token order a stack-order copy of lse),
 * zero-filled before its first use.
 */
RA_API ra_status ra_ring_attn_bwd(const void *q, const void *k, const void *v, const float *o,
                                  const void *dout, const float *lse, float *dq, float *dk,
                                  float *dv, const int32_t *cu_seqlens, int n_seqs, int64_t B,
                                  int64_t L, int64_t H, int64_t H_kv, int d, int N, int layout,
                                  int causal, float scale, unsigned flags, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* Workspace bytes ra_ring_attn_bwd needs (0 on bad arguments). */
RA_API size_t ra_ring_attn_bwd_workspace_bytes(int64_t B, int64_t L, int64_t H, int d, int N);

/*
 * ra_check_status -- synchronise `stream`, read the status word at the start
 * of `workspace`, clear it, and return RA_ERR_TIMEOUT if a kernel recorded a
 * timeout since the last check, RA_ERR_ALIGNMENT if a kernel found its
 * dynamic shared memory base not 1024-byte aligned (it then computed
 * nothing), RA_OK otherwise.
 */
RA_API ra_status ra_check_status(void *workspace, void *stream);

/* Message for the last non-OK status returned on this host thread. */
RA_API const char *ra_last_error(void);

/* Library version string. */
RA_API const char *ra_version(void);

/* ra_ring_step_pairs -- how many (query, key) pairs query shard q_rank and
 * key/value shard kv_rank have in common under `layout` over N ranks of S
 * tokens: S * S without the causal mask, else the pairs whose key position is
 * not after the query's ([USP] §3.4; the count the attention kernels' masks
 * give).  0 means a ring step with nothing to compute (contiguous, a later
 * rank's shard).  Host only, O(S); -1 on bad arguments. */
RA_API int64_t ra_ring_step_pairs(int layout, int64_t S, int N, int q_rank, int kv_rank, int causal);

/* ra_set_launch_chunk_budget -- set the launch-order chunk budget (see
 * "Launch order" above) to `bytes` for every later launch in the process;
 * bytes <= 0 restores the default of 48 MiB.  Returns the previous budget.
 * Host only; it never changes a result, only the order units run in. */
RA_API int64_t ra_set_launch_chunk_budget(int64_t bytes);

/* ra_launch_chunk_pairs -- how many (batch, head) pairs the attention kernels
 * interleave per chunk of their launch order (see "Launch order" above) when a
 * pair streams per_pair_bytes.  With B the budget (48 MiB unless
 * ra_set_launch_chunk_budget changed it): all pairs if they stream at most
 * 5/3 B together (one chunk: the whole launch runs heaviest units first);
 * otherwise the fewest chunks of at most B each, made near-equal
 * (ceil(pairs / n) pairs for n = ceil(pairs / floor(B / per_pair_bytes))), at
 * least 1.  Host only; launches nothing.  Returns 1 for per_pair_bytes <= 0
 * and pairs for pairs < 1. */
RA_API int64_t ra_launch_chunk_pairs(int64_t per_pair_bytes, int64_t pairs);

#ifdef __cplusplus
}
#endif
#endif /* RA_GB300_H */
