// ra_internal.h -- launchers shared between the C-ABI layer and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ra.h"

namespace ra {

// Bits of the device status word (first 4 bytes of every workspace).
constexpr unsigned RA_DEV_TIMEOUT_BIT = 1u;
// A kernel that lays out its shared memory from a 1024-byte-aligned dynamic
// base found the base unaligned, and returned before touching it.
constexpr unsigned RA_DEV_SMEM_ALIGN_BIT = 2u;

// One attention launch: every query unit of `num_q_ranks` ranks sweeps its
// key/value shards.  Ring mode: q/k/v are [N, B, S, H, d] stacks, each query
// rank i visits ranks (i - s) mod N for s = 0..N-1.  Block mode: q is the
// [B, S, H, d] shard of q_rank, k/v that of kv_rank, one step.
struct AttnLaunch {
    const void *q, *k, *v;
    void *o;            // bf16 (ring) or fp32 (block)
    float *lse;
    unsigned *status;   // device status word
    int64_t B, S, H;
    int64_t H_kv;         // key/value heads (grouped-query attention); 0 means H
    int d, N, layout, causal;
    float scale;
    bool ring;
    int q_rank, kv_rank;  // block mode only
    int ring_step;        // ring mode: -1 sweeps all N steps; s >= 0 runs step s only
    bool out_f32;
    bool inject_stall;    // test hook, see RA_FLAG_INJECT_STALL
    const int *cu_seqlens;  // packed sequences (device, n_seqs + 1 boundaries), or null
    int n_seqs;
    bool seq_order;       // ring mode: q/k/v/o [B, L, H, d] and LSE [B, H, L] in sequence order
};

ra_status launch_attention(const AttnLaunch &a, cudaStream_t stream, const char **err);

// Bytes of streamed operands per chunk of (batch, head) pairs whose units a
// launch interleaves heaviest first (decode_unit): 48 MiB, or what
// ra_set_launch_chunk_budget last set.
int64_t l2_chunk_bytes();

// Pairs per chunk for `per_pair` streamed bytes each, between 1 and `pairs`
// (ra_launch_chunk_pairs).
inline int chunk_pairs(int64_t per_pair, int64_t pairs) {
    return (int)ra_launch_chunk_pairs(per_pair, pairs);
}

// One backward: D = rowsum(dO * O), then the dK / dV pass and the dQ pass.
// q, dout: bf16 [N, B, S, H, d]; k, v: bf16 [N, B, S, H_kv, d]; o: fp32
// [N, B, S, H, d]; lse, dvec: fp32 [N, B, H, S]; dq: fp32 like q; dk, dv:
// fp32 like k.
struct BwdLaunch {
    const void *q, *k, *v, *dout;
    const float *o, *lse;
    float *dvec;
    float *dq, *dk, *dv;
    unsigned *status;
    const int *cu_seqlens;
    int n_seqs;
    int64_t B, S, H, H_kv;
    int d, N, layout, causal;
    float scale;
    bool seq_order;       // q/k/v/o/dout/dq/dk/dv [B, L, ., d] and lse [B, H, L] in token order
    float *lse_stack;     // token order: workspace for the [N, B, H, S] copy of lse
};

ra_status launch_attention_bwd(const BwdLaunch &a, cudaStream_t stream, const char **err);

ra_status launch_permute(const void *src, void *dst, int op, int layout, int64_t B, int64_t L,
                         int64_t H, int64_t d, int R, int U, int elem_bytes, cudaStream_t stream,
                         const char **err);

ra_status launch_lse_to_seq(const float *src, float *dst, int layout, int64_t B, int64_t L,
                            int64_t H, int R, int U, cudaStream_t stream, const char **err);

// O [B, S, H, d] and LSE [B, H, S] (the ring calls' tensors)
ra_status launch_lse_merge(float *o_acc, float *lse_acc, const float *o_b, const float *lse_b,
                           int64_t B, int64_t S, int64_t H, int d, cudaStream_t stream,
                           const char **err);
// `rows` rows: O row r at o + r * row_stride (floats), its LSE at lse[r]
ra_status launch_lse_merge_rows(float *o_acc, float *lse_acc, const float *o_b, const float *lse_b,
                                int64_t rows, int d, int64_t acc_row_stride, int64_t b_row_stride,
                                cudaStream_t stream, const char **err);

// fp32 -> bf16 copy of n elements (n a multiple of 4): the stepwise ring finish
ra_status launch_f32_to_bf16(const float *src, void *dst, int64_t n, cudaStream_t stream,
                             const char **err);

// The 4-D view of a [..., cols] tensor that the attention kernels' TMA maps
// use (tile_coords gives a tile's coordinates in it): the columns, then three
// outer extents n[] with their element strides st[]; rows are outer dimension
// row_dim (0 or 1).  Shard stacks [stacks, B, S, cols]; in token order
// ([B, L, cols], L = N*S) the layout's view: contiguous [B, N, S], striped
// [B, S, N] (position s*N + r), zigzag [B, 2N, S/2].
struct TileView {
    int64_t n[3], st[3];
    int row_dim;
};
inline TileView tile_view(bool seq_order, int layout, int64_t S, int64_t B, int64_t N, int64_t stacks,
                          int64_t cols) {
    TileView v;
    v.row_dim = 0;
    if (!seq_order) {
        v.n[0] = S, v.n[1] = B, v.n[2] = stacks;
        v.st[0] = cols, v.st[1] = S * cols, v.st[2] = B * S * cols;
    } else if (layout == RA_STRIPED) {
        v.n[0] = N, v.n[1] = S, v.n[2] = B;
        v.st[0] = cols, v.st[1] = N * cols, v.st[2] = N * S * cols;
        v.row_dim = 1;
    } else if (layout == RA_ZIGZAG) {
        const int64_t C = S / 2;
        v.n[0] = C, v.n[1] = 2 * N, v.n[2] = B;
        v.st[0] = cols, v.st[1] = C * cols, v.st[2] = N * S * cols;
    } else {
        v.n[0] = S, v.n[1] = N, v.n[2] = B;
        v.st[0] = cols, v.st[1] = S * cols, v.st[2] = N * S * cols;
    }
    return v;
}

// Record `msg` as this host thread's ra_last_error() text and return `st`.
ra_status set_error(ra_status st, const char *msg);

// The host-side range checks every attention entry point applies to a ring or
// block problem of shard length S (the sizes the kernels index with 32-bit
// ints and the tensor maps' stride limit); RA_OK or the failing status, with
// the message recorded.
ra_status check_attn_sizes(int64_t B, int64_t S, int64_t H, int d, int N, int layout, float scale);

}  // namespace ra
