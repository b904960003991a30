// api.cu -- the C ABI (include/ra.h): argument checks, workspace layout and
// launch order.  Every check runs on the host before any CUDA call, so a
// rejected call touches neither the device nor the stream.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

#include "ra_internal.h"
#include "ra_positions.cuh"

namespace {

thread_local std::string g_last_error;

ra_status fail(ra_status st, const std::string &msg) {
    g_last_error = msg;
    return st;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_layout(int layout) {
    return layout == RA_CONTIGUOUS || layout == RA_STRIPED || layout == RA_ZIGZAG;
}

// Workspace layout: [0, 256) status word + reserved; then, for the stepwise
// sweep, the fp32 output accumulator (bf16 O only) and one fp32 partial (O
// and LSE), each starting on a 256-byte boundary.
constexpr size_t kHeader = RA_WORKSPACE_MIN_BYTES;

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct StepwiseLayout {
    size_t o_acc, o_part, lse_part, total;
};

// With an fp32 O the caller's O is the accumulator and needs no workspace copy.
StepwiseLayout stepwise_layout(int64_t B, int64_t L, int64_t H, int d, bool o_bf16) {
    const size_t n_o = (size_t)B * (size_t)L * (size_t)H * (size_t)d;  // N*B*S*H*d
    const size_t n_lse = (size_t)B * (size_t)L * (size_t)H;
    StepwiseLayout s;
    s.o_acc = kHeader;
    s.o_part = s.o_acc + (o_bf16 ? round256(n_o * 4) : 0);
    s.lse_part = s.o_part + round256(n_o * 4);
    s.total = s.lse_part + round256(n_lse * 4);
    return s;
}

ra_status check_attn_common(int64_t B, int64_t S, int64_t H, int d, int N, int layout, float scale) {
    if (B < 0 || S < 0 || H < 0) return fail(RA_ERR_SHAPE, "B, S and H must be non-negative");
    if (N < 1) return fail(RA_ERR_SHAPE, "N (ring degree) must be at least 1");
    if (!valid_layout(layout)) return fail(RA_ERR_INVALID_ARG, "layout must be RA_CONTIGUOUS, RA_STRIPED or RA_ZIGZAG");
    if (d != 64 && d != 128) return fail(RA_ERR_UNSUPPORTED, "head dimension d must be 64 or 128");
    if (std::isnan(scale) || std::isinf(scale)) return fail(RA_ERR_INVALID_ARG, "scale must be finite");
    if (layout == RA_ZIGZAG && (S % 2) != 0)
        return fail(RA_ERR_SHAPE, "zigzag needs an even shard length (2N | L)");
    if (S > (int64_t)1 << 30 || H > (int64_t)1 << 20 || B > (int64_t)1 << 20)
        return fail(RA_ERR_UNSUPPORTED, "B, S or H beyond the supported range");
    if ((int64_t)N * B > (int64_t)1 << 30)
        return fail(RA_ERR_UNSUPPORTED, "N * B beyond the supported range");
    if (S * H * d * 2 >= ((int64_t)1 << 40))
        return fail(RA_ERR_UNSUPPORTED, "one shard exceeds the 2^40-byte tensor-map stride limit");
    return RA_OK;
}

}  // namespace

ra_status ra::set_error(ra_status st, const char *msg) { return fail(st, msg); }

ra_status ra::check_attn_sizes(int64_t B, int64_t S, int64_t H, int d, int N, int layout, float scale) {
    return check_attn_common(B, S, H, d, N, layout, scale);
}

namespace {
constexpr int64_t kDefaultChunkBytes = (int64_t)48 << 20;
std::atomic<int64_t> g_chunk_bytes{kDefaultChunkBytes};
}  // namespace

int64_t ra::l2_chunk_bytes() { return g_chunk_bytes.load(std::memory_order_relaxed); }

extern "C" {

const char *ra_last_error(void) { return g_last_error.c_str(); }

const char *ra_version(void) { return "ra_gb300 0.1 (sm_103a)"; }

int64_t ra_set_launch_chunk_budget(int64_t bytes) {
    const int64_t prev = g_chunk_bytes.load();
    g_chunk_bytes.store(bytes > 0 ? bytes : kDefaultChunkBytes);
    return prev;
}

int64_t ra_ring_step_pairs(int layout, int64_t S, int N, int q_rank, int kv_rank, int causal) {
    if (!valid_layout(layout) || N < 1 || S < 0 || q_rank < 0 || q_rank >= N || kv_rank < 0 || kv_rank >= N)
        return -1;
    if (layout == RA_ZIGZAG && (S % 2)) return -1;
    if (S > ((int64_t)1 << 30)) return -1;
    if (!causal) return S * S;
    int64_t pairs = 0;
    for (int64_t a = 0; a < S; ++a)
        pairs += ra::keys_upto(layout, kv_rank, ra::token_pos(layout, q_rank, a, N, S), N, S);
    return pairs;
}

int64_t ra_launch_chunk_pairs(int64_t per_pair_bytes, int64_t pairs) {
    if (pairs < 1) return pairs;
    if (per_pair_bytes <= 0) return 1;
    const int64_t budget = ra::l2_chunk_bytes();
    // every pair's operands fit in L2 together: one chunk, heaviest units first overall
    if (per_pair_bytes <= (budget + budget * 2 / 3) / pairs) return pairs;
    int64_t fit = budget / per_pair_bytes;
    if (fit < 1) fit = 1;
    if (fit >= pairs) return pairs;
    // as many chunks as the budget needs, of near-equal size
    const int64_t n = (pairs + fit - 1) / fit;
    return (pairs + n - 1) / n;
}

ra_status ra_shard_permute(const void *src, void *dst, int op, int layout, int64_t B, int64_t L,
                           int64_t H, int64_t d, int R, int U, int elem_bytes, void *stream) {
    if (op < RA_SEQ_TO_SHARDS || op > RA_ULYSSES_HEAD_TO_SEQ)
        return fail(RA_ERR_INVALID_ARG, "unknown permute op");
    if (!valid_layout(layout)) return fail(RA_ERR_INVALID_ARG, "unknown layout");
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
        return fail(RA_ERR_INVALID_ARG, "elem_bytes must be 1, 2, 4 or 8");
    if (B < 0 || L < 0 || H < 0 || d < 0) return fail(RA_ERR_SHAPE, "sizes must be non-negative");
    if (R < 1 || U < 1) return fail(RA_ERR_SHAPE, "R and U must be at least 1");
    const int64_t P = (int64_t)R * U;
    if (L % P) return fail(RA_ERR_SHAPE, "U*R must divide L");
    if (layout == RA_ZIGZAG && (L % (2 * (int64_t)R)))
        return fail(RA_ERR_SHAPE, "zigzag needs 2R | L");
    const bool ulysses = op == RA_ULYSSES_SEQ_TO_HEAD || op == RA_ULYSSES_HEAD_TO_SEQ;
    if (ulysses && (H % U)) return fail(RA_ERR_SHAPE, "U must divide H");
    if ((H * d * elem_bytes) % 16)
        return fail(RA_ERR_ALIGNMENT, "a token's H*d*elem_bytes must be a multiple of 16 bytes");
    if (ulysses && (((H / U) * d * elem_bytes) % 16))
        return fail(RA_ERR_ALIGNMENT, "a head slice (H/U)*d*elem_bytes must be a multiple of 16 bytes");
    if (B * L * H * d == 0) return RA_OK;
    if (!src || !dst) return fail(RA_ERR_INVALID_ARG, "null src or dst");
    if (!aligned16(src) || !aligned16(dst)) return fail(RA_ERR_ALIGNMENT, "src and dst must be 16-byte aligned");
    if (src == dst) return fail(RA_ERR_INVALID_ARG, "src and dst must not be the same buffer");
    const char *err = nullptr;
    ra_status st = ra::launch_permute(src, dst, op, layout, B, L, H, d, R, U, elem_bytes,
                                      static_cast<cudaStream_t>(stream), &err);
    return st == RA_OK ? st : fail(st, err ? err : "permute launch failed");
}

ra_status ra_lse_to_seq(const float *src, float *dst, int layout, int64_t B, int64_t L, int64_t H,
                        int R, int U, void *stream) {
    if (!valid_layout(layout)) return fail(RA_ERR_INVALID_ARG, "unknown layout");
    if (B < 0 || L < 0 || H < 0) return fail(RA_ERR_SHAPE, "sizes must be non-negative");
    if (R < 1 || U < 1) return fail(RA_ERR_SHAPE, "R and U must be at least 1");
    if (L % R) return fail(RA_ERR_SHAPE, "R must divide L");
    if (layout == RA_ZIGZAG && (L % (2 * (int64_t)R))) return fail(RA_ERR_SHAPE, "zigzag needs 2R | L");
    if (H % U) return fail(RA_ERR_SHAPE, "U must divide H");
    if (B * L * H == 0) return RA_OK;
    if (!src || !dst) return fail(RA_ERR_INVALID_ARG, "null src or dst");
    if (!aligned16(src) || !aligned16(dst)) return fail(RA_ERR_ALIGNMENT, "src and dst must be 16-byte aligned");
    const char *err = nullptr;
    ra_status st = ra::launch_lse_to_seq(src, dst, layout, B, L, H, R, U,
                                         static_cast<cudaStream_t>(stream), &err);
    return st == RA_OK ? st : fail(st, err ? err : "lse_to_seq launch failed");
}

}  // extern "C"

namespace {

ra_status check_kv_heads(int64_t H, int64_t H_kv) {
    if (H_kv < 1 || H_kv > H || H % H_kv)
        return fail(RA_ERR_SHAPE, "the key/value head count must divide the query head count");
    return RA_OK;
}

ra_status block_attn(const void *q, const void *k, const void *v, float *o, float *lse, int64_t B,
                     int64_t S, int64_t H, int64_t H_kv, int d, int N, int q_rank, int kv_rank,
                     int layout, int causal, float scale, void *workspace, size_t workspace_bytes,
                     void *stream) {
    ra_status st = check_attn_common(B, S, H, d, N, layout, scale);
    if (st != RA_OK) return st;
    if (H > 0 && (st = check_kv_heads(H, H_kv)) != RA_OK) return st;
    if (q_rank < 0 || q_rank >= N || kv_rank < 0 || kv_rank >= N)
        return fail(RA_ERR_INVALID_ARG, "q_rank and kv_rank must lie in [0, N)");
    if (B * S * H == 0) return RA_OK;
    if (!q || !k || !v || !o || !lse || !workspace) return fail(RA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(workspace))
        return fail(RA_ERR_ALIGNMENT, "every pointer must be 16-byte aligned");
    if (workspace_bytes < RA_WORKSPACE_MIN_BYTES)
        return fail(RA_ERR_INVALID_ARG, "workspace smaller than RA_WORKSPACE_MIN_BYTES");
    ra::AttnLaunch a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    a.status = static_cast<unsigned *>(workspace);
    a.B = B;
    a.S = S;
    a.H = H;
    a.H_kv = H_kv;
    a.d = d;
    a.N = N;
    a.layout = layout;
    a.causal = causal;
    a.scale = scale;
    a.ring = false;
    a.q_rank = q_rank;
    a.kv_rank = kv_rank;
    a.ring_step = -1;
    a.out_f32 = true;
    const char *err = nullptr;
    st = ra::launch_attention(a, static_cast<cudaStream_t>(stream), &err);
    return st == RA_OK ? st : fail(st, err ? err : "attention launch failed");
}

}  // namespace

extern "C" {

ra_status ra_block_attn_fwd(const void *q, const void *k, const void *v, float *o, float *lse,
                            int64_t B, int64_t S, int64_t H, int d, int N, int q_rank, int kv_rank,
                            int layout, int causal, float scale, void *workspace,
                            size_t workspace_bytes, void *stream) {
    return block_attn(q, k, v, o, lse, B, S, H, H, d, N, q_rank, kv_rank, layout, causal, scale,
                      workspace, workspace_bytes, stream);
}

ra_status ra_block_attn_fwd_gqa(const void *q, const void *k, const void *v, float *o, float *lse,
                                int64_t B, int64_t S, int64_t H, int64_t H_kv, int d, int N,
                                int q_rank, int kv_rank, int layout, int causal, float scale,
                                void *workspace, size_t workspace_bytes, void *stream) {
    return block_attn(q, k, v, o, lse, B, S, H, H_kv, d, N, q_rank, kv_rank, layout, causal, scale,
                      workspace, workspace_bytes, stream);
}

ra_status ra_lse_merge(float *o_acc, float *lse_acc, const float *o_b, const float *lse_b, int64_t rows,
                       int d, int64_t acc_row_stride, int64_t b_row_stride, void *stream) {
    if (rows < 0 || d < 0) return fail(RA_ERR_SHAPE, "rows and d must be non-negative");
    if (d % 4 || d > 256) return fail(RA_ERR_UNSUPPORTED, "d must be a multiple of 4, at most 256");
    if (rows == 0 || d == 0) return RA_OK;
    if (acc_row_stride < d || b_row_stride < d)
        return fail(RA_ERR_SHAPE, "a row stride is smaller than d: rows would overlap");
    if (acc_row_stride % 4 || b_row_stride % 4)
        return fail(RA_ERR_ALIGNMENT, "row strides must be multiples of 4 floats (16 bytes)");
    if (rows > ((int64_t)1 << 40) / acc_row_stride || rows > ((int64_t)1 << 40) / b_row_stride)
        return fail(RA_ERR_UNSUPPORTED, "rows * row stride beyond the supported range");
    if (!o_acc || !lse_acc || !o_b || !lse_b) return fail(RA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(o_acc) || !aligned16(o_b))
        return fail(RA_ERR_ALIGNMENT, "the O pointers must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(lse_acc) & 3u) || (reinterpret_cast<uintptr_t>(lse_b) & 3u))
        return fail(RA_ERR_ALIGNMENT, "the LSE pointers must be 4-byte aligned");
    const char *err = nullptr;
    ra_status st = ra::launch_lse_merge_rows(o_acc, lse_acc, o_b, lse_b, rows, d, acc_row_stride, b_row_stride,
                                             static_cast<cudaStream_t>(stream), &err);
    return st == RA_OK ? st : fail(st, err ? err : "merge launch failed");
}

ra_status ra_lse_merge_bshd(float *o_acc, float *lse_acc, const float *o_b, const float *lse_b, int64_t B,
                            int64_t S, int64_t H, int d, void *stream) {
    if (B < 0 || S < 0 || H < 0 || d < 0) return fail(RA_ERR_SHAPE, "sizes must be non-negative");
    if (d % 4 || d > 256) return fail(RA_ERR_UNSUPPORTED, "d must be a multiple of 4, at most 256");
    if (B * S * H * d == 0) return RA_OK;
    if (B > ((int64_t)1 << 20) || H > ((int64_t)1 << 20) || S > ((int64_t)1 << 30) ||
        B * S * H * d > ((int64_t)1 << 40))
        return fail(RA_ERR_UNSUPPORTED, "B, S, H beyond the supported range");
    if (!o_acc || !lse_acc || !o_b || !lse_b) return fail(RA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(o_acc) || !aligned16(lse_acc) || !aligned16(o_b) || !aligned16(lse_b))
        return fail(RA_ERR_ALIGNMENT, "every pointer must be 16-byte aligned");
    const char *err = nullptr;
    ra_status st = ra::launch_lse_merge(o_acc, lse_acc, o_b, lse_b, B, S, H, d,
                                        static_cast<cudaStream_t>(stream), &err);
    return st == RA_OK ? st : fail(st, err ? err : "merge launch failed");
}

size_t ra_ring_attn_workspace_bytes(int64_t B, int64_t L, int64_t H, int d, int N, unsigned flags) {
    if (B < 0 || L < 0 || H < 0 || N < 1 || (d != 64 && d != 128)) return 0;
    if (flags & ~(RA_FLAG_STEPWISE | RA_FLAG_O_BF16 | RA_FLAG_SEQ_ORDER | RA_FLAG_INJECT_STALL)) return 0;
    if ((flags & RA_FLAG_SEQ_ORDER) && (flags & RA_FLAG_STEPWISE)) return 0;
    if (flags & RA_FLAG_STEPWISE) return stepwise_layout(B, L, H, d, (flags & RA_FLAG_O_BF16) != 0).total;
    return kHeader;
}

}  // extern "C"

namespace {

ra_status ring_attn(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                    int64_t L, int64_t H, int64_t H_kv, int d, int N, int layout, int causal,
                    float scale, unsigned flags, void *workspace, size_t workspace_bytes,
                    void *stream, const int *cu_seqlens = nullptr, int n_seqs = 0) {
    if (flags & ~(RA_FLAG_STEPWISE | RA_FLAG_O_BF16 | RA_FLAG_SEQ_ORDER | RA_FLAG_INJECT_STALL))
        return fail(RA_ERR_INVALID_ARG, "unknown flag bits");
    if ((flags & RA_FLAG_INJECT_STALL) && (flags & RA_FLAG_STEPWISE))
        return fail(RA_ERR_INVALID_ARG, "RA_FLAG_INJECT_STALL applies to the fused sweep only");
    if ((flags & RA_FLAG_SEQ_ORDER) && (flags & RA_FLAG_STEPWISE))
        return fail(RA_ERR_INVALID_ARG, "RA_FLAG_SEQ_ORDER applies to the fused sweep only");
    const bool o_bf16 = (flags & RA_FLAG_O_BF16) != 0;
    if (N < 1) return fail(RA_ERR_SHAPE, "N (ring degree) must be at least 1");
    if (L < 0) return fail(RA_ERR_SHAPE, "L must be non-negative");
    if (L % N) return fail(RA_ERR_SHAPE, "N must divide L");
    if (layout == RA_ZIGZAG && (L % (2 * (int64_t)N))) return fail(RA_ERR_SHAPE, "zigzag needs 2N | L");
    const int64_t S = L / N;
    if ((flags & RA_FLAG_SEQ_ORDER) && layout == RA_ZIGZAG && (S / 2) % 128)
        return fail(RA_ERR_UNSUPPORTED, "RA_FLAG_SEQ_ORDER with zigzag needs L / 2N to be a multiple of 128");
    ra_status st = check_attn_common(B, S, H, d, N, layout, scale);
    if (st != RA_OK) return st;
    if (H > 0 && (st = check_kv_heads(H, H_kv)) != RA_OK) return st;
    if (B * L * H == 0) return RA_OK;
    if (!q || !k || !v || !o || !lse || !workspace) return fail(RA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(workspace))
        return fail(RA_ERR_ALIGNMENT, "every pointer must be 16-byte aligned");
    const size_t need = ra_ring_attn_workspace_bytes(B, L, H, d, N, flags);
    if (workspace_bytes < need)
        return fail(RA_ERR_INVALID_ARG, "workspace smaller than ra_ring_attn_workspace_bytes()");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const char *err = nullptr;
    ra::AttnLaunch a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.lse = lse;
    a.status = static_cast<unsigned *>(workspace);
    a.B = B;
    a.S = S;
    a.H = H;
    a.H_kv = H_kv;
    a.d = d;
    a.N = N;
    a.layout = layout;
    a.causal = causal;
    a.scale = scale;
    a.ring = true;
    a.cu_seqlens = cu_seqlens;
    a.n_seqs = n_seqs;
    a.seq_order = (flags & RA_FLAG_SEQ_ORDER) != 0;
    if (!(flags & RA_FLAG_STEPWISE)) {
        a.o = o;
        a.ring_step = -1;
        a.out_f32 = !o_bf16;
        a.inject_stall = (flags & RA_FLAG_INJECT_STALL) != 0;
        st = ra::launch_attention(a, s, &err);
        return st == RA_OK ? st : fail(st, err ? err : "attention launch failed");
    }
    // Stepwise: the pages' per-step structure -- at step s every rank meets
    // KV shard (i - s) mod N, then the partial result is merged in.
    StepwiseLayout wl = stepwise_layout(B, L, H, d, o_bf16);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *o_acc = o_bf16 ? reinterpret_cast<float *>(ws + wl.o_acc) : static_cast<float *>(o);
    float *o_part = reinterpret_cast<float *>(ws + wl.o_part);
    float *lse_part = reinterpret_cast<float *>(ws + wl.lse_part);
    a.out_f32 = true;
    for (int step = 0; step < N; ++step) {
        a.ring_step = step;
        a.o = step == 0 ? o_acc : o_part;
        a.lse = step == 0 ? lse : lse_part;
        st = ra::launch_attention(a, s, &err);
        if (st != RA_OK) return fail(st, err ? err : "attention launch failed");
        if (step > 0) {
            st = ra::launch_lse_merge(o_acc, lse, o_part, lse_part, (int64_t)N * B, S, H, d, s, &err);
            if (st != RA_OK) return fail(st, err ? err : "merge launch failed");
        }
    }
    if (!o_bf16) return RA_OK;
    st = ra::launch_f32_to_bf16(o_acc, o, (int64_t)N * B * S * H * d, s, &err);
    return st == RA_OK ? st : fail(st, err ? err : "conversion launch failed");
}

}  // namespace

extern "C" {

ra_status ra_ring_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                           int64_t B, int64_t L, int64_t H, int d, int N, int layout, int causal,
                           float scale, unsigned flags, void *workspace, size_t workspace_bytes,
                           void *stream) {
    return ring_attn(q, k, v, o, lse, B, L, H, H, d, N, layout, causal, scale, flags, workspace,
                     workspace_bytes, stream);
}

ra_status ra_ring_attn_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
                               int64_t B, int64_t L, int64_t H, int64_t H_kv, int d, int N,
                               int layout, int causal, float scale, unsigned flags,
                               void *workspace, size_t workspace_bytes, void *stream) {
    return ring_attn(q, k, v, o, lse, B, L, H, H_kv, d, N, layout, causal, scale, flags, workspace,
                     workspace_bytes, stream);
}

ra_status ra_ring_attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                                  const int32_t *cu_seqlens, int n_seqs, int64_t L, int64_t H,
                                  int64_t H_kv, int d, int N, int layout, int causal, float scale,
                                  unsigned flags, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    if (n_seqs < 1) return fail(RA_ERR_SHAPE, "n_seqs must be at least 1");
    if (L > 0 && (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)))
        return fail(RA_ERR_INVALID_ARG, "cu_seqlens must be a 4-byte-aligned device pointer");
    if (L >= ((int64_t)1 << 31)) return fail(RA_ERR_UNSUPPORTED, "packed length must fit in int32");
    return ring_attn(q, k, v, o, lse, 1, L, H, H_kv, d, N, layout, causal, scale, flags, workspace,
                     workspace_bytes, stream, cu_seqlens, n_seqs);
}

size_t ra_ring_attn_bwd_workspace_bytes(int64_t B, int64_t L, int64_t H, int d, int N) {
    if (B < 0 || L < 0 || H < 0 || N < 1 || (d != 64 && d != 128)) return 0;
    // the status word, D, and the stack-order copy of lse a token-order call makes
    return kHeader + 2 * round256((size_t)B * (size_t)L * (size_t)H * 4);
}

ra_status ra_ring_attn_bwd(const void *q, const void *k, const void *v, const float *o,
                           const void *dout, const float *lse, float *dq, float *dk, float *dv,
                           const int32_t *cu_seqlens, int n_seqs, int64_t B, int64_t L, int64_t H,
                           int64_t H_kv, int d, int N, int layout, int causal, float scale,
                           unsigned flags, void *workspace, size_t workspace_bytes, void *stream) {
    if (flags & ~RA_FLAG_SEQ_ORDER) return fail(RA_ERR_INVALID_ARG, "unknown flag bits");
    if (N < 1) return fail(RA_ERR_SHAPE, "N (ring degree) must be at least 1");
    if (L < 0) return fail(RA_ERR_SHAPE, "L must be non-negative");
    if (L % N) return fail(RA_ERR_SHAPE, "N must divide L");
    if (layout == RA_ZIGZAG && (L % (2 * (int64_t)N))) return fail(RA_ERR_SHAPE, "zigzag needs 2N | L");
    const int64_t S = L / N;
    if ((flags & RA_FLAG_SEQ_ORDER) && layout == RA_ZIGZAG && (S / 2) % 128)
        return fail(RA_ERR_UNSUPPORTED, "RA_FLAG_SEQ_ORDER with zigzag needs L / 2N to be a multiple of 128");
    ra_status st = check_attn_common(B, S, H, d, N, layout, scale);
    if (st != RA_OK) return st;
    if (H > 0 && (st = check_kv_heads(H, H_kv)) != RA_OK) return st;
    if (cu_seqlens) {
        if (B != 1) return fail(RA_ERR_SHAPE, "packed sequences need B = 1");
        if (n_seqs < 1) return fail(RA_ERR_SHAPE, "n_seqs must be at least 1");
        if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)
            return fail(RA_ERR_ALIGNMENT, "cu_seqlens must be 4-byte aligned");
    }
    if (B * L * H == 0) return RA_OK;
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
        return fail(RA_ERR_INVALID_ARG, "null pointer argument");
    const void *ptrs[] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(RA_ERR_ALIGNMENT, "every tensor pointer must be 16-byte aligned");
    if (workspace_bytes < ra_ring_attn_bwd_workspace_bytes(B, L, H, d, N))
        return fail(RA_ERR_INVALID_ARG, "workspace smaller than ra_ring_attn_bwd_workspace_bytes()");
    ra::BwdLaunch a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.dout = dout;
    a.o = o;
    a.lse = lse;
    a.dvec = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kHeader);
    a.lse_stack = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kHeader +
                                            round256((size_t)B * (size_t)L * (size_t)H * 4));
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.status = static_cast<unsigned *>(workspace);
    a.cu_seqlens = cu_seqlens;
    a.n_seqs = n_seqs;
    a.B = B;
    a.S = S;
    a.H = H;
    a.H_kv = H_kv;
    a.seq_order = (flags & RA_FLAG_SEQ_ORDER) != 0;
    a.d = d;
    a.N = N;
    a.layout = layout;
    a.causal = causal;
    a.scale = scale;
    const char *err = nullptr;
    st = ra::launch_attention_bwd(a, static_cast<cudaStream_t>(stream), &err);
    return st == RA_OK ? st : fail(st, err ? err : "backward launch failed");
}

ra_status ra_check_status(void *workspace, void *stream) {
    if (!workspace) return fail(RA_ERR_INVALID_ARG, "null workspace");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return fail(RA_ERR_CUDA, "cudaStreamSynchronize failed");
    if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail(RA_ERR_CUDA, "reading the status word failed");
    if (word) {
        const unsigned zero = 0;
        if (cudaMemcpy(workspace, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return fail(RA_ERR_CUDA, "clearing the status word failed");
        if (word & ra::RA_DEV_TIMEOUT_BIT)
            return fail(RA_ERR_TIMEOUT, "a kernel gave up on a bounded wait (status word set)");
        if (word & ra::RA_DEV_SMEM_ALIGN_BIT)
            return fail(RA_ERR_ALIGNMENT, "a kernel found its dynamic shared memory base not 1024-byte aligned");
    }
    return RA_OK;
}

}  // extern "C"
