// permute.cu -- token moves between the full sequence, the ring shard stacks
// and the Ulysses head-sharded state, plus the LSE un-shard.  Pure copies.
//
// A token's [H, d] (or its [H/U, d] head slice) is one contiguous run of
// bytes ("slab") in both source and destination, so every op is a gather
// or scatter of slabs.  A warp moves one slab at a time with 16-byte loads
// and stores (coalesced: consecutive lanes take consecutive vectors).  The
// grid is a multiple of the SM count and loops over the slabs.
//
// Index formulas ("From Ring Attention to DeepSpeed Ulysses to USP",
// jsqmd.com/news/734632): §4 contiguous / striped split, §6.1 zigzag split,
// §5.1 and §7.2 the Ulysses all-to-all (scatter heads, gather sequence),
// §7.1 the USP grid numbering p = u*R + r.
#include "ra_internal.h"

namespace ra {

__device__ __forceinline__ int64_t layout_pos(int layout, int64_t r, int64_t s, int64_t N, int64_t S) {
    if (layout == RA_CONTIGUOUS) return r * S + s;
    if (layout == RA_STRIPED) return s * N + r;
    const int64_t C = S >> 1;
    return s < C ? r * C + s : (2 * N - 1 - r) * C + (s - C);
}

// Inverse of layout_pos: global token t -> (rank, local index).
__device__ __forceinline__ void layout_inv(int layout, int64_t t, int64_t N, int64_t S, int64_t &r,
                                           int64_t &s) {
    if (layout == RA_CONTIGUOUS) {
        r = t / S;
        s = t - r * S;
    } else if (layout == RA_STRIPED) {
        s = t / N;
        r = t - s * N;
    } else {
        const int64_t C = S >> 1;
        const int64_t c = t / C;
        const int64_t off = t - c * C;
        if (c < N) {
            r = c;
            s = off;
        } else {
            r = 2 * N - 1 - c;
            s = C + off;
        }
    }
}

struct PermArgs {
    const uint8_t *src;
    uint8_t *dst;
    int op, layout;
    int64_t B, L, R, U, Lp;   // Lp = L / (U*R)
    int64_t slab_vecs;        // 16-byte vectors per slab
    int64_t total_vecs;
    int64_t seq_slab_vecs;    // vectors per full-token [H, d] run (Ulysses ops)
};

// Byte offsets (in 16-byte vectors) of one slab copy: its place in the shard
// / head-sharded stack and its place on the other side.
__device__ __forceinline__ void slab_ends(const PermArgs &a, int64_t slab, int64_t &shard_vec,
                                          int64_t &other_vec) {
    if (a.op == RA_SEQ_TO_SHARDS || a.op == RA_SHARDS_TO_SEQ) {
        // slab indexes the shard stack [P, B, Lp]
        const int64_t s = slab % a.Lp;
        const int64_t rest = slab / a.Lp;
        const int64_t b = rest % a.B;
        const int64_t p = rest / a.B;
        const int64_t u = p / a.R, r = p - u * a.R;
        const int64_t t = layout_pos(a.layout, r, u * a.Lp + s, a.R, a.L / a.R);
        shard_vec = slab * a.slab_vecs;
        other_vec = (b * a.L + t) * a.slab_vecs;
    } else {
        // slab indexes the head-sharded state [R, U(head group), B, U(member), Lp]
        int64_t rest = slab;
        const int64_t s = rest % a.Lp;
        rest /= a.Lp;
        const int64_t u = rest % a.U;
        rest /= a.U;
        const int64_t b = rest % a.B;
        rest /= a.B;
        const int64_t up = rest % a.U;
        const int64_t r = rest / a.U;
        const int64_t tok = ((u * a.R + r) * a.B + b) * a.Lp + s;   // seq-sharded token slab
        shard_vec = slab * a.slab_vecs;
        other_vec = tok * a.seq_slab_vecs + up * a.slab_vecs;
    }
}

// One warp per slab: the index arithmetic runs once per slab, then the lanes
// stream the slab with 16-byte loads, up to four in flight per lane.
__global__ void __launch_bounds__(256) permute_kernel(const PermArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t n_slabs = a.total_vecs / a.slab_vecs;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.src);
    uint4 *dst = reinterpret_cast<uint4 *>(a.dst);
    const bool gather = a.op == RA_SEQ_TO_SHARDS || a.op == RA_ULYSSES_SEQ_TO_HEAD;
    for (int64_t slab = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); slab < n_slabs;
         slab += warps) {
        int64_t shard_vec, other_vec;
        slab_ends(a, slab, shard_vec, other_vec);
        const uint4 *from = src + (gather ? other_vec : shard_vec);
        uint4 *to = dst + (gather ? shard_vec : other_vec);
        const int n = (int)a.slab_vecs;
        int i = lane;
        for (; i + 96 < n; i += 128) {
            const uint4 x0 = from[i], x1 = from[i + 32], x2 = from[i + 64], x3 = from[i + 96];
            to[i] = x0;
            to[i + 32] = x1;
            to[i + 64] = x2;
            to[i + 96] = x3;
        }
        for (; i < n; i += 32) to[i] = from[i];
    }
}

struct LseArgs {
    const float *src;
    float *dst;
    int layout;
    int64_t B, L, H, R, U, Hu, LR;
};

// dst [B, H, L] <- src [R, U*B, H/U, L/R]; one thread per destination element
__global__ void __launch_bounds__(256) lse_to_seq_kernel(const LseArgs a) {
    const int64_t total = a.B * a.H * a.L;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t t = i % a.L;
        const int64_t bh = i / a.L;
        const int64_t hg = bh % a.H, b = bh / a.H;
        const int64_t u = hg / a.Hu, hh = hg - u * a.Hu;
        int64_t r, s;
        layout_inv(a.layout, t, a.R, a.LR, r, s);
        a.dst[i] = a.src[((r * (a.U * a.B) + u * a.B + b) * a.Hu + hh) * a.LR + s];
    }
}

static int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
    }
    return n;
}

static unsigned grid_for(int64_t work, int threads, int per_sm) {
    int64_t want = (work + threads - 1) / threads;
    int64_t cap = (int64_t)num_sms() * per_sm;
    if (want > cap) want = cap;
    return (unsigned)(want < 1 ? 1 : want);
}

ra_status launch_permute(const void *src, void *dst, int op, int layout, int64_t B, int64_t L,
                         int64_t H, int64_t d, int R, int U, int elem_bytes, cudaStream_t stream,
                         const char **err) {
    PermArgs a;
    a.src = static_cast<const uint8_t *>(src);
    a.dst = static_cast<uint8_t *>(dst);
    a.op = op;
    a.layout = layout;
    a.B = B;
    a.L = L;
    a.R = R;
    a.U = U;
    a.Lp = L / ((int64_t)U * R);
    const int64_t tok_bytes = H * d * elem_bytes;
    a.seq_slab_vecs = tok_bytes / 16;
    if (op == RA_SEQ_TO_SHARDS || op == RA_SHARDS_TO_SEQ) {
        a.slab_vecs = tok_bytes / 16;
        a.total_vecs = B * L * a.slab_vecs;
    } else {
        a.slab_vecs = (H / U) * d * elem_bytes / 16;
        a.total_vecs = B * L * a.seq_slab_vecs;
    }
    if (a.total_vecs == 0) return RA_OK;
    const int64_t n_slabs = a.total_vecs / a.slab_vecs;
    permute_kernel<<<grid_for(n_slabs * 32, 256, 8), 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = cudaGetErrorString(e);
        return RA_ERR_CUDA;
    }
    return RA_OK;
}

ra_status launch_lse_to_seq(const float *src, float *dst, int layout, int64_t B, int64_t L,
                            int64_t H, int R, int U, cudaStream_t stream, const char **err) {
    LseArgs a;
    a.src = src;
    a.dst = dst;
    a.layout = layout;
    a.B = B;
    a.L = L;
    a.H = H;
    a.R = R;
    a.U = U;
    a.Hu = H / U;
    a.LR = L / R;
    const int64_t total = B * H * L;
    if (total == 0) return RA_OK;
    lse_to_seq_kernel<<<grid_for(total, 256, 8), 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = cudaGetErrorString(e);
        return RA_ERR_CUDA;
    }
    return RA_OK;
}

}  // namespace ra
