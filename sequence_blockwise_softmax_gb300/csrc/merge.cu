// merge.cu -- LSE merge of two partial attention results, and the fp32 -> bf16
// finish of the stepwise ring sweep.
//
// The merge ("From Ring Attention to DeepSpeed Ulysses to USP",
// jsqmd.com/news/734632, §6.3):
//   lse = max(lse_a, lse_b) + ln(1 + exp(-|lse_a - lse_b|))
//   O   = O_a exp(lse_a - lse) + O_b exp(lse_b - lse)
// with -inf marking an empty partial (weight 0; two empties stay empty).
//
// Rows come in groups: group g (of n_groups) holds `rows` consecutive LSE
// entries (lse[g * rows + s]) whose O rows sit `row_stride` floats apart,
// the group itself starting at (g / gh) * stride_hi + (g % gh) * stride_lo.
// The plain strided merge is one group; the [B, S, H, d] / [B, H, S] tensors
// of the ring calls are B * H groups of S rows (gh = H, stride_hi = S*H*d,
// stride_lo = d, row_stride = H*d).  One warp takes 32 rows of a group: lane
// i loads the two LSEs of row i (coalesced), computes the merged LSE and both
// weights, and the warp then walks the 32 O rows, receiving each row's weights
// from its owner lane by shuffle and streaming the row with 16-byte loads and
// stores.
#include "ra_internal.h"

namespace ra {

struct MergeArgs {
    float *o_acc;
    float *lse_acc;
    const float *o_b;
    const float *lse_b;
    int64_t n_groups, rows, gh;
    int64_t acc_hi, acc_lo, acc_row;   // strides (floats) of the accumulator's O
    int64_t b_hi, b_lo, b_row;         // strides (floats) of partial b's O
    int d;
};

__global__ void __launch_bounds__(256) lse_merge_kernel(const MergeArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t chunks = (a.rows + 31) / 32;
    const int64_t n_chunks = a.n_groups * chunks;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int vec_per_row = a.d >> 2;
    for (int64_t ci = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); ci < n_chunks;
         ci += warps_total) {
        const int64_t g = ci / chunks;
        const int64_t s0 = (ci - g * chunks) * 32;
        const int64_t ghi = g / a.gh, glo = g - ghi * a.gh;
        const int64_t s = s0 + lane;
        float wa = 0.f, wb = 0.f;
        if (s < a.rows) {
            const int64_t li = g * a.rows + s;
            const float la = a.lse_acc[li], lb = a.lse_b[li];
            const float hi = fmaxf(la, lb);
            float lse = -INFINITY;
            if (hi != -INFINITY) {
                lse = hi + log1pf(expf(-fabsf(la - lb)));
                wa = expf(la - lse);
                wb = expf(lb - lse);
            }
            a.lse_acc[li] = lse;
        }
        float *oa0 = a.o_acc + ghi * a.acc_hi + glo * a.acc_lo + s0 * a.acc_row;
        const float *ob0 = a.o_b + ghi * a.b_hi + glo * a.b_lo + s0 * a.b_row;
        const int n = (int)((a.rows - s0) < 32 ? (a.rows - s0) : 32);
        for (int i = 0; i < n; ++i) {
            const float ra_ = __shfl_sync(0xffffffffu, wa, i);
            const float rb_ = __shfl_sync(0xffffffffu, wb, i);
            float4 *oa = reinterpret_cast<float4 *>(oa0 + i * a.acc_row);
            const float4 *ob = reinterpret_cast<const float4 *>(ob0 + i * a.b_row);
            for (int c = lane; c < vec_per_row; c += 32) {
                const float4 x = oa[c], y = ob[c];
                oa[c] = make_float4(x.x * ra_ + y.x * rb_, x.y * ra_ + y.y * rb_,
                                    x.z * ra_ + y.z * rb_, x.w * ra_ + y.w * rb_);
            }
        }
    }
}

__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float4 *src, uint2 *dst, int64_t n4) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 x = src[i];
        uint32_t lo, hi;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(x.y), "f"(x.x));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(x.w), "f"(x.z));
        dst[i] = make_uint2(lo, hi);
    }
}

static int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
    }
    return n;
}

static ra_status run_merge(const MergeArgs &a, cudaStream_t stream, const char **err) {
    const int64_t n_chunks = a.n_groups * ((a.rows + 31) / 32);
    if (n_chunks == 0) return RA_OK;
    int64_t blocks = (n_chunks + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    lse_merge_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = cudaGetErrorString(e);
        return RA_ERR_CUDA;
    }
    return RA_OK;
}

ra_status launch_lse_merge(float *o_acc, float *lse_acc, const float *o_b, const float *lse_b,
                           int64_t B, int64_t S, int64_t H, int d, cudaStream_t stream,
                           const char **err) {
    const int64_t row = H * d;
    MergeArgs a{o_acc, lse_acc, o_b, lse_b, B * H, S, H, S * row, d, row, S * row, d, row, d};
    return run_merge(a, stream, err);
}

ra_status launch_lse_merge_rows(float *o_acc, float *lse_acc, const float *o_b, const float *lse_b,
                                int64_t rows, int d, int64_t acc_row_stride, int64_t b_row_stride,
                                cudaStream_t stream, const char **err) {
    MergeArgs a{o_acc, lse_acc, o_b, lse_b, 1, rows, 1, 0, 0, acc_row_stride, 0, 0, b_row_stride, d};
    return run_merge(a, stream, err);
}

ra_status launch_f32_to_bf16(const float *src, void *dst, int64_t n, cudaStream_t stream,
                             const char **err) {
    const int64_t n4 = n / 4;
    if (n4 == 0) return RA_OK;
    int64_t blocks = (n4 + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    f32_to_bf16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const float4 *>(src),
                                                            static_cast<uint2 *>(dst), n4);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = cudaGetErrorString(e);
        return RA_ERR_CUDA;
    }
    return RA_OK;
}

}  // namespace ra
