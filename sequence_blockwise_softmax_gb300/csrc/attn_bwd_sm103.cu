// attn_bwd_sm103.cu -- gradients of the ring attention on the sm_103a tensor cores.
//
// The pages give the forward pass only; these kernels differentiate it:
// for one head, with P = softmax(S), S = Q K^T * scale under the forward's
// masks, and dO the gradient of O,
//     dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  D = rowsum(dO * O),
//     dQ = dS K * scale,  dK = dS^T Q * scale.
// P is rebuilt exactly from the forward's LSE: P = exp2(S * scale * log2 e -
// LSE * log2 e); no online softmax is needed.
//
// Two passes, no atomics, deterministic:
//   dot kernel   D = rowsum(dO * O), one warp per row, reduced by shuffles.
//   pass A       one CTA per 128 keys of one (kv rank, batch, kv head):
//                S^T = K Q^T and dP^T = V dO^T into tensor memory for each
//                visible 128-query tile of every query rank and every query
//                head of the group; the elementwise threads build P^T from
//                S^T alone (bf16, into shared memory at d = 128, into free
//                tensor-memory columns at d = 64) and then dS^T once dP^T is
//                there (bf16, back into tensor memory); dV += P^T dO and
//                dK += dS^T Q accumulate in tensor memory.  With P^T out of
//                S^T's columns, S^T(t+1) only waits until S^T(t) is in registers, so
//                P^T(t+1) can start as soon as dS^T(t) is done; dP^T(t+1)
//                waits for dK(t), which reads the columns it overwrites.
//   pass B       one CTA per 128 queries: S = Q K^T and dP = dO V^T for each
//                visible key tile in ring order; one thread per query builds
//                dS; dQ += dS K accumulates in tensor memory.  S/dS is double
//                buffered and dP is taken into registers first, so S(t+1) and
//                dP(t+1) run while dS(t) is built.
// Masks (causal by position, packed sequences) are the forward's: in every
// layout positions increase along a rank, so the visible partners of a row in
// a shard form one interval of local indices.
//
// Warp roles (384 threads): warp 0 TMA producer, warps 1-3 MMA issuers
// (elect.sync; so that a wait of one never holds back another's products: the
// tensor pipe takes only a few MMAs ahead of execution) -- in pass A warp 1
// issues S^T and dP^T and warp 3 the gradient products, in pass B warp 1 dP,
// warp 2 S and warp 3 dQ -- warp 2 also allocates tensor memory, warps 4-11
// the elementwise
// threads, two per tensor-memory lane: warps 4-7 take the first 64 columns of
// a tile and warps 8-11 the last 64 (no product here reduces along a row, so
// the halves never exchange data).  Every wait is bounded.
//
// Operands come through the forward's 4-D views (shard stacks or token order,
// tile_view / tile_coords); in token order the gradient rows are stored at
// their token positions, and the dot kernel leaves D and a copy of LSE in
// stack order so that both passes read a tile's vectors contiguously.
#include <cmath>

#include "ra_device.cuh"
#include "ra_internal.h"
#include "ra_positions.cuh"

namespace ra {

// lse and dvec are [Z, H, S] (Z = N * B) in both forms (in token order lse
// is the stack-order copy bwd_dot makes).  dq [Z, S, H, d] and dk, dv
// [Z, S, H_kv, d] in shard stacks; in token order (seq_order) dq [B, L, H, d]
// and dk, dv [B, L, H_kv, d], a row at its token position.
struct BwdArgs {
    const float *lse;       // natural log (forward output)
    const float *dvec;      // D = rowsum(dO * O)
    float *dq;
    float *dk, *dv;
    unsigned *status;
    const int *cu_seqlens;
    int n_seqs;
    int B, S, H, Hkv, N, layout, causal;
    float scale, scale_log2;
    int n_tiles_seq;        // ceil(S / 128)
    int bh_chunk_q;         // (batch, head) pairs interleaved heavy-first in the dQ pass
    int bh_chunk_kv;        // (batch, key/value head) pairs, the same in the dK/dV pass
    int seq_order;          // token-order tensors (the layout is the tiles' addresses)
};

__device__ __forceinline__ uint8_t *bwd_align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void bwd_timeout(unsigned *status, volatile int *abort) {
    *abort = 1;
    atomicOr(status, RA_DEV_TIMEOUT_BIT);
}

// S-style product: D[tmem] = A B^T over K = d, both operands K-major 128-row
// tiles stored as 64-column boxes (offsets in 16-byte units).
template <int D>
__device__ __forceinline__ void issue_kmajor(uint32_t d_tmem, uint64_t a0, uint64_t b0) {
    constexpr uint32_t IDESC = idesc_bf16_f32(128, 128, false);
    mma_ss_elect<0, 0>(d_tmem, a0, b0, IDESC, 0u);
    mma_ss_elect<2, 2>(d_tmem, a0, b0, IDESC, 1u);
    mma_ss_elect<4, 4>(d_tmem, a0, b0, IDESC, 1u);
    mma_ss_elect<6, 6>(d_tmem, a0, b0, IDESC, 1u);
    if (D == 128) {
        constexpr uint32_t h = (128u * 128u) >> 4;
        mma_ss_elect<h, h>(d_tmem, a0, b0, IDESC, 1u);
        mma_ss_elect<h + 2, h + 2>(d_tmem, a0, b0, IDESC, 1u);
        mma_ss_elect<h + 4, h + 4>(d_tmem, a0, b0, IDESC, 1u);
        mma_ss_elect<h + 6, h + 6>(d_tmem, a0, b0, IDESC, 1u);
    }
}

// Accumulating product: D[tmem] (+)= A[tmem, bf16, 128 x 128] B[smem], B a
// 128-row tile read MN-major (N = d), 16 rows per k-step.
template <int D>
__device__ __forceinline__ void issue_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0, bool first) {
    constexpr uint32_t IDESC = idesc_bf16_f32(128, D, true);
    mma_ts_elect<0, 0>(d_tmem, a_tmem, b0, IDESC, first ? 0u : 1u);
    mma_ts_elect<8, 128>(d_tmem, a_tmem, b0, IDESC, 1u);
    mma_ts_elect<16, 256>(d_tmem, a_tmem, b0, IDESC, 1u);
    mma_ts_elect<24, 384>(d_tmem, a_tmem, b0, IDESC, 1u);
    mma_ts_elect<32, 512>(d_tmem, a_tmem, b0, IDESC, 1u);
    mma_ts_elect<40, 640>(d_tmem, a_tmem, b0, IDESC, 1u);
    mma_ts_elect<48, 768>(d_tmem, a_tmem, b0, IDESC, 1u);
    mma_ts_elect<56, 896>(d_tmem, a_tmem, b0, IDESC, 1u);
}

// The same product in two halves of the 128-long K dimension (HALF 0: rows
// 0-63 of B / columns 0-31 of A; HALF 1: the rest), so the first half can run
// while the elementwise warps still produce the second.
template <int D, int HALF>
__device__ __forceinline__ void issue_ts_half(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0, bool first) {
    constexpr uint32_t IDESC = idesc_bf16_f32(128, D, true);
    if (HALF == 0) {
        mma_ts_elect<0, 0>(d_tmem, a_tmem, b0, IDESC, first ? 0u : 1u);
        mma_ts_elect<8, 128>(d_tmem, a_tmem, b0, IDESC, 1u);
        mma_ts_elect<16, 256>(d_tmem, a_tmem, b0, IDESC, 1u);
        mma_ts_elect<24, 384>(d_tmem, a_tmem, b0, IDESC, 1u);
    } else {
        mma_ts_elect<32, 512>(d_tmem, a_tmem, b0, IDESC, 1u);
        mma_ts_elect<40, 640>(d_tmem, a_tmem, b0, IDESC, 1u);
        mma_ts_elect<48, 768>(d_tmem, a_tmem, b0, IDESC, 1u);
        mma_ts_elect<56, 896>(d_tmem, a_tmem, b0, IDESC, 1u);
    }
}

// The same accumulating product with A in shared memory: a 128 x 128 bf16
// K-major tile stored as two 64-column boxes (HALF 0: columns 0-63, the first
// box; HALF 1: the second), B as in issue_ts_half.
template <int D, int HALF>
__device__ __forceinline__ void issue_ss_half(uint32_t d_tmem, uint64_t a0, uint64_t b0, bool first) {
    constexpr uint32_t IDESC = idesc_bf16_f32(128, D, true);
    constexpr uint32_t hb = (128u * 128u) >> 4;
    if (HALF == 0) {
        mma_ss_elect<0, 0>(d_tmem, a0, b0, IDESC, first ? 0u : 1u);
        mma_ss_elect<2, 128>(d_tmem, a0, b0, IDESC, 1u);
        mma_ss_elect<4, 256>(d_tmem, a0, b0, IDESC, 1u);
        mma_ss_elect<6, 384>(d_tmem, a0, b0, IDESC, 1u);
    } else {
        mma_ss_elect<hb, 512>(d_tmem, a0, b0, IDESC, 1u);
        mma_ss_elect<hb + 2, 640>(d_tmem, a0, b0, IDESC, 1u);
        mma_ss_elect<hb + 4, 768>(d_tmem, a0, b0, IDESC, 1u);
        mma_ss_elect<hb + 6, 896>(d_tmem, a0, b0, IDESC, 1u);
    }
}

// Write 32 accumulator columns of one row (scaled) as fp32.
__device__ __forceinline__ void store_row32(float *dst, const uint32_t (&r)[32], float mul) {
    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int c = 0; c < 8; ++c)
        d4[c] = make_float4(__uint_as_float(r[4 * c]) * mul, __uint_as_float(r[4 * c + 1]) * mul,
                            __uint_as_float(r[4 * c + 2]) * mul, __uint_as_float(r[4 * c + 3]) * mul);
}

// ---------------------------------------------------------------- D = rowsum(dO * O)
// One warp per row (z, s, h) of the [Z, S, H] shard stacks, Z = N * B:
// D[(z * H + h) * S + s] = dO . O.  In token order the row's O and dO are read
// at its token position, and its LSE ([B, H, L]) is copied to the same
// stack-order index of lse_stack, so that both passes read D and LSE of a
// tile's rows as one contiguous run.
template <int D>
__global__ void __launch_bounds__(256) bwd_dot_kernel(const uint16_t *dout, const float *o, float *dvec,
                                                      int64_t rows, int H, int64_t S, int seq_order, int layout,
                                                      int N, int B, const float *lse_tok, float *lse_stack) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    constexpr int PER = D / 32;   // elements per lane: one 8-byte (d = 128) or 4-byte dO load, one 16- or 8-byte O load
    constexpr int R = 4;          // rows per warp and iteration
    static_assert(PER == 2 || PER == 4, "d is 64 or 128");
    // R rows per warp and iteration: every row's dO and O loads, and (lane u
    // for row u) its LSE load, are issued before any reduction, so that one
    // memory round trip serves R rows.
    for (int64_t r0 = R * ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)); r0 < rows;
         r0 += R * warps) {
        int64_t dst[R];
        uint32_t dw[R][PER / 2];
        float ov[R][PER];
        float my_lse = 0.f;   // lane u < R: the LSE of row u
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int64_t r = r0 + u;
            dst[u] = -1;
#pragma unroll
            for (int e = 0; e < PER; ++e) ov[u][e] = 0.f;
#pragma unroll
            for (int e = 0; e < PER / 2; ++e) dw[u][e] = 0u;
            if (r >= rows) continue;
            const int64_t h = r % H, zs = r / H;
            const int64_t s = zs % S, z = zs / S;
            int64_t src = r;
            if (seq_order) {
                const int rank = (int)(z / B), b = (int)(z % B);
                const int64_t p = token_pos(layout, rank, s, N, S);
                src = ((int64_t)b * N * S + p) * H + h;
                if (lane == u) my_lse = lse_tok[((int64_t)b * H + h) * N * S + p];
            }
            dst[u] = (z * H + h) * S + s;
            const uint16_t *dp = dout + src * D + lane * PER;
            const float *op = o + src * D + lane * PER;
            if constexpr (PER == 4) {
                const uint2 w = *reinterpret_cast<const uint2 *>(dp);
                const float4 f = *reinterpret_cast<const float4 *>(op);
                dw[u][0] = w.x;
                dw[u][1] = w.y;
                ov[u][0] = f.x;
                ov[u][1] = f.y;
                ov[u][2] = f.z;
                ov[u][3] = f.w;
            } else {
                dw[u][0] = *reinterpret_cast<const uint32_t *>(dp);
                const float2 f = *reinterpret_cast<const float2 *>(op);
                ov[u][0] = f.x;
                ov[u][1] = f.y;
            }
        }
#pragma unroll
        for (int u = 0; u < R; ++u) {
            // bf16 widened exactly (element 2k is the low half of word k),
            // accumulated in element order
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                const uint32_t w = dw[u][e >> 1];
                acc += __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16)) * ov[u][e];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (dst[u] >= 0) {
                if (lane == 0) dvec[dst[u]] = acc;
                if (seq_order && lane == u) lse_stack[dst[u]] = my_lse;
            }
        }
    }
}

// ---------------------------------------------------------------- pass B: dQ
template <int D>
struct BwdQSmem {
    // K lives until dQ(t) has read it, V only until dP(t) has: three K
    // stages keep the next K loaded while dQ of the one before runs
    static constexpr int kKStages = 3, kVStages = 2;
    static constexpr uint32_t kTile = 128u * D * 2u;
    static constexpr uint32_t kBox = 128u * 128u;
    static constexpr uint32_t kQ = 0, kDO = kTile, kK = 2 * kTile;
    static constexpr uint32_t kV = kK + kKStages * kTile;
    static constexpr uint32_t kBars = kV + kVStages * kTile;
    // Q+dO full, K full[3], K empty[3], V full[2], V empty[2], S full[2] (one
    // per S buffer), dP full, dP free, dS full (keys 0-63), dS full (keys
    // 64-127), dS seen by the dQ issuer, dQ done[2] (one per S buffer), final
    static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 10;
    static constexpr uint32_t kMisc = kBars + kNumBars * 8;
    static constexpr uint32_t kBytes = kMisc + 16 + 1024;
};

template <int D>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                       const BwdArgs args) {
    using L = BwdQSmem<D>;
    constexpr int NK = L::kKStages, NV = L::kVStages;
    constexpr int HALVES = D / 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = bwd_align1024(smem_raw);
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar0 = s_base + L::kBars;
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    const int B_QFULL = 0, B_KFULL = 1, B_KEMPTY = 1 + NK, B_VFULL = 1 + 2 * NK, B_VEMPTY = 1 + 2 * NK + NV,
              B_SFULL = 1 + 2 * NK + 2 * NV, B_DPFULL = B_SFULL + 2, B_DPFREE = B_SFULL + 3,
              B_DSFULL = B_SFULL + 4, B_DSFULL2 = B_SFULL + 5, B_DSACK = B_SFULL + 6,
              B_DQDONE = B_SFULL + 7, B_FINAL = B_SFULL + 9;
    // tensor memory: S/dS double buffer at columns 0 and 384, dP at 128, dQ at 256
    auto s_col = [](int t) -> uint32_t { return (t & 1) ? 384u : 0u; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int S = args.S, H = args.H, N = args.N;
    // causal work grows with the query position: heaviest tiles first
    const UnitId unit = decode_unit(blockIdx.x, args.bh_chunk_q, args.B, H, N, args.n_tiles_seq, args.layout);
    const int b = unit.b, h = unit.h, qi = unit.qi, qt = unit.qt;
    const int zq = qi * args.B + b;
    const int row0 = qt * 128;
    const int row_end = min(S, row0 + 128);
    const int hk = h / (H / args.Hkv);
    const int64_t total = (int64_t)N * S;

    const TileWalk walk0 = unit_walk(args.layout, N, S, qi, -1, N, 0, row0, row_end, args.causal, args.cu_seqlens,
                                     args.n_seqs);

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_QFULL), 1);
        for (int s = 0; s < NK; ++s) {
            mbar_init(BAR(B_KFULL + s), 1);
            mbar_init(BAR(B_KEMPTY + s), 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(BAR(B_VFULL + s), 1);
            mbar_init(BAR(B_VEMPTY + s), 1);
        }
        mbar_init(BAR(B_SFULL), 1);
        mbar_init(BAR(B_SFULL + 1), 1);
        mbar_init(BAR(B_DPFULL), 1);
        mbar_init(BAR(B_DPFREE), 256);
        mbar_init(BAR(B_DSFULL), 128);
        mbar_init(BAR(B_DSFULL2), 128);
        mbar_init(BAR(B_DSACK), 1);
        mbar_init(BAR(B_DQDONE), 1);
        mbar_init(BAR(B_DQDONE + 1), 1);
        mbar_init(BAR(B_FINAL), 3);   // the three MMA issuers
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ producer
        int t = 0, k_issued = 0, v_issued = 0;
        bool ok = true;
        if (lane == 0) {
            mbar_arrive_expect_tx(BAR(B_QFULL), 2 * L::kTile);
            int c1, c2, c3;
            tile_coords(args.seq_order, args.layout, S, N, qi, b, row0, c1, c2, c3);
            for (int c = 0; c < HALVES; ++c) {
                tma_load_4d(s_base + L::kQ + c * L::kBox, &tmq, BAR(B_QFULL), h * D + 64 * c, c1, c2, c3);
                tma_load_4d(s_base + L::kDO + c * L::kBox, &tmdo, BAR(B_QFULL), h * D + 64 * c, c1, c2, c3);
            }
        }
        __syncwarp();
        TileWalk w = walk0;
        w.start_step();
        for (; w.valid(); w.next(), ++t) {
            const int sk = t % NK, sv = t % NV;
            int k1, k2, k3;
            tile_coords(args.seq_order, args.layout, S, N, w.j, b, w.tile * 128, k1, k2, k3);
            if (t >= NK && !(ok = warp_wait(BAR(B_KEMPTY + sk), ((t / NK) - 1) & 1, abort_flag))) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(BAR(B_KFULL + sk), L::kTile);
                for (int c = 0; c < HALVES; ++c)
                    tma_load_4d(s_base + L::kK + sk * L::kTile + c * L::kBox, &tmk, BAR(B_KFULL + sk),
                                hk * D + 64 * c, k1, k2, k3);
            }
            __syncwarp();
            k_issued = t + 1;
            if (t >= NV && !(ok = warp_wait(BAR(B_VEMPTY + sv), ((t / NV) - 1) & 1, abort_flag))) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(BAR(B_VFULL + sv), L::kTile);
                for (int c = 0; c < HALVES; ++c)
                    tma_load_4d(s_base + L::kV + sv * L::kTile + c * L::kBox, &tmv, BAR(B_VFULL + sv),
                                hk * D + 64 * c, k1, k2, k3);
            }
            __syncwarp();
            v_issued = t + 1;
        }
        if (!ok) {
            if (lane == 0) bwd_timeout(args.status, abort_flag);
            volatile int never = 0;
            mbar_wait(BAR(B_QFULL), 0, &never);
            for (int u = (k_issued > NK ? k_issued - NK : 0); u < k_issued; ++u)
                mbar_wait(BAR(B_KFULL + u % NK), (u / NK) & 1, &never);
            for (int u = (v_issued > NV ? v_issued - NV : 0); u < v_issued; ++u)
                mbar_wait(BAR(B_VFULL + u % NV), (u / NV) & 1, &never);
        }
    } else if (warp >= 1 && warp <= 3) {
        // ------------------------------------------------ MMA issuers
        // Warp 1 issues dP, warp 2 S and warp 3 dQ, so that a wait of one never
        // holds back another's products (the tensor pipe takes only a few
        // MMAs ahead).  Per tile u, warp 1: dP(u) once the elementwise warps
        // hold dP(u-1) in registers; warp 2: S(u) into the S buffer dQ(u-2)
        // read dS from, once that dQ is done; warp 3: dQ(u) in two key halves
        // as the halves of dS(u) arrive.  Each issuer commits its own products.
        const uint64_t dq_desc = sdesc_sw128(s_base + L::kQ, 16, 1024);
        const uint64_t ddo_desc = sdesc_sw128(s_base + L::kDO, 16, 1024);
        const uint64_t dk_k = sdesc_sw128(s_base + L::kK, 16, 1024);       // K as K-major operand
        const uint64_t dk_mn = sdesc_sw128(s_base + L::kK, L::kBox, 1024); // K as MN-major operand
        const uint64_t dv_k = sdesc_sw128(s_base + L::kV, 16, 1024);
        auto issue_s = [&](int u) {
            issue_kmajor<D>(tmem + s_col(u), dq_desc, dk_k + (uint64_t)((u % NK) * (L::kTile >> 4)));
            tc_commit_elect(BAR(B_SFULL + (u & 1)));
        };
        auto issue_dp = [&](int u) {
            issue_kmajor<D>(tmem + 128, ddo_desc, dv_k + (uint64_t)((u % NV) * (L::kTile >> 4)));
            tc_commit_elect(BAR(B_DPFULL));
            tc_commit_elect(BAR(B_VEMPTY + u % NV));
        };
        bool ok = warp_wait(BAR(B_QFULL), 0, abort_flag);
        TileWalk w = walk0;
        w.start_step();
        int t = 0;
        if (warp == 1) {
            // dP(u) once the elementwise warps hold dP(u-1) in registers
            for (; ok && w.valid(); w.next(), ++t) {
                if (!(ok = warp_wait(BAR(B_VFULL + t % NV), (t / NV) & 1, abort_flag))) break;
                if (t > 0 && !(ok = warp_wait(BAR(B_DPFREE), (t - 1) & 1, abort_flag))) break;
                tc_fence_after();
                issue_dp(t);
                __syncwarp();
            }
        } else if (warp == 2) {
            // S(u) into the S buffer dQ(u-2) read dS from, once that dQ is done
            // (one dQ-done barrier per buffer, so neither can run two phases
            // ahead of this wait)
            for (; ok && w.valid(); w.next(), ++t) {
                if (!(ok = warp_wait(BAR(B_KFULL + t % NK), (t / NK) & 1, abort_flag))) break;
                if (t > 1 && !(ok = warp_wait(BAR(B_DQDONE + ((t - 2) & 1)), ((t - 2) >> 1) & 1, abort_flag)))
                    break;
                tc_fence_after();
                issue_s(t);
                __syncwarp();
            }
        } else {
            for (; ok && w.valid(); w.next(), ++t) {
                const uint64_t koff = (uint64_t)((t % NK) * (L::kTile >> 4));
                if (!(ok = warp_wait(BAR(B_KFULL + t % NK), (t / NK) & 1, abort_flag))) break;
                if (!(ok = warp_wait(BAR(B_DSFULL), t & 1, abort_flag))) break;
                tc_fence_after();
                issue_ts_half<D, 0>(tmem + 256, tmem + s_col(t), dk_mn + koff, t == 0);  // dQ += dS K, keys 0-63
                __syncwarp();
                if (!(ok = warp_wait(BAR(B_DSFULL2), t & 1, abort_flag))) break;
                if (lane == 0) mbar_arrive(BAR(B_DSACK));     // both halves of dS(t) seen
                tc_fence_after();
                issue_ts_half<D, 1>(tmem + 256, tmem + s_col(t) + 32, dk_mn + koff, false);   // keys 64-127
                tc_commit_elect(BAR(B_DQDONE + (t & 1)));
                tc_commit_elect(BAR(B_KEMPTY + t % NK));
                __syncwarp();
            }
        }
        if (!ok && lane == 0) bwd_timeout(args.status, abort_flag);
        // every product this warp issued has finished before tensor memory is freed
        __syncwarp();
        tc_commit_elect(BAR(B_FINAL));
        __syncwarp();
        volatile int never = 0;
        mbar_wait(BAR(B_FINAL), 0, &never);
    } else if (warp >= 4) {
        // ------------------------------------------------ dS, two threads per query row:
        // warps 4-7 take keys 0-63, warps 8-11 keys 64-127 (dS has no row
        // reduction, so the halves never talk).  Each half writes its packed dS
        // over its own S columns: keys 0-63 at 0-31, keys 64-127 at 64-95.
        const int wq = warp & 3;
        const int hh = (warp - 4) >> 2;
        const int r = wq * 32 + lane;
        const int a = row0 + r;
        const int a_c = a < S ? a : S - 1;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off, tP = tmem + lane_off + 128, tQ = tmem + lane_off + 256;
        const int64_t my_pos = token_pos(args.layout, qi, a_c, N, S);
        int64_t lo_pos, hi_pos;
        row_key_bounds(args.cu_seqlens, args.n_seqs, total, my_pos, args.causal, lo_pos, hi_pos);
        const size_t vi = ((size_t)zq * H + h) * S + a_c;
        const float lse_v = args.lse[vi];
        const float lse2 = lse_v > -INFINITY ? lse_v * 1.4426950408889634f : 0.f;   // no key: P = 0 anyway
        const float dval = args.dvec[vi];
        const float sl2 = args.scale_log2;
        TileWalk w = walk0;
        w.start_step();
        int t = 0, cur_step = -1, klo = 0, khi = S;
        bool ok = true;
        for (; w.valid(); w.next(), ++t) {
            if (w.step != cur_step) {
                cur_step = w.step;
                klo = (int)keys_upto(args.layout, w.j, lo_pos, N, S);
                khi = (int)keys_upto(args.layout, w.j, hi_pos, N, S);
            }
            // Tile t starts only once the MMA warp has seen both halves of
            // dS(t-1).  dP(t) is issued before that, so without this wait the
            // warps could publish dS(t) before the MMA warp waited for dS(t-1),
            // or a fast warp could count towards tile t while a slow one is
            // still on tile t-1: the dS-full barriers count arrivals, not tiles.
            if (t > 0 && !(ok = warp_wait(BAR(B_DSACK), (t - 1) & 1, abort_flag))) break;
            // this half's dP(t) into registers first, so the next dP can be
            // computed meanwhile
            if (!(ok = warp_wait(BAR(B_DPFULL), t & 1, abort_flag))) break;
            tc_fence_after();
            uint32_t dpv[2][32];
#pragma unroll
            for (int j = 0; j < 2; ++j) tmem_ld32(tP + 64 * hh + 32 * j, dpv[j]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(BAR(B_DPFREE));
            if (!(ok = warp_wait(BAR(B_SFULL + (t & 1)), (t >> 1) & 1, abort_flag))) break;
            tc_fence_after();
            const uint32_t tSb = tS + s_col(t);
            const int lim = khi - w.tile * 128, lim_lo = klo - w.tile * 128;
            const bool partial = lim < 128 || lim_lo > 0;
            const uint64_t sl2x2 = f32x2(sl2, sl2), nl2 = f32x2(-lse2, -lse2), dd2 = f32x2(dval, dval);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c0 = 64 * hh + 32 * j;      // first key column of this chunk
                uint32_t sv[32], out[16];
                tmem_ld32(tSb + c0, sv);
                tmem_wait_ld();
                if (partial) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (c0 + c >= lim || c0 + c < lim_lo) sv[c] = __float_as_uint(-INFINITY);
                }
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    float x0, x1;
                    f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, nl2),
                                x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    float d0, d1;
                    f32x2_split(mul_f32x2(f32x2(p0, p1),
                                          sub_f32x2(f32x2(__uint_as_float(dpv[j][c]), __uint_as_float(dpv[j][c + 1])),
                                                    dd2)), d0, d1);
                    out[c >> 1] = pack_bf16x2(d0, d1);
                }
                tmem_st16(tSb + 64 * hh + 16 * j, out);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(hh == 0 ? B_DSFULL : B_DSFULL2));
        }
        if (!ok) {
            if (lane == 0) bwd_timeout(args.status, abort_flag);
        } else {
            const int T = t;
            if (T > 0) {
                ok = warp_wait(BAR(B_DQDONE + ((T - 1) & 1)), ((T - 1) >> 1) & 1, abort_flag);
                if (!ok && lane == 0) bwd_timeout(args.status, abort_flag);
                tc_fence_after();
            }
            // tensor-memory loads are warp-wide; only the stores depend on the row.
            // Each half writes half of the d columns.
            if (ok) {
                float *dst = args.dq + ((args.seq_order ? (size_t)b * total + (size_t)my_pos
                                                        : (size_t)zq * S + a_c) * H + h) * D;
#pragma unroll
                for (int q = hh * (D / 64); q < (hh + 1) * (D / 64); ++q) {
                    uint32_t v[32];
                    if (T > 0) {
                        tmem_ld32(tQ + 32 * q, v);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c) v[c] = 0u;
                    }
                    if (a < S) store_row32(dst + 32 * q, v, args.scale);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- pass A: dK, dV
template <int D>
struct BwdKVSmem {
    static constexpr int kStages = 2;
    static constexpr uint32_t kTile = 128u * D * 2u;
    static constexpr uint32_t kBox = 128u * 128u;
    static constexpr uint32_t kK = 0, kV = kTile;
    static constexpr uint32_t kQ = 2 * kTile;
    static constexpr uint32_t kDO = kQ + kStages * kTile;
    static constexpr uint32_t kP = kDO + kStages * kTile;         // P^T: 128 keys x 128 queries bf16, two boxes
    static constexpr uint32_t kVec = kP + 2 * kBox;               // per stage: -lse*log2 e [128], D[128]
    static constexpr uint32_t kBars = kVec + kStages * 1024;
    // K+V full, Q full[2], Q empty[2], S full, S free, dP full, P full
    // (queries 0-63), P full (queries 64-127), dS full (0-63), dS full
    // (64-127), dV done, dK done, final
    static constexpr int kNumBars = 1 + 2 * kStages + 10;
    static constexpr uint32_t kMisc = kBars + kNumBars * 8;
    // no alignment slack: the kernel requires (and checks) a 1024-byte-aligned
    // dynamic base, which is what leaves room for P^T
    static constexpr uint32_t kBytes = kMisc + 16;
};

template <int D>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                        const BwdArgs args) {
    using L = BwdKVSmem<D>;
    constexpr int NS = L::kStages;
    constexpr int HALVES = D / 64;
    // At d = 64 S^T, dP^T, dV and dK leave tensor-memory columns 384-511
    // free, so P^T goes there (queries 0-63 packed in 384-415, 64-127 in
    // 416-447) and dV reads it as the A operand of a TS product: no P^T
    // stores through shared memory and no proxy fence.  At d = 128 the four
    // accumulators fill all 512 columns and P^T goes through shared memory.
    constexpr bool PT_IN_TMEM = D == 64;
    constexpr uint32_t kColPT = 384;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    if ((smem_u32(smem) & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicOr(args.status, RA_DEV_SMEM_ALIGN_BIT);
        return;
    }
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar0 = s_base + L::kBars;
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    const int B_KVFULL = 0, B_QFULL = 1, B_QEMPTY = 1 + NS, B_SFULL = 1 + 2 * NS, B_SFREE = B_SFULL + 1,
              B_DPFULL = B_SFULL + 2, B_PFULL = B_SFULL + 3, B_PFULL2 = B_SFULL + 4, B_DSFULL = B_SFULL + 5,
              B_DSFULL2 = B_SFULL + 6, B_DVDONE = B_SFULL + 7, B_DKDONE = B_SFULL + 8,
              B_FINAL = B_SFULL + 9;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int S = args.S, H = args.H, N = args.N, Hkv = args.Hkv;
    const int group = H / Hkv;
    // causal work shrinks with the key position: earliest keys first
    const UnitId unit = decode_key_block(blockIdx.x, args.bh_chunk_kv, args.B, Hkv, N, args.n_tiles_seq,
                                         args.layout);
    const int b = unit.b, hk = unit.h, kj = unit.qi, kt = unit.qt;
    const int zk = kj * args.B + b;
    const int c0 = kt * 128;
    const int c_end = min(S, c0 + 128);
    const int64_t total = (int64_t)N * S;

    const QWalk walk0 = key_block_walk(args.layout, N, S, kj, group, c0, c_end, args.causal, args.cu_seqlens,
                                       args.n_seqs);

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_KVFULL), 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(BAR(B_QFULL + s), 33);    // the TMA arrival + 32 lanes storing lse2 / D
            mbar_init(BAR(B_QEMPTY + s), 1);
        }
        mbar_init(BAR(B_SFULL), 1);
        mbar_init(BAR(B_SFREE), 256);
        mbar_init(BAR(B_DPFULL), 1);
        mbar_init(BAR(B_PFULL), 128);
        mbar_init(BAR(B_PFULL2), 128);
        mbar_init(BAR(B_DSFULL), 128);
        mbar_init(BAR(B_DSFULL2), 128);
        mbar_init(BAR(B_DVDONE), 1);
        mbar_init(BAR(B_DKDONE), 1);
        mbar_init(BAR(B_FINAL), 2);   // both MMA issuers
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ producer
        bool ok = true;
        int t = 0, issued = 0;
        if (lane == 0) {
            mbar_arrive_expect_tx(BAR(B_KVFULL), 2 * L::kTile);
            int c1, c2, c3;
            tile_coords(args.seq_order, args.layout, S, N, kj, b, c0, c1, c2, c3);
            for (int c = 0; c < HALVES; ++c) {
                tma_load_4d(s_base + L::kK + c * L::kBox, &tmk, BAR(B_KVFULL), hk * D + 64 * c, c1, c2, c3);
                tma_load_4d(s_base + L::kV + c * L::kBox, &tmv, BAR(B_KVFULL), hk * D + 64 * c, c1, c2, c3);
            }
        }
        __syncwarp();
        QWalk w = walk0;
        w.start();
        for (; w.valid(); w.next(), ++t) {
            const int st = t % NS;
            const int h = hk * group + w.head;
            const int y = w.tile * 128;
            // -lse*log2(e) and D of the 128 query rows (0 past the shard's end),
            // read before the stage wait so their latency overlaps it
            const size_t base = ((size_t)(w.i * args.B + b) * H + h) * S;
            float nl[4], dd[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = y + lane * 4 + e;
                const float lv = row < S ? args.lse[base + row] : 0.f;
                nl[e] = lv > -INFINITY ? lv * -1.4426950408889634f : 0.f;
                dd[e] = row < S ? args.dvec[base + row] : 0.f;
            }
            int c1, c2, c3;
            tile_coords(args.seq_order, args.layout, S, N, w.i, b, y, c1, c2, c3);
            if (t >= NS && !(ok = warp_wait(BAR(B_QEMPTY + st), ((t / NS) - 1) & 1, abort_flag))) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(BAR(B_QFULL + st), 2 * L::kTile);
                for (int c = 0; c < HALVES; ++c) {
                    tma_load_4d(s_base + L::kQ + st * L::kTile + c * L::kBox, &tmq, BAR(B_QFULL + st),
                                h * D + 64 * c, c1, c2, c3);
                    tma_load_4d(s_base + L::kDO + st * L::kTile + c * L::kBox, &tmdo, BAR(B_QFULL + st),
                                h * D + 64 * c, c1, c2, c3);
                }
            }
            float *vec = reinterpret_cast<float *>(smem + L::kVec + st * 1024);
            *reinterpret_cast<float4 *>(vec + lane * 4) = make_float4(nl[0], nl[1], nl[2], nl[3]);
            *reinterpret_cast<float4 *>(vec + 128 + lane * 4) = make_float4(dd[0], dd[1], dd[2], dd[3]);
            mbar_arrive(BAR(B_QFULL + st));
            __syncwarp();
            issued = t + 1;
        }
        if (!ok) {
            if (lane == 0) bwd_timeout(args.status, abort_flag);
            volatile int never = 0;
            mbar_wait(BAR(B_KVFULL), 0, &never);
            for (int u = (issued > NS ? issued - NS : 0); u < issued; ++u)
                mbar_wait(BAR(B_QFULL + u % NS), (u / NS) & 1, &never);
        }
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------ MMA issuers
        const uint64_t dk_k = sdesc_sw128(s_base + L::kK, 16, 1024);
        const uint64_t dv_k = sdesc_sw128(s_base + L::kV, 16, 1024);
        const uint64_t dq_k = sdesc_sw128(s_base + L::kQ, 16, 1024);
        const uint64_t ddo_k = sdesc_sw128(s_base + L::kDO, 16, 1024);
        const uint64_t dq_mn = sdesc_sw128(s_base + L::kQ, L::kBox, 1024);
        const uint64_t ddo_mn = sdesc_sw128(s_base + L::kDO, L::kBox, 1024);
        // Warp 1 issues S^T and dP^T, warp 3 dV and dK, so that a wait of one
        // (for the next query stage, say) never holds back the other's
        // products.  Per query tile t, warp 1: S^T(t+1) once the elementwise
        // threads hold S^T(t) in registers (P^T lives in shared memory), then
        // dP^T(t+1) once dK(t) has read dS^T from the columns it overwrites;
        // warp 3: dV(t) and dK(t), each in two query halves as the halves of
        // P^T(t) and dS^T(t) arrive.  Each issuer commits its own products.
        auto issue_sT = [&](int u) {
            issue_kmajor<D>(tmem, dk_k, dq_k + (uint64_t)((u % NS) * (L::kTile >> 4)));   // S^T = K Q^T
            tc_commit_elect(BAR(B_SFULL));
        };
        auto issue_dpT = [&](int u) {
            issue_kmajor<D>(tmem + 128, dv_k, ddo_k + (uint64_t)((u % NS) * (L::kTile >> 4)));  // dP^T = V dO^T
            tc_commit_elect(BAR(B_DPFULL));
        };
        const uint64_t dp_k = sdesc_sw128(s_base + L::kP, 16, 1024);   // P^T as a K-major operand
        bool ok = warp_wait(BAR(B_KVFULL), 0, abort_flag);
        QWalk w = walk0;
        w.start();
        int t = 0;
        if (warp == 1) {
            if (ok && w.valid()) {
                ok = warp_wait(BAR(B_QFULL), 0, abort_flag);
                if (ok) {
                    tc_fence_after();
                    issue_sT(0);
                    issue_dpT(0);
                }
                __syncwarp();
            }
            while (ok && w.valid()) {
                w.next();
                if (!w.valid()) break;
                const int u = t + 1;
                if (!(ok = warp_wait(BAR(B_SFREE), t & 1, abort_flag))) break;
                if (!(ok = warp_wait(BAR(B_QFULL + u % NS), (u / NS) & 1, abort_flag))) break;
                tc_fence_after();
                issue_sT(u);
                __syncwarp();
                if (!(ok = warp_wait(BAR(B_DKDONE), t & 1, abort_flag))) break;
                tc_fence_after();
                issue_dpT(u);
                __syncwarp();
                ++t;
            }
        } else {
            for (; ok && w.valid(); w.next(), ++t) {
                const int st = t % NS;
                const uint64_t soff = (uint64_t)(st * (L::kTile >> 4));
                if (!(ok = warp_wait(BAR(B_QFULL + st), (t / NS) & 1, abort_flag))) break;
                if (!(ok = warp_wait(BAR(B_PFULL), t & 1, abort_flag))) break;
                tc_fence_after();
                // dV += P^T dO
                if constexpr (PT_IN_TMEM) issue_ts_half<D, 0>(tmem + 256, tmem + kColPT, ddo_mn + soff, t == 0);
                else issue_ss_half<D, 0>(tmem + 256, dp_k, ddo_mn + soff, t == 0);
                __syncwarp();
                if (!(ok = warp_wait(BAR(B_PFULL2), t & 1, abort_flag))) break;
                tc_fence_after();
                if constexpr (PT_IN_TMEM) issue_ts_half<D, 1>(tmem + 256, tmem + kColPT, ddo_mn + soff, false);
                else issue_ss_half<D, 1>(tmem + 256, dp_k, ddo_mn + soff, false);
                tc_commit_elect(BAR(B_DVDONE));
                __syncwarp();
                if (!(ok = warp_wait(BAR(B_DSFULL), t & 1, abort_flag))) break;
                tc_fence_after();
                issue_ts_half<D, 0>(tmem + 256 + D, tmem + 128, dq_mn + soff, t == 0); // dK += dS^T Q
                __syncwarp();
                if (!(ok = warp_wait(BAR(B_DSFULL2), t & 1, abort_flag))) break;
                tc_fence_after();
                issue_ts_half<D, 1>(tmem + 256 + D, tmem + 128 + 32, dq_mn + soff, false);
                tc_commit_elect(BAR(B_DKDONE));
                tc_commit_elect(BAR(B_QEMPTY + st));
                __syncwarp();
            }
        }
        if (!ok && lane == 0) bwd_timeout(args.status, abort_flag);
        // every product this warp issued has finished before tensor memory is freed
        __syncwarp();
        tc_commit_elect(BAR(B_FINAL));
        __syncwarp();
        volatile int never = 0;
        mbar_wait(BAR(B_FINAL), 0, &never);
    } else if (warp >= 4) {
        // ------------------------------------------------ P^T, dS^T, two threads per key:
        // warps 4-7 take queries 0-63, warps 8-11 queries 64-127 (neither P^T nor
        // dS^T has a row reduction, so the halves never talk).  Each half writes
        // its packed result over its own columns: queries 0-63 at 0-31,
        // queries 64-127 at 64-95.
        const int wq = warp & 3;
        const int hh = (warp - 4) >> 2;
        const int r = wq * 32 + lane;
        const int kk = c0 + r;
        const int kk_c = kk < S ? kk : S - 1;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off, tP = tmem + lane_off + 128;
        const uint32_t tV = tmem + lane_off + 256, tK = tmem + lane_off + 256 + D;
        const int64_t kpos = token_pos(args.layout, kj, kk_c, N, S);
        int64_t lo_pos, hi_pos;
        col_query_bounds(args.cu_seqlens, args.n_seqs, total, kpos, args.causal, lo_pos, hi_pos);
        const float sl2 = args.scale_log2;
        QWalk w = walk0;
        w.start();
        int t = 0, cur = -1, qlo = 0, qhi = S;
        bool ok = true;
        for (; w.valid(); w.next(), ++t) {
            if (w.step != cur) {
                cur = w.step;
                qlo = (int)keys_upto(args.layout, w.i, lo_pos, N, S);
                qhi = (int)keys_upto(args.layout, w.i, hi_pos, N, S);
            }
            const int st = t % NS;
            // phase 1: P^T from S^T alone (the vectors came with the Q stage)
            if (!(ok = warp_wait(BAR(B_SFULL), t & 1, abort_flag))) break;
            if (!(ok = warp_wait(BAR(B_QFULL + st), (t / NS) & 1, abort_flag))) break;
            tc_fence_after();
            const float *vec = reinterpret_cast<const float *>(smem + L::kVec + st * 1024);
            const int lim = qhi - w.tile * 128, lim_lo = qlo - w.tile * 128;
            uint32_t pv[2][32];
#pragma unroll
            for (int j = 0; j < 2; ++j) tmem_ld32(tS + 64 * hh + 32 * j, pv[j]);
            tmem_wait_ld();
            // S^T(t) is in registers: the next S^T may overwrite its columns
            tc_fence_before();
            mbar_arrive(BAR(B_SFREE));
            // masked queries get S = -inf (P = 0) in a loop of their own, so the
            // exponential loop below stays one block the compiler can schedule
            if (lim < 128 || lim_lo > 0) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int col = 64 * hh + 32 * j + c;
                        if (col >= lim || col < lim_lo) pv[j][c] = __float_as_uint(-INFINITY);
                    }
            }
            const uint64_t sl2x2 = f32x2(sl2, sl2);
            // P^T stays in registers only as the packed bf16 the dV product uses
            uint32_t pk[2][16];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint64_t *nl2 = reinterpret_cast<const uint64_t *>(vec + 64 * hh + 32 * j);
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    float x0, x1;
                    f32x2_split(fma_f32x2(f32x2(__uint_as_float(pv[j][c]), __uint_as_float(pv[j][c + 1])),
                                          sl2x2, nl2[c >> 1]), x0, x1);
                    pk[j][c >> 1] = pack_bf16x2(ex2(x0), ex2(x1));
                }
            }
            // P^T(t) goes where dV reads it once dV(t-1) has read P^T(t-1): at
            // d = 64 to tensor memory (query 2c and 2c + 1 of the half in column c,
            // the first in the low half), at d = 128 to shared memory (the K-major
            // A operand of dV, in the 128-byte-swizzled layout a TMA box load would
            // give: 16-byte chunk j of row r at chunk j ^ (r mod 8))
            if (t > 0 && !(ok = warp_wait(BAR(B_DVDONE), (t - 1) & 1, abort_flag))) break;
            if constexpr (PT_IN_TMEM) {
                tmem_st32(tmem + lane_off + kColPT + 32 * hh, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0][0]));
                tmem_wait_st();
                tc_fence_before();
            } else {
                uint8_t *prow = smem + L::kP + hh * L::kBox + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                    *reinterpret_cast<uint4 *>(prow + ((jj ^ (r & 7)) << 4)) =
                        make_uint4(pk[jj >> 2][(jj & 3) * 4], pk[jj >> 2][(jj & 3) * 4 + 1],
                                   pk[jj >> 2][(jj & 3) * 4 + 2], pk[jj >> 2][(jj & 3) * 4 + 3]);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            mbar_arrive(BAR(hh == 0 ? B_PFULL : B_PFULL2));
            // phase 2: dS^T = P^T (dP^T - D), 32 columns at a time
            if (!(ok = warp_wait(BAR(B_DPFULL), t & 1, abort_flag))) break;
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                uint32_t dp[32], outs[16];
                tmem_ld32(tP + 64 * hh + 32 * j, dp);
                tmem_wait_ld();
                const uint64_t *dd2 = reinterpret_cast<const uint64_t *>(vec + 128 + 64 * hh + 32 * j);
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    // the rounded P the dV product used: bf16 halves widened exactly
                    const uint32_t w = pk[j][c >> 1];
                    const float p0 = __uint_as_float(w << 16), p1 = __uint_as_float(w & 0xffff0000u);
                    float d0, d1;
                    f32x2_split(mul_f32x2(f32x2(p0, p1),
                                          sub_f32x2(f32x2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])),
                                                    dd2[c >> 1])), d0, d1);
                    outs[c >> 1] = pack_bf16x2(d0, d1);
                }
                tmem_st16(tP + 64 * hh + 16 * j, outs);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(hh == 0 ? B_DSFULL : B_DSFULL2));
        }
        if (!ok) {
            if (lane == 0) bwd_timeout(args.status, abort_flag);
        } else {
            const int T = t;
            if (T > 0) {
                ok = warp_wait(BAR(B_DVDONE), (T - 1) & 1, abort_flag) &&
                     warp_wait(BAR(B_DKDONE), (T - 1) & 1, abort_flag);
                if (!ok && lane == 0) bwd_timeout(args.status, abort_flag);
                tc_fence_after();
            }
            // tensor-memory loads are warp-wide; only the stores depend on the row.
            // Each half writes half of the d columns.
            if (ok) {
                const size_t row = ((args.seq_order ? (size_t)b * total + (size_t)kpos
                                                    : (size_t)zk * S + kk_c) * Hkv + hk) * D;
#pragma unroll
                for (int q = hh * (D / 64); q < (hh + 1) * (D / 64); ++q) {
                    uint32_t v[32];
                    if (T > 0) {
                        tmem_ld32(tV + 32 * q, v);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c) v[c] = 0u;
                    }
                    if (kk < S) store_row32(args.dv + row + 32 * q, v, 1.f);
                    if (T > 0) {
                        tmem_ld32(tK + 32 * q, v);
                        tmem_wait_ld();
                    }
                    if (kk < S) store_row32(args.dk + row + 32 * q, v, args.scale);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- host
typedef CUresult (*BwdEncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static BwdEncodeFn bwd_encode_fn() {
    static BwdEncodeFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<BwdEncodeFn>(p);
    }
    return fn;
}

// The 4-D view tile_view describes (shard stacks or token order), bf16, with
// a box of 64 columns by 128 rows in the 128-byte swizzle.
static bool bwd_map(CUtensorMap *map, const void *base, const BwdLaunch &a, int64_t heads, int d) {
    BwdEncodeFn enc = bwd_encode_fn();
    if (!enc) return false;
    const TileView tv = tile_view(a.seq_order, a.layout, a.S, a.B, a.N, a.N, heads * d);
    cuuint64_t dims[4] = {(cuuint64_t)(heads * d), (cuuint64_t)tv.n[0], (cuuint64_t)tv.n[1], (cuuint64_t)tv.n[2]};
    cuuint64_t strides[3] = {(cuuint64_t)tv.st[0] * 2, (cuuint64_t)tv.st[1] * 2, (cuuint64_t)tv.st[2] * 2};
    cuuint32_t box[4] = {64, tv.row_dim == 0 ? 128u : 1u, tv.row_dim == 1 ? 128u : 1u, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static ra_status bwd_launch_t(const BwdLaunch &a, BwdArgs args, cudaStream_t stream, const char **err) {
    const int64_t Z = (int64_t)a.N * a.B;
    CUtensorMap mq, mk, mv, mdo;
    if (!bwd_map(&mq, a.q, a, a.H, D) || !bwd_map(&mk, a.k, a, a.H_kv, D) || !bwd_map(&mv, a.v, a, a.H_kv, D) ||
        !bwd_map(&mdo, a.dout, a, a.H, D)) {
        *err = "cuTensorMapEncodeTiled failed for the backward tensor maps";
        return RA_ERR_CUDA;
    }
    // D = rowsum(dO * O) (and, in token order, the stack-order LSE copy)
    {
        const int64_t rows = Z * a.S * a.H;
        int dev = 0, sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        int64_t blocks = (rows + 31) / 32;   // 8 warps of 4 rows
        if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
        bwd_dot_kernel<D><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint16_t *>(a.dout), a.o,
                                                                 a.dvec, rows, (int)a.H, a.S, a.seq_order ? 1 : 0,
                                                                 a.layout, a.N, (int)a.B, a.lse, a.lse_stack);
    }
    auto kq = attn_bwd_dq_kernel<D>;
    auto kkv = attn_bwd_dkv_kernel<D>;
    if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BwdQSmem<D>::kBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BwdKVSmem<D>::kBytes) !=
            cudaSuccess) {
        *err = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize) failed";
        return RA_ERR_CUDA;
    }
    const int64_t grid_kv = Z * a.H_kv * args.n_tiles_seq;
    const int64_t grid_q = Z * a.H * args.n_tiles_seq;
    if (grid_kv > 0x7fffffffLL || grid_q > 0x7fffffffLL) {
        *err = "too many tiles for one launch";
        return RA_ERR_UNSUPPORTED;
    }
    kkv<<<(unsigned)grid_kv, 384, BwdKVSmem<D>::kBytes, stream>>>(mq, mk, mv, mdo, args);
    kq<<<(unsigned)grid_q, 384, BwdQSmem<D>::kBytes, stream>>>(mq, mk, mv, mdo, args);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = cudaGetErrorString(e);
        return RA_ERR_CUDA;
    }
    return RA_OK;
}

ra_status launch_attention_bwd(const BwdLaunch &a, cudaStream_t stream, const char **err) {
    BwdArgs args;
    args.lse = a.seq_order ? a.lse_stack : a.lse;
    args.dvec = a.dvec;
    args.dq = a.dq;
    args.dk = a.dk;
    args.dv = a.dv;
    args.status = a.status;
    args.cu_seqlens = a.cu_seqlens;
    args.n_seqs = a.n_seqs;
    args.B = (int)a.B;
    args.S = (int)a.S;
    args.H = (int)a.H;
    args.Hkv = (int)a.H_kv;
    args.N = a.N;
    args.layout = a.layout;
    args.causal = a.causal ? 1 : 0;
    args.scale = a.scale > 0.f ? a.scale : 1.0f / std::sqrt((float)a.d);
    args.scale_log2 = args.scale * 1.4426950408889634f;
    args.n_tiles_seq = (int)((a.S + 127) / 128);
    args.seq_order = a.seq_order ? 1 : 0;
    if ((int64_t)a.N * a.B * a.S * a.H == 0) return RA_OK;
    {
        // bytes a tile's sweep streams per (batch, head) pair: keys + values
        // per query head in the dQ pass (shared by a GQA group), queries + dO
        // of the whole group per key/value head in the dK/dV pass
        const int64_t group = a.H / a.H_kv;
        const int64_t per_head = 2 * (int64_t)a.N * a.S * a.d * 2;
        args.bh_chunk_q = chunk_pairs(per_head / group, a.B * a.H);
        args.bh_chunk_kv = chunk_pairs(per_head * group, a.B * a.H_kv);
    }
    return a.d == 128 ? bwd_launch_t<128>(a, args, stream, err) : bwd_launch_t<64>(a, args, stream, err);
}

}  // namespace ra
