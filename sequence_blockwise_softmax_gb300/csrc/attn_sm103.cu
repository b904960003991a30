// attn_sm103.cu -- blockwise exact attention on the sm_103a tensor cores.
//
// One CTA owns a "unit": 256 query rows (two 128-row Q tiles) of one
// (query rank, batch, head).  It sweeps the key/value shards in ring order
// ("From Ring Attention to DeepSpeed Ulysses to USP", jsqmd.com/news/734632,
// §3.1: at step s rank i holds the KV of rank (i - s) mod N) and folds every
// 128-key tile into the running (m, l, O) state of §3.2, so the partial
// results never leave the SM.  Here m is the reference point of the
// exponentials, not necessarily the running max (see kSumLo below).
//
// Causal masking by position (same article §3.4; "What problem does sequence
// parallelism solve?", model.playoffer.cn, engineering notes: the ring decides
// the mask from the token positions).  In every layout a rank's local tokens
// are in increasing global order, so the keys of shard j that query row a may
// see are exactly a prefix 0..kc(a)-1 of that shard.  A unit visits only the
// key tiles that prefix covers for its last row (fully masked tiles are
// skipped), and each softmax thread masks the columns past its own row's
// prefix (diagonal tiles are masked in-tile).
//
// Warp roles (384 threads):
//   warp 0      TMA producer: Q tiles once, then K and V tiles into one ring
//               of three shared-memory slots, K a tile ahead of V.
//   warp 1      MMA issuer (one elected lane): S_g = Q_g K^T into tensor
//               memory, and at d = 64 also O_g += P_g V with P_g read from
//               tensor memory.
//   warp 2      tensor-memory allocator.
//   warp 3      at d = 128, the PV issuer, so that a wait of either issuer
//               never holds back the other's products (the tensor pipe takes
//               only a few MMAs ahead of execution).
//   warps 4-7   softmax for Q tile 0, warps 8-11 for Q tile 1: one thread per
//               query row (the 32x32b tensor-memory load gives a thread its
//               whole row, so row sums need no shuffles), exp2 with the
//               scale folded into log2(e), P written as bf16 to shared memory
//               (d = 128) or tensor memory (d = 64), O rescaled in place when
//               the reference point moves,
//               and the final normalisation, with O staged in shared memory
//               for TMA stores.  At d = 128 warp 4 first counts the unit's
//               key tiles for the two issuers, one ring step per lane.
// Tensor memory (512 columns x 128 lanes): S_0 [0,128), S_1 [128,256),
// O_0 [256, 256+d), O_1 [256+d, 256+2d), and at d = 64 P_0 [384, 448),
// P_1 [448, 512) (bf16 pairs), which PV reads from there; at d = 128 P goes
// through shared memory.  Because P does not live in S's
// columns, S_g(t+1) may be computed while PV_g(t) still runs: the softmax
// releases S_g once P is computed and its denominator checked (the rare
// second pass reloads S), and each tile's critical chain is S -> softmax ->
// PV with no wait on the previous PV in between.
//
// Addressing: every tile moves through a 4-D tensor map of either the shard
// stacks [N, B, S, H, d] or the token-order tensors [B, L, H, d]
// (tile_view / tile_coords).  In token order a layout is only a choice of view
// (§4, §6.1 of the same article), so the sweep reads each rank's shard and
// writes its result in place and no permute runs.
#include <cmath>
#include <cstdio>

#include "ra_device.cuh"
#include "ra_internal.h"
#include "ra_positions.cuh"

namespace ra {

struct AttnArgs {
    void *o;
    float *lse;
    unsigned *status;
    int B, S, H, N;
    int layout, causal;
    float scale_log2;   // softmax scale * log2(e)
    int num_q_ranks;    // N in ring mode, 1 in block mode
    int q_rank_fixed;   // block mode: the query rank; ring mode: -1
    int kv_rank_fixed;  // block mode: the key/value rank; ring mode: -1
    int num_steps;      // N for a full sweep, 1 for one ring step or block mode
    int step_base;      // ring mode: the first step visited (0 for a full sweep)
    int n_units_seq;    // ceil(S / 256)
    int inject_stall;   // test hook: CTA 0 never loads its second K tile
    int kv_group;       // query heads per key/value head (1 without GQA)
    const int *cu_seqlens;  // packed sequences: n_seqs + 1 boundaries, or null
    int n_seqs;
    int bh_chunk;       // (batch, head) pairs whose units are interleaved heavy-first
    int seq_order;      // q/k/v/o in sequence order [B, L, H, d], LSE [B, H, L] (ring mode)
};

__device__ __forceinline__ void record_timeout(unsigned *status, volatile int *abort) {
    *abort = 1;
    atomicOr(status, RA_DEV_TIMEOUT_BIT);
}

template <int D>
struct AttnSmem {
    static constexpr int kSlots = 3;                     // K/V tile ring
    static constexpr uint32_t kTile = 128u * D * 2u;     // 128 rows x d bf16
    static constexpr uint32_t kBox = 128u * 128u;        // 128 rows x 64 columns
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kRing = 2 * kTile;
    static constexpr uint32_t kP = kRing + kSlots * kTile;   // P_g: 128 rows x 128 keys bf16, two boxes each
    static constexpr uint32_t kBars = kP + 2 * 2 * kBox;
    // barriers: Q full, slot full[3], slot empty[3], S full[2], S free[2],
    // P full[2], PV done[2], final, tile count posted
    static constexpr int kNumBars = 1 + 2 * kSlots + 2 + 2 + 2 + 2 + 1 + 1;
    static constexpr uint32_t kMisc = kBars + kNumBars * 8;
    // the tile-skipping variant's step table: per ring step (at most
    // kMaxSteps) the unit's key-tile range and each Q tile's own range inside
    // it, six ints
    static constexpr int kMaxSteps = 64;
    static constexpr uint32_t kTab = kMisc + 16;
    // no alignment slack: the kernel requires (and checks) a 1024-byte-aligned
    // dynamic base, which is what leaves room for P
    static constexpr uint32_t kBytes = kMisc + 16;
    static constexpr uint32_t kBytesSkip = kTab + kMaxSteps * 6 * 4;
};

// The key tiles of a unit's walk as the tile-skipping variant sees them: the
// walk visits tiles [lo, hi) of each step's shard in step order, and Q tile g
// needs only tiles [glo_g, ghi_g) of them.  With no table (more steps than it
// holds) every tile is needed by both Q tiles.
struct StepCursor {
    const int *tab;   // null: no table
    int ns, s, tile, hi, lo0, hi0, lo1, hi1;   // the current step's ranges
    __device__ void seek() {
        while (s < ns && tab[6 * s] >= tab[6 * s + 1]) ++s;
        if (s < ns) {
            tile = tab[6 * s];
            hi = tab[6 * s + 1];
            lo0 = tab[6 * s + 2];
            hi0 = tab[6 * s + 3];
            lo1 = tab[6 * s + 4];
            hi1 = tab[6 * s + 5];
        }
    }
    __device__ void start(const int *t, int n) {
        tab = t;
        ns = n;
        s = 0;
        tile = 0;
        if (tab) seek();
    }
    __device__ void next() {
        if (tab && ++tile >= hi) {
            ++s;
            seek();
        }
    }
    __device__ bool need(int g) const {
        return !tab || (g == 0 ? (lo0 <= tile && tile < hi0) : (lo1 <= tile && tile < hi1));
    }
};

// Reference point of the exponentials.  The online softmax of §3.2 subtracts
// the running row max m only to keep exp() in range: O / l and m + ln l are
// the same for any reference.  A row therefore starts at reference 0 and
// computes P = 2^(s*scale*log2e - m) without a row max; the reference moves
// only when the running denominator would leave [kSumLo, kSumHi] (or is not
// a number), to max(tile max, m + log2 l), which brings the sum into
// [1, 129].  With l <= 2^32 no P and no partial sum of P can overflow, and
// with l >= 2^-32 over at most 2^24 keys the largest term is at least
// 2^-56, so what ex2 flushes to zero (below 2^-126) is less than 2^-70 of
// it.  For scores of ordinary size (|s * scale| up to about 20) the
// reference never moves at all.
constexpr float kSumLo = 0x1p-32f, kSumHi = 0x1p32f;

// SKIP: each Q tile of a unit skips the key tiles none of its own rows sees
// (packed sequences in the striped layout, where a unit's 256 rows span many
// short sequences); the MMA issuers skip those tiles' S and PV.
template <int D, bool OUT_F32, bool SKIP>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                    const AttnArgs args) {
    using L = AttnSmem<D>;
    constexpr int NSL = L::kSlots;
    constexpr int HALVES = D / 64;
    constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, true);
    // At d = 128 warp 1 issues the S products and warp 3 the PV products; at
    // d = 64, where the split measured slower, warp 1 issues both.
    constexpr bool TWO_ISSUERS = D == 128;
    // At d = 64 tensor memory has room for P next to S and O (columns 384-511),
    // so P_g goes there and PV_g reads it as the A operand (a TS product): no
    // P stores through shared memory and no proxy fence.  At d = 128 S and O
    // fill all 512 columns and P goes through shared memory.
    constexpr bool P_IN_TMEM = D == 64;
    // registers per thread of warps 0-3 after setmaxnreg: the second issuer
    // needs more than 64 to issue without spilling
    constexpr uint32_t LOW_REGS = TWO_ISSUERS ? 72u : 64u;
    static_assert(!SKIP || TWO_ISSUERS, "tile skipping is built on the two-issuer pipeline");

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    const uint32_t s_base = smem_u32(smem);
    if ((s_base & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicOr(args.status, RA_DEV_SMEM_ALIGN_BIT);
        return;
    }
    const uint32_t bar0 = s_base + L::kBars;
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    const int B_QFULL = 0, B_SLOTF = 1, B_SLOTE = 1 + NSL, B_SFULL = 1 + 2 * NSL, B_SFREE = B_SFULL + 2,
              B_PFULL = B_SFREE + 2, B_PVDONE = B_PFULL + 2, B_FINAL = B_PVDONE + 2, B_TCOUNT = B_FINAL + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    volatile int *tile_count = reinterpret_cast<volatile int *>(smem + L::kMisc + 8);
    volatile int *tab_ok = reinterpret_cast<volatile int *>(smem + L::kMisc + 12);
    int *step_tab = reinterpret_cast<int *>(smem + L::kTab);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- unit decode: heavy units first, in L2-sized chunks of (batch, head)
    // pairs (decode_unit)
    const int S = args.S, H = args.H, N = args.N;
    const UnitId unit = decode_unit(blockIdx.x, args.bh_chunk, args.B, H, args.num_q_ranks, args.n_units_seq,
                                    args.layout);
    const int b = unit.b, h = unit.h, qi = unit.qi, qt = unit.qt;
    const bool ring = args.q_rank_fixed < 0;
    const int q_rank = ring ? qi : args.q_rank_fixed;
    const int zq = (ring ? qi * args.B : 0) + b;
    const int row0 = qt * 256;
    const int row_end = min(S, row0 + 256);

    const TileWalk walk0 = unit_walk(args.layout, N, S, q_rank, args.kv_rank_fixed, args.num_steps,
                                     args.step_base, row0, row_end, args.causal, args.cu_seqlens, args.n_seqs);

    // ---- setup
    if (threadIdx.x == 0) {
        mbar_init(BAR(B_QFULL), 1);
        for (int s = 0; s < NSL; ++s) {
            mbar_init(BAR(B_SLOTF + s), 1);
            mbar_init(BAR(B_SLOTE + s), 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(BAR(B_SFULL + g), 1);
            mbar_init(BAR(B_SFREE + g), 128);
            mbar_init(BAR(B_PFULL + g), 128);
            mbar_init(BAR(B_PVDONE + g), 1);
        }
        mbar_init(BAR(B_FINAL), TWO_ISSUERS ? 2 : 1);   // one arrival per MMA issuer
        mbar_init(BAR(B_TCOUNT), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmo);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // 384 threads x 168 registers at launch: the producer / MMA / allocator
    // warpgroup (warps 0-3) gives registers to the two softmax warpgroups,
    // 128 x LOW_REGS + 256 x 216 <= 384 x 168 (equal at LOW_REGS = 72); each
    // role makes the call on entry.
    if (warp == 0) {
        // ================================================= TMA producer
        regs_shrink<LOW_REGS>();
        const int xh = h * D;                        // Q columns of head h
        const int xkv = (h / args.kv_group) * D;     // K/V columns of its key/value head
        if (lane == 0) {
            mbar_arrive_expect_tx(BAR(B_QFULL), 2 * L::kTile);
            for (int g = 0; g < 2; ++g) {
                int c1, c2, c3;
                tile_coords(args.seq_order, args.layout, args.S, args.N, ring ? qi : 0, b, row0 + 128 * g, c1, c2, c3);
                for (int c = 0; c < HALVES; ++c)
                    tma_load_4d(s_base + L::kQ + g * L::kTile + c * L::kBox, &tmq, BAR(B_QFULL),
                                xh + 64 * c, c1, c2, c3);
            }
        }
        __syncwarp();
        // K and V tiles share a ring of three slots.  Load order K(0), K(1),
        // V(0), K(2), V(1), ...: K runs a tile ahead, because S(t+1) is issued
        // while P(t) is still being built.  Load i goes to slot i % 3 once the
        // load three before it has been released (K after both S products of
        // its tile, V after both PV products).
        // one walk over the key tiles; V(t) reuses the coordinates K(t) had
        TileWalk wk = walk0;
        wk.start_step();
        int vj = 0, vtile = 0;
        int i = 0, withheld = -1;
        bool ok = true;
        auto load = [&](int wj, int wtile, bool is_k) -> bool {
            const int sl = i % NSL;
            if (i >= NSL && !warp_wait(BAR(B_SLOTE + sl), ((i / NSL) - 1) & 1, abort_flag)) return false;
            const bool withhold = args.inject_stall && blockIdx.x == 0 && i == 1;
            if (lane == 0 && !withhold) {
                const uint32_t dst = s_base + L::kRing + sl * L::kTile;
                int c1, c2, c3;
                tile_coords(args.seq_order, args.layout, args.S, args.N, ring ? wj : 0, b, wtile * 128, c1, c2, c3);
                mbar_arrive_expect_tx(BAR(B_SLOTF + sl), L::kTile);
                for (int c = 0; c < HALVES; ++c) {
                    if (is_k) tma_load_4d(dst + c * L::kBox, &tmk, BAR(B_SLOTF + sl), xkv + 64 * c, c1, c2, c3);
                    else tma_load_4d(dst + c * L::kBox, &tmv, BAR(B_SLOTF + sl), xkv + 64 * c, c1, c2, c3);
                }
            }
            __syncwarp();
            if (withhold) withheld = i;
            ++i;
            return true;
        };
        if (wk.valid()) {
            ok = load(wk.j, wk.tile, true);
            vj = wk.j;
            vtile = wk.tile;
            wk.next();
            while (ok) {
                const bool more = wk.valid();
                if (more && !(ok = load(wk.j, wk.tile, true))) break;
                if (!(ok = load(vj, vtile, false)) || !more) break;
                vj = wk.j;
                vtile = wk.tile;
                wk.next();
            }
        }
        if (!ok) {
            if (lane == 0) record_timeout(args.status, abort_flag);
            // let the copies already issued land before the CTA exits
            volatile int never = 0;
            mbar_wait(BAR(B_QFULL), 0, &never);
            for (int u = (i > NSL ? i - NSL : 0); u < i; ++u)
                if (u != withheld) mbar_wait(BAR(B_SLOTF + u % NSL), (u / NSL) & 1, &never);
        }
    } else if (warp == 1 && !TWO_ISSUERS) {
        // ================================================= MMA issuer (d = 64)
        regs_shrink<LOW_REGS>();
        // Issue order per key tile t (pipe order):
        //   S_0(t+1), PV_0(t), S_1(t+1), PV_1(t)
        // P_g goes to shared memory, so S_g(t+1) may overwrite S_g(t) in
        // tensor memory as soon as the softmax warps of tile g are done with it
        // (S free); nothing here waits for a PV product.  Descriptors are built
        // once; each k-step adds a compile-time offset (16-byte units) to the
        // start-address field: 32 B per 16-element step inside a 64-column box
        // and one box (16 KB) for columns 64-127 of Q, K and P, and 16 rows
        // (2 KB) per step of V.  The whole warp runs the issue code and
        // elect.sync picks the issuing lane.
        const uint64_t dq[2] = {sdesc_sw128(s_base + L::kQ, 16, 1024),
                                sdesc_sw128(s_base + L::kQ + L::kTile, 16, 1024)};
        const uint64_t dp[2] = {sdesc_sw128(s_base + L::kP, 16, 1024),
                                sdesc_sw128(s_base + L::kP + 2 * L::kBox, 16, 1024)};
        const uint64_t dk0 = sdesc_sw128(s_base + L::kRing, 16, 1024);
        const uint64_t dv0 = sdesc_sw128(s_base + L::kRing, L::kBox, 1024);
        auto issue_s = [&](int g, int slot) {
            const uint64_t a0 = dq[g], b0 = dk0 + (uint64_t)(slot * (L::kTile >> 4));
            const uint32_t d = tmem + g * 128;
            mma_ss_elect<0, 0>(d, a0, b0, IDESC_S, 0u);
            mma_ss_elect<2, 2>(d, a0, b0, IDESC_S, 1u);
            mma_ss_elect<4, 4>(d, a0, b0, IDESC_S, 1u);
            mma_ss_elect<6, 6>(d, a0, b0, IDESC_S, 1u);
            if (D == 128) {
                constexpr uint32_t h = L::kBox >> 4;
                mma_ss_elect<h, h>(d, a0, b0, IDESC_S, 1u);
                mma_ss_elect<h + 2, h + 2>(d, a0, b0, IDESC_S, 1u);
                mma_ss_elect<h + 4, h + 4>(d, a0, b0, IDESC_S, 1u);
                mma_ss_elect<h + 6, h + 6>(d, a0, b0, IDESC_S, 1u);
            }
            tc_commit_elect(BAR(B_SFULL + g));
        };
        auto issue_pv = [&](int g, int slot, bool first) {
            constexpr uint32_t hb = L::kBox >> 4;
            const uint64_t a0 = dp[g], b0 = dv0 + (uint64_t)(slot * (L::kTile >> 4));
            const uint32_t d = tmem + 256 + g * D;
            if constexpr (P_IN_TMEM) {
                // A = P_g in tensor memory: 16 keys (8 packed columns) per k-step
                const uint32_t at = tmem + 384 + g * 64;
                mma_ts_elect<0, 0>(d, at, b0, IDESC_O, first ? 0u : 1u);
                mma_ts_elect<8, 128>(d, at, b0, IDESC_O, 1u);
                mma_ts_elect<16, 256>(d, at, b0, IDESC_O, 1u);
                mma_ts_elect<24, 384>(d, at, b0, IDESC_O, 1u);
                mma_ts_elect<32, 512>(d, at, b0, IDESC_O, 1u);
                mma_ts_elect<40, 640>(d, at, b0, IDESC_O, 1u);
                mma_ts_elect<48, 768>(d, at, b0, IDESC_O, 1u);
                mma_ts_elect<56, 896>(d, at, b0, IDESC_O, 1u);
            } else {
                mma_ss_elect<0, 0>(d, a0, b0, IDESC_O, first ? 0u : 1u);
                mma_ss_elect<2, 128>(d, a0, b0, IDESC_O, 1u);
                mma_ss_elect<4, 256>(d, a0, b0, IDESC_O, 1u);
                mma_ss_elect<6, 384>(d, a0, b0, IDESC_O, 1u);
                mma_ss_elect<hb, 512>(d, a0, b0, IDESC_O, 1u);
                mma_ss_elect<hb + 2, 640>(d, a0, b0, IDESC_O, 1u);
                mma_ss_elect<hb + 4, 768>(d, a0, b0, IDESC_O, 1u);
                mma_ss_elect<hb + 6, 896>(d, a0, b0, IDESC_O, 1u);
            }
            tc_commit_elect(BAR(B_PVDONE + g));
        };
        bool ok = warp_wait(BAR(B_QFULL), 0, abort_flag);
        TileWalk w = walk0;
        w.start_step();
        int t = 0;
        if (ok && w.valid()) {
            ok = warp_wait(BAR(B_SLOTF + 0), 0, abort_flag);   // K(0) is load 0
            tc_fence_after();
            if (ok) {
                issue_s(0, 0);
                issue_s(1, 0);
                tc_commit_elect(BAR(B_SLOTE + 0));
            }
            __syncwarp();
        }
        while (ok && w.valid()) {
            w.next();
            const bool has_next = w.valid();
            const int ki = 2 * t + 1;                        // load index of K(t+1)
            const int vi = has_next ? 2 * t + 2 : 2 * t + 1; // load index of V(t)
            if (has_next && !(ok = warp_wait(BAR(B_SLOTF + ki % NSL), (ki / NSL) & 1, abort_flag))) break;
            if (has_next) {
                if (!(ok = warp_wait(BAR(B_SFREE + 0), t & 1, abort_flag))) break;
                tc_fence_after();
                issue_s(0, ki % NSL);
                __syncwarp();
            }
            if (!(ok = warp_wait(BAR(B_SLOTF + vi % NSL), (vi / NSL) & 1, abort_flag))) break;
            if (!(ok = warp_wait(BAR(B_PFULL + 0), t & 1, abort_flag))) break;
            tc_fence_after();
            issue_pv(0, vi % NSL, t == 0);
            __syncwarp();
            if (has_next) {
                if (!(ok = warp_wait(BAR(B_SFREE + 1), t & 1, abort_flag))) break;
                tc_fence_after();
                issue_s(1, ki % NSL);
                tc_commit_elect(BAR(B_SLOTE + ki % NSL));
                __syncwarp();
            }
            if (!(ok = warp_wait(BAR(B_PFULL + 1), t & 1, abort_flag))) break;
            tc_fence_after();
            issue_pv(1, vi % NSL, t == 0);
            tc_commit_elect(BAR(B_SLOTE + vi % NSL));
            __syncwarp();
            ++t;
        }
        if (!ok && lane == 0) record_timeout(args.status, abort_flag);
        // every MMA issued above has finished before tensor memory is freed
        __syncwarp();
        tc_commit_elect(BAR(B_FINAL));
        __syncwarp();
        volatile int never = 0;
        mbar_wait(BAR(B_FINAL), 0, &never);
    } else if (warp == 1) {
        // ================================================= MMA issuers (d = 128)
        regs_shrink<LOW_REGS>();
        // Warp 1 issues the S products and warp 3 the PV products, so that a
        // wait of one never holds back the other (the tensor pipe takes only a
        // few MMAs ahead of execution).  Each commits its own products: warp 1
        // releases K slots, warp 3 V slots.
        // Per key tile t, warp 1: S_0(t+1), S_1(t+1); warp 3: PV_0(t), PV_1(t).
        // P_g goes to shared memory, so S_g(t+1) may overwrite S_g(t) in
        // tensor memory as soon as the softmax warps of tile g are done with it
        // (S free); no S product waits for a PV product.  Descriptors are built
        // once; each k-step adds a compile-time offset (16-byte units) to the
        // start-address field: 32 B per 16-element step inside a 64-column box
        // and one box (16 KB) for columns 64-127 of Q, K and P, and 16 rows
        // (2 KB) per step of V.  The whole warp runs the issue code and
        // elect.sync picks the issuing lane.
        const uint64_t dq[2] = {sdesc_sw128(s_base + L::kQ, 16, 1024),
                                sdesc_sw128(s_base + L::kQ + L::kTile, 16, 1024)};
        const uint64_t dk0 = sdesc_sw128(s_base + L::kRing, 16, 1024);
        auto issue_s = [&](int g, int slot) {
            const uint64_t a0 = dq[g], b0 = dk0 + (uint64_t)(slot * (L::kTile >> 4));
            const uint32_t d = tmem + g * 128;
            mma_ss_elect<0, 0>(d, a0, b0, IDESC_S, 0u);
            mma_ss_elect<2, 2>(d, a0, b0, IDESC_S, 1u);
            mma_ss_elect<4, 4>(d, a0, b0, IDESC_S, 1u);
            mma_ss_elect<6, 6>(d, a0, b0, IDESC_S, 1u);
            if (D == 128) {
                constexpr uint32_t h = L::kBox >> 4;
                mma_ss_elect<h, h>(d, a0, b0, IDESC_S, 1u);
                mma_ss_elect<h + 2, h + 2>(d, a0, b0, IDESC_S, 1u);
                mma_ss_elect<h + 4, h + 4>(d, a0, b0, IDESC_S, 1u);
                mma_ss_elect<h + 6, h + 6>(d, a0, b0, IDESC_S, 1u);
            }
            tc_commit_elect(BAR(B_SFULL + g));
        };
        // the issuers need only the number of key tiles the walk visits,
        // which warp 4 counts (and, when skipping, its step table)
        bool ok = warp_wait(BAR(B_TCOUNT), 0, abort_flag);
        const int T = ok ? *tile_count : 0;
        ok = ok && warp_wait(BAR(B_QFULL), 0, abort_flag);
        if constexpr (!SKIP) {
            int t = 0;
            if (ok && T > 0) {
                ok = warp_wait(BAR(B_SLOTF + 0), 0, abort_flag);   // K(0) is load 0
                tc_fence_after();
                if (ok) {
                    issue_s(0, 0);
                    issue_s(1, 0);
                    tc_commit_elect(BAR(B_SLOTE + 0));
                }
                __syncwarp();
            }
#pragma unroll 1
            for (; ok && t + 1 < T; ++t) {
                const int ki = 2 * t + 1;                    // load index of K(t+1)
                if (!(ok = warp_wait(BAR(B_SLOTF + ki % NSL), (ki / NSL) & 1, abort_flag))) break;
                if (!(ok = warp_wait(BAR(B_SFREE + 0), t & 1, abort_flag))) break;
                tc_fence_after();
                issue_s(0, ki % NSL);
                __syncwarp();
                if (!(ok = warp_wait(BAR(B_SFREE + 1), t & 1, abort_flag))) break;
                tc_fence_after();
                issue_s(1, ki % NSL);
                tc_commit_elect(BAR(B_SLOTE + ki % NSL));
                __syncwarp();
            }
        } else {
            // S_g is issued only for the tiles Q tile g needs; each group's
            // S-free wait counts that group's own products.  A K slot is
            // released after its tile, whether or not any S read it.
            StepCursor cs;
            cs.start((ok && *tab_ok) ? step_tab : nullptr, args.num_steps);
            int ks0 = 0, ks1 = 0;         // S products issued per Q tile
            if (ok && T > 0) {
                ok = warp_wait(BAR(B_SLOTF + 0), 0, abort_flag);   // K(0) is load 0
                tc_fence_after();
                if (ok) {
                    if (cs.need(0)) {
                        issue_s(0, 0);
                        ++ks0;
                    }
                    if (cs.need(1)) {
                        issue_s(1, 0);
                        ++ks1;
                    }
                    tc_commit_elect(BAR(B_SLOTE + 0));
                }
                __syncwarp();
            }
#pragma unroll 1
            for (int t = 0; ok && t + 1 < T; ++t) {
                cs.next();
                const int ki = 2 * t + 1;                    // load index of K(t+1)
                if (!(ok = warp_wait(BAR(B_SLOTF + ki % NSL), (ki / NSL) & 1, abort_flag))) break;
                if (cs.need(0)) {
                    if (ks0 > 0 && !(ok = warp_wait(BAR(B_SFREE + 0), (ks0 - 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    issue_s(0, ki % NSL);
                    ++ks0;
                    __syncwarp();
                }
                if (cs.need(1)) {
                    if (ks1 > 0 && !(ok = warp_wait(BAR(B_SFREE + 1), (ks1 - 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    issue_s(1, ki % NSL);
                    ++ks1;
                }
                tc_commit_elect(BAR(B_SLOTE + ki % NSL));
                __syncwarp();
            }
        }
        if (!ok && lane == 0) record_timeout(args.status, abort_flag);
        // every MMA this warp issued has finished before tensor memory is freed
        __syncwarp();
        tc_commit_elect(BAR(B_FINAL));
        __syncwarp();
        volatile int never = 0;
        mbar_wait(BAR(B_FINAL), 0, &never);
    } else if (warp == 3 && TWO_ISSUERS) {
        // ================================================= MMA issuer for PV (see warp 1)
        regs_shrink<LOW_REGS>();
        const uint64_t dp[2] = {sdesc_sw128(s_base + L::kP, 16, 1024),
                                sdesc_sw128(s_base + L::kP + 2 * L::kBox, 16, 1024)};
        const uint64_t dv0 = sdesc_sw128(s_base + L::kRing, L::kBox, 1024);
        auto issue_pv = [&](int g, int slot, bool first) {
            constexpr uint32_t hb = L::kBox >> 4;
            const uint64_t a0 = dp[g], b0 = dv0 + (uint64_t)(slot * (L::kTile >> 4));
            const uint32_t d = tmem + 256 + g * D;
            mma_ss_elect<0, 0>(d, a0, b0, IDESC_O, first ? 0u : 1u);
            mma_ss_elect<2, 128>(d, a0, b0, IDESC_O, 1u);
            mma_ss_elect<4, 256>(d, a0, b0, IDESC_O, 1u);
            mma_ss_elect<6, 384>(d, a0, b0, IDESC_O, 1u);
            mma_ss_elect<hb, 512>(d, a0, b0, IDESC_O, 1u);
            mma_ss_elect<hb + 2, 640>(d, a0, b0, IDESC_O, 1u);
            mma_ss_elect<hb + 4, 768>(d, a0, b0, IDESC_O, 1u);
            mma_ss_elect<hb + 6, 896>(d, a0, b0, IDESC_O, 1u);
            tc_commit_elect(BAR(B_PVDONE + g));
        };
        // the issuers need only the number of key tiles the walk visits,
        // which warp 4 counts (and, when skipping, its step table)
        bool ok = warp_wait(BAR(B_TCOUNT), 0, abort_flag);
        const int T = ok ? *tile_count : 0;
        ok = ok && warp_wait(BAR(B_QFULL), 0, abort_flag);
        if constexpr (!SKIP) {
            int t = 0;
#pragma unroll 1
            for (; ok && t < T; ++t) {
                const bool has_next = t + 1 < T;
                const int vi = has_next ? 2 * t + 2 : 2 * t + 1; // load index of V(t)
                if (!(ok = warp_wait(BAR(B_SLOTF + vi % NSL), (vi / NSL) & 1, abort_flag))) break;
                if (!(ok = warp_wait(BAR(B_PFULL + 0), t & 1, abort_flag))) break;
                tc_fence_after();
                issue_pv(0, vi % NSL, t == 0);
                __syncwarp();
                if (!(ok = warp_wait(BAR(B_PFULL + 1), t & 1, abort_flag))) break;
                tc_fence_after();
                issue_pv(1, vi % NSL, t == 0);
                tc_commit_elect(BAR(B_SLOTE + vi % NSL));
                __syncwarp();
            }
        } else {
            // PV_g only for the tiles Q tile g needs; P-full waits and the
            // accumulate flag count that group's own products
            StepCursor cv;
            cv.start((ok && *tab_ok) ? step_tab : nullptr, args.num_steps);
            int kv0 = 0, kv1 = 0;         // PV products issued per Q tile
#pragma unroll 1
            for (int t = 0; ok && t < T; ++t) {
                const bool has_next = t + 1 < T;
                const int vi = has_next ? 2 * t + 2 : 2 * t + 1; // load index of V(t)
                if (!(ok = warp_wait(BAR(B_SLOTF + vi % NSL), (vi / NSL) & 1, abort_flag))) break;
                if (cv.need(0)) {
                    if (!(ok = warp_wait(BAR(B_PFULL + 0), kv0 & 1, abort_flag))) break;
                    tc_fence_after();
                    issue_pv(0, vi % NSL, kv0 == 0);
                    ++kv0;
                    __syncwarp();
                }
                if (cv.need(1)) {
                    if (!(ok = warp_wait(BAR(B_PFULL + 1), kv1 & 1, abort_flag))) break;
                    tc_fence_after();
                    issue_pv(1, vi % NSL, kv1 == 0);
                    ++kv1;
                }
                tc_commit_elect(BAR(B_SLOTE + vi % NSL));
                __syncwarp();
                cv.next();
            }
        }
        if (!ok && lane == 0) record_timeout(args.status, abort_flag);
        // every MMA this warp issued has finished before tensor memory is freed
        __syncwarp();
        tc_commit_elect(BAR(B_FINAL));
        __syncwarp();
        volatile int never = 0;
        mbar_wait(BAR(B_FINAL), 0, &never);
    } else if (warp < 4) {
        regs_shrink<LOW_REGS>();
    } else {
        // ================================================= softmax
        regs_grow<216>();
        if (TWO_ISSUERS && warp == 4) {
            // the number of key tiles of the walk, one ring step per lane, for
            // the two MMA issuers (the S issuer waits for it before S(0)).  The
            // tile-skipping variant also writes the step table: for each ring
            // step (one lane per step) the unit's key-tile range and each Q
            // tile's own range inside it, from its first row's sequence start
            // to its last row (or that row's sequence end without the causal
            // mask).  Past kMaxSteps steps there is no table and every tile
            // counts for both Q tiles.
            int T = 0;
            bool have_tab = false;
            if constexpr (SKIP) have_tab = args.num_steps <= L::kMaxSteps;
            if (have_tab) {
                int64_t glo_pos[2], ghi_pos[2];
                bool gvalid[2];
#pragma unroll
                for (int gg = 0; gg < 2; ++gg) {
                    const int fr = row0 + 128 * gg, lrow = min(S, fr + 128) - 1;
                    gvalid[gg] = fr < S;
                    int64_t unused;
                    row_key_bounds(args.cu_seqlens, args.n_seqs, (int64_t)N * S,
                                   token_pos(args.layout, q_rank, gvalid[gg] ? fr : 0, N, S), args.causal,
                                   glo_pos[gg], unused);
                    row_key_bounds(args.cu_seqlens, args.n_seqs, (int64_t)N * S,
                                   token_pos(args.layout, q_rank, gvalid[gg] ? lrow : 0, N, S), args.causal,
                                   unused, ghi_pos[gg]);
                }
                for (int s0 = 0; s0 < args.num_steps; s0 += 32) {
                    const int st = s0 + lane;
                    int cnt = 0;
                    if (st < args.num_steps) {
                        const int j = walk0.kv_fixed >= 0 ? walk0.kv_fixed
                                                          : ((q_rank - st - walk0.step_base) % N + N) % N;
                        int e[6];
                        step_tile_ranges(args.layout, N, S, j, walk0.lo_pos, walk0.hi_pos, glo_pos, ghi_pos,
                                         gvalid, e);
#pragma unroll
                        for (int c = 0; c < 6; ++c) step_tab[6 * st + c] = e[c];
                        cnt = e[1] - e[0];
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
                    T += cnt;
                }
            } else {
                // one lane per ring step, summed over the warp
                for (int s0 = 0; s0 < args.num_steps; s0 += 32) {
                    int cnt = s0 + lane < args.num_steps ? walk0.step_tiles(s0 + lane) : 0;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
                    T += cnt;
                }
            }
            __syncwarp();
            if (lane == 0) {
                *tile_count = T;
                if constexpr (SKIP) *tab_ok = have_tab ? 1 : 0;
                mbar_arrive(BAR(B_TCOUNT));
            }
            __syncwarp();
        }
        const int g = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;                 // row inside Q tile g (= TMEM lane)
        const int a = row0 + g * 128 + r;             // local query row in the shard
        const int a_c = a < S ? a : S - 1;
        const int64_t my_pos = token_pos(args.layout, q_rank, a_c, N, S);
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + g * 128;
        const uint32_t tO = tmem + lane_off + 256 + g * D;
        const float sl2 = args.scale_log2;

        float m_ref = 0.f;        // reference point of the exponentials (log2 units)
        float l = 0.f;            // running denominator, relative to m_ref
        float lr = 0.f;           // the same sum over the bf16-rounded P the MMA uses
        int64_t my_lo_pos, my_hi_pos;
        row_key_bounds(args.cu_seqlens, args.n_seqs, (int64_t)N * S, my_pos, args.causal, my_lo_pos, my_hi_pos);
        TileWalk w = walk0;
        w.start_step();
        int t = 0;              // key tiles this Q tile has processed
        bool ok = true;
        bool have_tab = false;  // tile skipping: the step table was written
        if constexpr (SKIP) {
            ok = warp_wait(BAR(B_TCOUNT), 0, abort_flag);
            have_tab = ok && *tab_ok != 0;
        }
        int cur_step = -1;
        int klo = 0, khi = S;   // this row's visible local keys [klo, khi) of shard w.j
        // (t counts the tiles processed: without skipping, every tile the walk visits)
        for (; (!SKIP || ok) && w.valid(); w.next(), t += SKIP ? 0 : 1) {
            if (w.step != cur_step) {
                cur_step = w.step;
                klo = (int)keys_upto(args.layout, w.j, my_lo_pos, N, S);
                khi = (int)keys_upto(args.layout, w.j, my_hi_pos, N, S);
            }
            // a tile no row of this Q tile sees (the tiles of shard w.j it
            // sees are [e[0], e[1])): the MMA issuers skip its S and PV too
            if (SKIP && have_tab) {
                const int *e = step_tab + 6 * w.step + 2 + 2 * g;
                if (w.tile < e[0] || w.tile >= e[1]) continue;
            }
            if (!(ok = warp_wait(BAR(B_SFULL + g), t & 1, abort_flag))) break;
            tc_fence_after();
            const int lim = khi - w.tile * 128;       // columns [lim_lo, lim) are visible
            const int lim_lo = klo - w.tile * 128;
            const bool partial = lim < 128 || lim_lo > 0;
            uint32_t sr[4][32];
            auto load_s = [&]() {
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sr[q]);
                tmem_wait_ld();
                if (__any_sync(0xffffffffu, partial)) {
                    // the warp's rows see columns [lim_lo, lim) each; a 32-column
                    // chunk inside [largest lim_lo, smallest lim) is visible to
                    // every row of the warp and needs no mask (a warp's limits
                    // differ by about one column per row, so at most two chunks
                    // of a tile are masked element by element)
                    const int hi_min = (int)__reduce_min_sync(0xffffffffu, (unsigned)min(max(lim, 0), 128));
                    const int lo_max = (int)__reduce_max_sync(0xffffffffu, (unsigned)min(max(lim_lo, 0), 128));
                    float *s = reinterpret_cast<float *>(&sr[0][0]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (32 * q >= lo_max && 32 * q + 32 <= hi_min) continue;
#pragma unroll
                        for (int c = 32 * q; c < 32 * q + 32; ++c)
                            if (c >= lim || c < lim_lo) s[c] = -INFINITY;
                    }
                }
            };
            // P is computed against the current reference point and kept in
            // registers until the row's denominator has been checked; only
            // when it would leave [kSumLo, kSumHi] (or is not a number) does the
            // warp reload S (still intact in tensor memory), move the
            // reference to max(tile max, reference + log2 l) -- the sum then
            // lies in [1, 129] -- rescale O, l and lr, and compute P again.
            uint32_t pr[4][16];
            float lt, lrt;
            auto p_pass = [&]() {
                const float *s = reinterpret_cast<const float *>(&sr[0][0]);
                const uint64_t sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(-m_ref, -m_ref);
                uint64_t lsum[4] = {0ull, 0ull, 0ull, 0ull};
                float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        float x0, x1;
                        f32x2_split(fma_f32x2(f32x2(s[32 * q + c], s[32 * q + c + 1]), sl2x2, negm2), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        lsum[(c >> 1) & 3] = add_f32x2(lsum[(c >> 1) & 3], f32x2(p0, p1));
                        const uint32_t pk = pack_bf16x2(p0, p1);
                        pr[q][c >> 1] = pk;
                        rs[(c >> 1) & 3] = add_bf16x2_to_f32(rs[(c >> 1) & 3], pk);
                    }
                }
                float a0, a1, b0, b1, c0, c1, d0, d1;
                f32x2_split(lsum[0], a0, a1);
                f32x2_split(lsum[1], b0, b1);
                f32x2_split(lsum[2], c0, c1);
                f32x2_split(lsum[3], d0, d1);
                lt = ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
                lrt = (rs[0] + rs[1]) + (rs[2] + rs[3]);
            };
            load_s();
            p_pass();
            {
                const float ln = l + lt;
                const bool bad = !(ln >= kSumLo && ln <= kSumHi);
                if (__builtin_expect(__any_sync(0xffffffffu, bad), 0)) {
                    load_s();
                    const float *s = reinterpret_cast<const float *>(&sr[0][0]);
                    float mA = s[0], mB = s[1];
#pragma unroll
                    for (int c = 2; c < 128; c += 4) {
                        mA = max3(mA, s[c], s[c + 1]);
                        mB = max3(mB, s[c + 2], s[c + 3]);
                    }
                    float m_new = m_ref;
                    if (bad) {
                        const float cand = fmaxf(fmaxf(mA, mB) * sl2, l > 0.f ? m_ref + lg2(l) : -INFINITY);
                        if (cand != -INFINITY) m_new = cand;
                    }
                    const float alpha = ex2(m_ref - m_new);
                    l *= alpha;
                    lr *= alpha;
                    m_ref = m_new;
                    // O holds PV of every earlier tile once PV_g(t-1) is done;
                    // the whole warp takes part in the reload
                    if (t > 0) {
                        if (!(ok = warp_wait(BAR(B_PVDONE + g), (t - 1) & 1, abort_flag))) break;
                        tc_fence_after();
#pragma unroll 1
                        for (int q = 0; q < D / 16; ++q) {
                            uint32_t o[16];
                            tmem_ld16(tO + q * 16, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                            tmem_st16(tO + q * 16, o);
                        }
                        // PV_g(t) accumulates into O only after P full, which
                        // follows the fence below
                        tmem_wait_st();
                    }
                    p_pass();
                }
            }
            l += lt;
            lr += lrt;
            // S_g(t) is no longer needed: the next S_g may overwrite it
            tc_fence_before();
            mbar_arrive(BAR(B_SFREE + g));
            // P_g(t) goes to shared memory -- the K-major A operand of PV in the
            // 128-byte-swizzled layout a TMA box load would give (16-byte chunk
            // j of row r at chunk j ^ (r mod 8); keys 0-63 in the first box) --
            // or, at d = 64, to its tensor-memory columns, once PV_g(t-1) has
            // read P_g(t-1) there
            if (t > 0 && !(ok = warp_wait(BAR(B_PVDONE + g), (t - 1) & 1, abort_flag))) break;
            if constexpr (P_IN_TMEM) {
                // the row's 128 keys as 64 packed columns (key c in the low half
                // of column c / 2), the layout a TS product reads A in
                const uint32_t tP = tmem + lane_off + 384 + g * 64;
                tmem_st32(tP, *reinterpret_cast<const uint32_t(*)[32]>(&pr[0][0]));
                tmem_st32(tP + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pr[2][0]));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(BAR(B_PFULL + g));
                if constexpr (SKIP) ++t;
                continue;
            }
            {
                // row base (1024-byte aligned group + 128 bytes per row) and the
                // row's chunk swizzle; both are recomputed every tile rather than
                // kept live across the loop
                uint32_t xr = (uint32_t)(r & 7) << 4;
                asm volatile("" : "+r"(xr));
                const uint32_t prow = s_base + L::kP + g * 2 * L::kBox + (r >> 3) * 1024 + xr * 8;
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t off = (q >> 1) * L::kBox + ((((q & 1) * 4 + m) << 4) ^ xr);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + off),
                                     "r"(pr[q][4 * m]), "r"(pr[q][4 * m + 1]), "r"(pr[q][4 * m + 2]),
                                     "r"(pr[q][4 * m + 3])
                                     : "memory");
                    }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(BAR(B_PFULL + g));
            if constexpr (SKIP) ++t;
        }
        const int T = t;
        if (!ok) {
            if (lane == 0) record_timeout(args.status, abort_flag);
        } else if (T > 0) {
            ok = warp_wait(BAR(B_PVDONE + g), (T - 1) & 1, abort_flag);
            if (!ok && lane == 0) record_timeout(args.status, abort_flag);
            tc_fence_after();
        }
        // O_g / l goes out through shared memory and TMA: staged in this
        // group's P buffer (and, for fp32 O at d = 128, its Q tile), both free
        // once PV_g(T-1) is done, as boxes of 128 rows x 128 bytes in the
        // 128-byte swizzle (16-byte chunk j of row r at chunk j ^ (r mod 8)).
        // A unit that sees no key writes O = 0.  Every warp of the group
        // reaches the barrier; after a timeout nothing is stored.
        constexpr int CPB = OUT_F32 ? 32 : 64;       // O columns per box
        constexpr int NBOX = D / CPB;
        auto box_addr = [&](int bx) -> uint32_t {
            return bx < 2 ? s_base + L::kP + g * 2 * L::kBox + bx * L::kBox
                          : s_base + L::kQ + g * L::kTile + (bx - 2) * L::kBox;
        };
        const float inv_l = lr > 0.f ? 1.f / lr : 0.f;
        if (ok) {
            const uint32_t xr = (uint32_t)(r & 7) << 4;
            const uint32_t row_off = (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                if (T > 0) {
                    tmem_ld32(tO + q * 32, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = 0u;
                }
                if (OUT_F32) {
                    // 32 columns = one box, eight 16-byte chunks
                    const uint32_t row = box_addr(q) + row_off;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((uint32_t)c << 4) ^ xr)),
                                     "f"(__uint_as_float(o[4 * c]) * inv_l), "f"(__uint_as_float(o[4 * c + 1]) * inv_l),
                                     "f"(__uint_as_float(o[4 * c + 2]) * inv_l), "f"(__uint_as_float(o[4 * c + 3]) * inv_l)
                                     : "memory");
                } else {
                    // 32 columns = half a box, four 16-byte chunks
                    const uint32_t row = box_addr(q >> 1) + row_off;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t w0 = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv_l, __uint_as_float(o[8 * c + 1]) * inv_l);
                        const uint32_t w1 = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv_l, __uint_as_float(o[8 * c + 3]) * inv_l);
                        const uint32_t w2 = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv_l, __uint_as_float(o[8 * c + 5]) * inv_l);
                        const uint32_t w3 = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv_l, __uint_as_float(o[8 * c + 7]) * inv_l);
                        const uint32_t chunk = (uint32_t)((q & 1) * 4 + c);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((chunk << 4) ^ xr)),
                                     "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                                     : "memory");
                    }
                }
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        named_barrier_sync(1 + g, 128);
        if (wq == 0 && lane == 0 && *abort_flag == 0) {
            // rows past the shard's end fall outside the tensor and are not written
            int c1, c2, c3;
            tile_coords(args.seq_order, args.layout, args.S, args.N, ring ? qi : 0, b, row0 + 128 * g, c1, c2, c3);
#pragma unroll
            for (int bx = 0; bx < NBOX; ++bx) tma_store_4d(&tmo, box_addr(bx), h * D + bx * CPB, c1, c2, c3);
            tma_store_commit();
            tma_store_wait_read();
        }
        if (ok && a < S) {
            // shard stacks: [N or 1, B, H, S]; sequence order: [B, H, L] at the row's position
            const size_t at = args.seq_order ? ((size_t)b * H + h) * ((size_t)N * S) + (size_t)my_pos
                                             : ((size_t)zq * H + h) * S + a;
            args.lse[at] = l > 0.f ? (m_ref + lg2(l)) * 0.6931471805599453f : -INFINITY;
        }
    }

    // ---- teardown: every role is here, all tensor-core work has finished
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// [Z, S, H*d] bf16 (or fp32) viewed as a 3-D tensor, boxes of 128 rows x
// 128 bytes (64 bf16 or 32 fp32 columns) with the 128-byte swizzle the MMA
// descriptors and the O staging expect.
// The 4-D view tile_view describes, for a [..., heads * d] tensor of the
// launch, with a box of 128 bytes of columns by 128 rows and the 128-byte
// swizzle the operand descriptors expect.
static bool make_map(CUtensorMap *map, const void *base, const AttnLaunch &a, int64_t heads, int d,
                     bool f32 = false) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t esz = f32 ? 4 : 2;
    const TileView tv = tile_view(a.seq_order, a.layout, a.S, a.B, a.N, a.ring ? a.N : 1, heads * d);
    cuuint64_t dims[4] = {(cuuint64_t)(heads * d), (cuuint64_t)tv.n[0], (cuuint64_t)tv.n[1], (cuuint64_t)tv.n[2]};
    cuuint64_t strides[3] = {(cuuint64_t)tv.st[0] * esz, (cuuint64_t)tv.st[1] * esz, (cuuint64_t)tv.st[2] * esz};
    cuuint32_t box[4] = {(cuuint32_t)(128 / esz), tv.row_dim == 0 ? 128u : 1u, tv.row_dim == 1 ? 128u : 1u, 1u};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                     const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, bool F32, bool SKIP>
static ra_status launch_t(const AttnLaunch &a, const AttnArgs &args, int64_t grid, cudaStream_t stream,
                          const char **err) {
    CUtensorMap mq, mk, mv, mo;
    const int64_t Hkv = a.H_kv > 0 ? a.H_kv : a.H;
    if (!make_map(&mq, a.q, a, a.H, D) || !make_map(&mk, a.k, a, Hkv, D) || !make_map(&mv, a.v, a, Hkv, D) ||
        !make_map(&mo, a.o, a, a.H, D, F32)) {
        *err = "cuTensorMapEncodeTiled failed for the q/k/v/o tensor maps";
        return RA_ERR_CUDA;
    }
    auto kern = attn_fwd_kernel<D, F32, SKIP>;
    const int smem = (int)(SKIP ? AttnSmem<D>::kBytesSkip : AttnSmem<D>::kBytes);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
        *err = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize) failed";
        return RA_ERR_CUDA;
    }
    kern<<<(unsigned)grid, 384, smem, stream>>>(mq, mk, mv, mo, args);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = cudaGetErrorString(e);
        return RA_ERR_CUDA;
    }
    return RA_OK;
}

ra_status launch_attention(const AttnLaunch &a, cudaStream_t stream, const char **err) {
    AttnArgs args;
    args.o = a.o;
    args.lse = a.lse;
    args.status = a.status;
    args.B = (int)a.B;
    args.S = (int)a.S;
    args.H = (int)a.H;
    args.N = a.N;
    args.layout = a.layout;
    args.causal = a.causal ? 1 : 0;
    const float scale = a.scale > 0.f ? a.scale : 1.0f / std::sqrt((float)a.d);
    args.scale_log2 = scale * 1.4426950408889634f;
    args.num_q_ranks = a.ring ? a.N : 1;
    args.q_rank_fixed = a.ring ? -1 : a.q_rank;
    args.kv_rank_fixed = a.ring ? -1 : a.kv_rank;
    args.num_steps = (a.ring && a.ring_step < 0) ? a.N : 1;
    args.step_base = a.ring_step < 0 ? 0 : a.ring_step;
    args.n_units_seq = (int)((a.S + 255) / 256);
    args.inject_stall = a.inject_stall ? 1 : 0;
    args.kv_group = (int)(a.H / (a.H_kv > 0 ? a.H_kv : a.H));
    args.cu_seqlens = a.cu_seqlens;
    args.n_seqs = a.n_seqs;
    // keys + values one query head sweeps, shared by the heads of a GQA group;
    // a chunk holds about 48 MB of them by default (L2 holds 129 MB)
    args.bh_chunk = chunk_pairs(2 * (a.ring ? a.N : 1) * a.S * a.d * 2 / args.kv_group, a.B * a.H);
    args.seq_order = a.seq_order ? 1 : 0;
    const int64_t grid = (int64_t)args.num_q_ranks * args.n_units_seq * a.B * a.H;
    if (grid == 0) return RA_OK;
    if (grid > 0x7fffffffLL) {
        *err = "too many query tiles for one launch";
        return RA_ERR_UNSUPPORTED;
    }
    // Packed sequences in the striped layout take the tile-skipping variant
    // (d = 128): there a unit's 256 rows span N x 256 positions, many short
    // sequences, and each Q tile sees few of the tiles the unit visits.
    // Elsewhere skipping removes little work and measured slower (zigzag
    // packed sequences too).
    const bool skip = a.d == 128 && a.cu_seqlens != nullptr && a.layout == RA_STRIPED;
    if (skip)
        return a.out_f32 ? launch_t<128, true, true>(a, args, grid, stream, err)
                         : launch_t<128, false, true>(a, args, grid, stream, err);
    if (a.d == 128)
        return a.out_f32 ? launch_t<128, true, false>(a, args, grid, stream, err)
                         : launch_t<128, false, false>(a, args, grid, stream, err);
    return a.out_f32 ? launch_t<64, true, false>(a, args, grid, stream, err)
                     : launch_t<64, false, false>(a, args, grid, stream, err);
}

}  // namespace ra
