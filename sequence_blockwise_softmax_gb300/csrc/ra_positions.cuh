// ra_positions.cuh -- token positions, visible-key counts, unit decode and the
// key-tile walk shared by the forward and backward attention kernels.
//
// Everything here is plain integer arithmetic callable from host and device,
// so that a CPU test can run the very walk the kernels run (tests/walk_probe.cu)
// and check the (query, key) pairs it visits against the layouts' token
// positions.
#pragma once
#include <cstdint>

#include "ra_internal.h"

#define RA_HD __host__ __device__ __forceinline__
// the walks' step changes: left to the compiler to inline or not, to keep the
// kernels' per-tile loops short
#define RA_HD_STEP __host__ __device__

namespace ra {

// Global position of local token s on rank r (the layout formulas of the
// article's §3.1 contiguous split, §4 striped split and §6.1 zigzag split).
RA_HD int64_t token_pos(int layout, int r, int64_t s, int N, int64_t S) {
    if (layout == RA_CONTIGUOUS) return (int64_t)r * S + s;
    if (layout == RA_STRIPED) return s * N + r;
    const int64_t C = S >> 1;
    return s < C ? (int64_t)r * C + s : (int64_t)(2 * N - 1 - r) * C + (s - C);
}

RA_HD int64_t clamp64(int64_t x, int64_t lo, int64_t hi) {
    return x < lo ? lo : (x > hi ? hi : x);
}

// How many keys of rank j sit at global positions <= p.  Because positions
// increase along a rank's local order, these are local keys 0..result-1.
// (The striped quotient is taken in 32 bits whenever it fits: a 64-bit
// division is several times longer, and the kernels evaluate this at every
// ring step of every row.)
RA_HD int64_t keys_upto(int layout, int j, int64_t p, int N, int64_t S) {
    if (layout == RA_CONTIGUOUS) return clamp64(p - (int64_t)j * S + 1, 0, S);
    if (layout == RA_STRIPED) {
        if (p < j) return 0;
        const int64_t q = p - j;
        const int64_t n = q <= 0x7fffffffLL ? (int64_t)((uint32_t)q / (uint32_t)N) + 1 : q / N + 1;
        return n < S ? n : S;
    }
    const int64_t C = S >> 1;
    return clamp64(p - (int64_t)j * C + 1, 0, C) + clamp64(p - (int64_t)(2 * N - 1 - j) * C + 1, 0, C);
}

// Packed variable-length sequences: the boundaries [start, end) of the
// sequence holding global position p (binary search; every read stays inside
// the n + 1 boundaries whatever they hold).  Without packing: [0, total).
RA_HD void seq_bounds(const int *cu, int n, int64_t total, int64_t p, int64_t &start, int64_t &end) {
    if (!cu) {
        start = 0;
        end = total;
        return;
    }
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)cu[mid] <= p) lo = mid;
        else hi = mid;
    }
    start = cu[lo];
    end = cu[lo + 1];
}

// The keys a query at global position p may see, as two positions: every key
// at a position in (lo_pos, hi_pos] -- after the start of p's sequence, and
// not after p (causal) or not past the end of p's sequence.  For shard j the
// visible local keys are then [keys_upto(j, lo_pos), keys_upto(j, hi_pos)).
RA_HD void row_key_bounds(const int *cu, int n, int64_t total, int64_t p, int causal, int64_t &lo_pos,
                          int64_t &hi_pos) {
    int64_t start, end;
    seq_bounds(cu, n, total, p, start, end);
    lo_pos = start - 1;
    hi_pos = causal ? p : end - 1;
}

// The sequence of (kv rank, key tile) pairs a unit visits.  The keys of
// shard j its rows may see are the local interval
// [keys_upto(j, lo_pos), keys_upto(j, hi_pos)): lo_pos is one before the
// start of the first row's sequence, hi_pos the last row's position (causal)
// or the end of its sequence minus one.  Every role walks it identically.
struct TileWalk {
    int step, tile, tile_end, j;
    int num_steps, step_base, q_rank, kv_fixed, N, layout, S;
    int64_t lo_pos, hi_pos;

    RA_HD_STEP void start_step() {
        while (step < num_steps) {
            j = kv_fixed >= 0 ? kv_fixed : ((q_rank - step - step_base) % N + N) % N;
            const int64_t lo = keys_upto(layout, j, lo_pos, N, S);
            const int64_t hi = keys_upto(layout, j, hi_pos, N, S);
            tile = (int)(lo / 128);
            tile_end = (int)((hi + 127) / 128);
            if (tile_end > tile) return;
            ++step;
        }
    }
    RA_HD_STEP bool valid() const { return step < num_steps; }
    // The number of key tiles step s visits (0 when its shard has no visible
    // key): what start_step finds for that step, without walking to it.
    RA_HD int step_tiles(int s) const {
        const int js = kv_fixed >= 0 ? kv_fixed : ((q_rank - s - step_base) % N + N) % N;
        const int t0 = (int)(keys_upto(layout, js, lo_pos, N, S) / 128);
        const int t1 = (int)((keys_upto(layout, js, hi_pos, N, S) + 127) / 128);
        return t1 > t0 ? t1 - t0 : 0;
    }
    RA_HD_STEP void next() {
        if (++tile >= tile_end) {
            ++step;
            start_step();
        }
    }
};

// The walk of the unit holding local query rows [row0, row_end) of rank
// q_rank: ring steps step_base .. step_base + num_steps - 1, where step s
// meets key/value rank (q_rank - s) mod N, or one step against kv_fixed >= 0.
// Not yet started (call start_step()).
RA_HD TileWalk unit_walk(int layout, int N, int S, int q_rank, int kv_fixed, int num_steps, int step_base,
                         int row0, int row_end, int causal, const int *cu, int n_seqs) {
    TileWalk w;
    w.step = 0;
    w.tile = w.tile_end = w.j = 0;
    w.num_steps = num_steps;
    w.step_base = step_base;
    w.q_rank = q_rank;
    w.kv_fixed = kv_fixed;
    w.N = N;
    w.layout = layout;
    w.S = S;
    const int64_t total = (int64_t)N * S;
    int64_t first_lo, first_hi, last_lo, last_hi;
    row_key_bounds(cu, n_seqs, total, token_pos(layout, q_rank, row0, N, S), causal, first_lo, first_hi);
    row_key_bounds(cu, n_seqs, total, token_pos(layout, q_rank, row_end - 1, N, S), causal, last_lo, last_hi);
    w.lo_pos = first_lo;
    w.hi_pos = last_hi;
    return w;
}

// The queries a key at global position p is visible to: every query at a
// position in (lo_pos, hi_pos] -- not before p (causal) or from the start of
// p's sequence, up to the end of p's sequence.  For query shard i they are the
// local rows [keys_upto(i, lo_pos), keys_upto(i, hi_pos)).
RA_HD void col_query_bounds(const int *cu, int n, int64_t total, int64_t p, int causal, int64_t &lo_pos,
                            int64_t &hi_pos) {
    int64_t start, end;
    seq_bounds(cu, n, total, p, start, end);
    lo_pos = causal ? p - 1 : start - 1;
    hi_pos = end - 1;
}

// The query tiles a block of keys meets (the dK / dV pass), for each query
// head of its group and each query rank in ring order (j, j+1, ...): for keys
// whose visible queries lie at positions in (lo_pos, hi_pos] the visible
// queries of rank i are the local interval [keys_upto(i, lo_pos),
// keys_upto(i, hi_pos)).
struct QWalk {
    int head, step, tile, tile_end, i;
    int heads, N, j, layout, S;
    int64_t lo_pos, hi_pos;

    RA_HD_STEP void start() {
        while (head < heads) {
            while (step < N) {
                i = (j + step) % N;
                const int64_t lo = keys_upto(layout, i, lo_pos, N, S);
                const int64_t hi = keys_upto(layout, i, hi_pos, N, S);
                tile = (int)(lo / 128);
                tile_end = (int)((hi + 127) / 128);
                if (tile_end > tile) return;
                ++step;
            }
            step = 0;
            ++head;
        }
    }
    RA_HD_STEP bool valid() const { return head < heads; }
    RA_HD_STEP void next() {
        if (++tile >= tile_end) {
            ++step;
            start();
        }
    }
};

// The walk of the key block holding local keys [c0, c_end) of rank kj, over
// `heads` query heads.  Not yet started (call start()).
RA_HD QWalk key_block_walk(int layout, int N, int S, int kj, int heads, int c0, int c_end, int causal,
                           const int *cu, int n_seqs) {
    QWalk w;
    w.head = 0;
    w.step = 0;
    w.tile = w.tile_end = w.i = 0;
    w.heads = heads;
    w.N = N;
    w.j = kj;
    w.layout = layout;
    w.S = S;
    const int64_t total = (int64_t)N * S;
    int64_t first_lo, first_hi, last_lo, last_hi;
    col_query_bounds(cu, n_seqs, total, token_pos(layout, kj, c0, N, S), causal, first_lo, first_hi);
    col_query_bounds(cu, n_seqs, total, token_pos(layout, kj, c_end - 1, N, S), causal, last_lo, last_hi);
    w.lo_pos = first_lo;
    w.hi_pos = last_hi;
    return w;
}

// Which query unit a CTA of the forward (or the dQ pass) runs.  Causal work
// grows with position, so units run heavy first: the (batch, head) pairs are
// taken in chunks of bh_chunk whose keys and values fit in L2 together, and
// inside a chunk the units of all its pairs are interleaved, heaviest first,
// so that no pair's heavy units are left for the tail of the launch.
// n_units_seq units of rows per rank and (batch, head); num_q_ranks ranks.
struct UnitId {
    int b, h, qi, qt;
};
RA_HD UnitId decode_unit(int block, int bh_chunk, int B, int H, int num_q_ranks, int n_units_seq, int layout) {
    const int per_bh = num_q_ranks * n_units_seq;
    const int BH = B * H;
    const int per_chunk = bh_chunk * per_bh;
    const int chunk = block / per_chunk;
    const int c_first = chunk * bh_chunk;
    const int c_size = (bh_chunk < BH - c_first) ? bh_chunk : BH - c_first;
    const int idx = block - chunk * per_chunk;
    const int bh = c_first + idx % c_size;
    const int rem = idx / c_size;
    UnitId u;
    u.b = bh / H;
    u.h = bh % H;
    if (layout == RA_CONTIGUOUS) {
        u.qi = num_q_ranks - 1 - rem / n_units_seq;
        u.qt = n_units_seq - 1 - rem % n_units_seq;
    } else {
        u.qt = n_units_seq - 1 - rem / num_q_ranks;
        u.qi = num_q_ranks - 1 - rem % num_q_ranks;
    }
    return u;
}

// Which key block a CTA of the dK / dV pass runs: (batch, key/value head)
// pairs in chunks of bh_chunk as in decode_unit, and inside a chunk the
// blocks of all its pairs interleaved; causal work shrinks with the key
// position, so the earliest keys go first.  Returned as b, h (the key/value
// head), qi (the key rank) and qt (the 128-key block).
RA_HD UnitId decode_key_block(int block, int bh_chunk, int B, int Hkv, int N, int n_tiles_seq, int layout) {
    const int per_bh = N * n_tiles_seq;
    const int BH = B * Hkv;
    const int per_chunk = bh_chunk * per_bh;
    const int chunk = block / per_chunk;
    const int c_first = chunk * bh_chunk;
    const int c_size = (bh_chunk < BH - c_first) ? bh_chunk : BH - c_first;
    const int idx = block - chunk * per_chunk;
    const int bh = c_first + idx % c_size;
    const int rem = idx / c_size;
    UnitId u;
    u.b = bh / Hkv;
    u.h = bh % Hkv;
    if (layout == RA_CONTIGUOUS) {
        u.qi = rem / n_tiles_seq;
        u.qt = rem % n_tiles_seq;
    } else {
        u.qt = rem / N;
        u.qi = rem % N;
    }
    return u;
}

// The tile-skipping variant's table entry for ring step s against shard j:
// e[0], e[1] the unit's key-tile range [lo, hi) (the walk's), and for each
// 128-row Q tile g present (gvalid) the tiles it sees, e[2 + 2g] .. e[3 + 2g],
// clipped to the unit's range; an absent Q tile gets the empty range at lo.
// glo / ghi are the Q tile's key bounds (row_key_bounds of its first row's lo
// and its last row's hi).
RA_HD void step_tile_ranges(int layout, int N, int S, int j, int64_t unit_lo, int64_t unit_hi,
                            const int64_t glo[2], const int64_t ghi[2], const bool gvalid[2], int e[6]) {
    const int ulo = (int)(keys_upto(layout, j, unit_lo, N, S) / 128);
    int uhi = (int)((keys_upto(layout, j, unit_hi, N, S) + 127) / 128);
    if (uhi < ulo) uhi = ulo;
    e[0] = ulo;
    e[1] = uhi;
    for (int g = 0; g < 2; ++g) {
        e[2 + 2 * g] = ulo;
        e[3 + 2 * g] = ulo;
        if (gvalid[g]) {
            const int lo = (int)(keys_upto(layout, j, glo[g], N, S) / 128);
            const int hi = (int)((keys_upto(layout, j, ghi[g], N, S) + 127) / 128);
            const int a = lo > ulo ? lo : ulo;
            const int c = hi < uhi ? hi : uhi;
            e[2 + 2 * g] = a;
            e[3 + 2 * g] = c > a ? c : a;
        }
    }
}

// The outer TMA coordinates (after the column) of local rows [row, row + 128)
// of rank `rank`'s shard of batch b, for the views tile_view describes.
// Shard stacks [N or 1, B, S, cols] are addressed (row, b, rank).  In token
// order the layout is the addressing: contiguous {S, N, B} (position r*S + s),
// striped {N, S, B} (position s*N + r, the row is the second coordinate),
// zigzag {C, 2N, B} with C = S/2 (rank r's rows are chunk r, then chunk
// 2N-1-r; C is a multiple of 128, so a 128-row tile never straddles the two).
// Rows past a shard's end fall outside the view: loads read zeros there and
// stores skip them.
RA_HD void tile_coords(int seq_order, int layout, int S, int N, int rank, int b, int row, int &c1, int &c2,
                       int &c3) {
    if (!seq_order) {
        c1 = row;
        c2 = b;
        c3 = rank;
    } else if (layout == RA_STRIPED) {
        c1 = rank;
        c2 = row;
        c3 = b;
    } else if (layout == RA_ZIGZAG) {
        const int C = S >> 1;
        const bool hi = row >= C;
        c1 = hi ? row - C : row;
        c2 = hi ? 2 * N - 1 - rank : rank;
        c3 = b;
    } else {
        c1 = row;
        c2 = rank;
        c3 = b;
    }
}

}  // namespace ra
