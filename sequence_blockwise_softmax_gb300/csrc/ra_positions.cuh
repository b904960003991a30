// ra_positions.cuh -- token positions and visible-key counts shared by the
// forward and backward attention kernels.
#pragma once
#include <cstdint>

#include "ra_internal.h"

namespace ra {

// Global position of local token s on rank r (the layout formulas of the
// article's §3.1 contiguous split, §4 striped split and §6.1 zigzag split).
__device__ __forceinline__ int64_t token_pos(int layout, int r, int64_t s, int N, int64_t S) {
    if (layout == RA_CONTIGUOUS) return (int64_t)r * S + s;
    if (layout == RA_STRIPED) return s * N + r;
    const int64_t C = S >> 1;
    return s < C ? (int64_t)r * C + s : (int64_t)(2 * N - 1 - r) * C + (s - C);
}

__device__ __forceinline__ int64_t clamp64(int64_t x, int64_t lo, int64_t hi) {
    return x < lo ? lo : (x > hi ? hi : x);
}

// How many keys of rank j sit at global positions <= p.  Because positions
// increase along a rank's local order, these are local keys 0..result-1.
__device__ __forceinline__ int64_t keys_upto(int layout, int j, int64_t p, int N, int64_t S) {
    if (layout == RA_CONTIGUOUS) return clamp64(p - (int64_t)j * S + 1, 0, S);
    if (layout == RA_STRIPED) return p < j ? 0 : (((p - j) / N + 1) < S ? (p - j) / N + 1 : S);
    const int64_t C = S >> 1;
    return clamp64(p - (int64_t)j * C + 1, 0, C) + clamp64(p - (int64_t)(2 * N - 1 - j) * C + 1, 0, C);
}

// Packed variable-length sequences: the boundaries [start, end) of the
// sequence holding global position p (binary search; every read stays inside
// the n + 1 boundaries whatever they hold).  Without packing: [0, total).
__device__ __forceinline__ void seq_bounds(const int *cu, int n, int64_t total, int64_t p,
                                           int64_t &start, int64_t &end) {
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

// The sequence of (kv rank, key tile) pairs a unit visits.  The keys of
// shard j its rows may see are the local interval
// [keys_upto(j, lo_pos), keys_upto(j, hi_pos)): lo_pos is one before the
// start of the first row's sequence, hi_pos the last row's position (causal)
// or the end of its sequence minus one.  Every role walks it identically.
struct TileWalk {
    int step, tile, tile_end, j;
    int num_steps, step_base, q_rank, kv_fixed, N, layout, S;
    int64_t lo_pos, hi_pos;

    __device__ void start_step() {
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
    __device__ bool valid() const { return step < num_steps; }
    __device__ void next() {
        if (++tile >= tile_end) {
            ++step;
            start_step();
        }
    }
};

// The outer TMA coordinates (after the column) of local rows [row, row + 128)
// of rank `rank`'s shard of batch b, for the views tile_view describes.
// Shard stacks [N or 1, B, S, cols] are addressed (row, b, rank).  In token
// order the layout is the addressing: contiguous {S, N, B} (position r*S + s),
// striped {N, S, B} (position s*N + r, the row is the second coordinate),
// zigzag {C, 2N, B} with C = S/2 (rank r's rows are chunk r, then chunk
// 2N-1-r; C is a multiple of 128, so a 128-row tile never straddles the two).
// Rows past a shard's end fall outside the view: loads read zeros there and
// stores skip them.
__host__ __device__ __forceinline__ void tile_coords(int seq_order, int layout, int S, int N, int rank, int b,
                                                     int row, int &c1, int &c2, int &c3) {
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
