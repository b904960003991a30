// Test helper, not part of the library: runs the attention kernels' own unit
// decode and key-tile walks (ra_positions.cuh: decode_unit, unit_walk,
// row_key_bounds, step_tile_ranges for the forward and the dQ pass;
// decode_key_block, key_block_walk, col_query_bounds for the dK / dV pass) on
// the host, and records for every query row which keys of every shard they
// make it visit once the in-tile mask is applied.  The CPU test compares that
// with the keys the layout's token positions allow.
#include <cstring>
#include <vector>

#include "ra_positions.cuh"

namespace {

// One unit's contribution: for each row a in [row0, row_end) and every tile of
// shard j the walk (or, with a step table, the row's Q tile) visits, the keys
// [max(klo, 128 t), min(khi, 128 t + 128)) the row's mask lets through are
// counted in cnt[(q_rank * S + a) * N + j]; klo / khi are recorded in lo / hi.
// A (row, shard, tile) visited twice by the launches of one unit sets *dup
// (the caller clears `seen` per unit).
struct Recorder {
    int N, S;
    int *lo, *hi, *cnt;
    std::vector<unsigned char> seen;   // (row, shard, tile) visits of the current unit
    int tiles;
    int *dup;
};

void record_unit(Recorder &rc, int layout, int causal, const int *cu, int n_seqs, int q_rank, int kv_fixed,
                 int num_steps, int step_base, int row0, int row_end, int skip) {
    const int N = rc.N, S = rc.S;
    const int64_t total = (int64_t)N * S;
    ra::TileWalk walk0 = ra::unit_walk(layout, N, S, q_rank, kv_fixed, num_steps, step_base, row0, row_end,
                                       causal, cu, n_seqs);
    // the tile-skipping variant's table (at most 64 steps; otherwise every tile)
    const bool have_tab = skip && num_steps <= 64;
    int64_t glo[2], ghi[2];
    bool gvalid[2];
    for (int g = 0; g < 2; ++g) {
        const int fr = row0 + 128 * g, lrow = (fr + 128 < S ? fr + 128 : S) - 1;
        gvalid[g] = fr < S;
        int64_t unused;
        ra::row_key_bounds(cu, n_seqs, total, ra::token_pos(layout, q_rank, gvalid[g] ? fr : 0, N, S), causal,
                           glo[g], unused);
        ra::row_key_bounds(cu, n_seqs, total, ra::token_pos(layout, q_rank, gvalid[g] ? lrow : 0, N, S), causal,
                           unused, ghi[g]);
    }
    // the per-step tile counts the forward's issuers are given agree with the walk
    int visited = 0, counted = 0;
    for (int s = 0; s < num_steps; ++s) counted += walk0.step_tiles(s);
    ra::TileWalk w = walk0;
    for (w.start_step(); w.valid(); w.next()) {
        ++visited;
        int e[6];
        if (have_tab) ra::step_tile_ranges(layout, N, S, w.j, walk0.lo_pos, walk0.hi_pos, glo, ghi, gvalid, e);
        for (int a = row0; a < row_end; ++a) {
            const int g = (a - row0) >> 7;
            if (have_tab && (w.tile < e[2 + 2 * g] || w.tile >= e[3 + 2 * g])) continue;
            int64_t lo_pos, hi_pos;
            ra::row_key_bounds(cu, n_seqs, total, ra::token_pos(layout, q_rank, a, N, S), causal, lo_pos, hi_pos);
            const int klo = (int)ra::keys_upto(layout, w.j, lo_pos, N, S);
            const int khi = (int)ra::keys_upto(layout, w.j, hi_pos, N, S);
            const size_t o = ((size_t)q_rank * S + a) * N + w.j;
            rc.lo[o] = klo;
            rc.hi[o] = khi;
            const int c0 = w.tile * 128 > klo ? w.tile * 128 : klo;
            const int c1 = w.tile * 128 + 128 < khi ? w.tile * 128 + 128 : khi;
            if (c1 > c0) {
                rc.cnt[o] += c1 - c0;
                unsigned char &s = rc.seen[((size_t)(a - row0) * N + w.j) * rc.tiles + w.tile];
                if (s) *rc.dup = 1;
                s = 1;
            }
        }
    }
    if (visited != counted) *rc.dup = 2;
}

}  // namespace

// The forward (and the dQ pass, unit_rows = 128) over one (batch, head) pair's
// N x S query rows.  mode 0: one fused launch (num_steps = N); mode 1: the
// stepwise sweep, N launches of one step each (step_base = s); mode 2: the
// block calls, one launch per (query rank, key/value rank).  skip: the
// tile-skipping variant's per-Q-tile table (unit_rows = 256 only).
// lo, hi, cnt: [N, S, N] ints (cnt zero-filled by the caller); lo / hi are
// the row's mask bounds for that shard, -1 where the shard was never visited.
// coverage: [B * H * N * n_units] ints, how often decode_unit hands out each
// unit across the whole grid.  Returns 0, or -1 on a bad argument.
extern "C" int ra_test_forward_walk(int layout, int N, int S, int causal, const int *cu, int n_seqs, int mode,
                                    int unit_rows, int skip, int B, int H, int bh_chunk, int *lo, int *hi, int *cnt,
                                    int *coverage, int *dup) {
    if (N < 1 || S < 1 || (unit_rows != 128 && unit_rows != 256)) return -1;
    const int n_units = (S + unit_rows - 1) / unit_rows;
    const int tiles = (S + 127) / 128;
    Recorder rc{N, S, lo, hi, cnt, std::vector<unsigned char>((size_t)unit_rows * N * tiles), tiles, dup};
    for (size_t i = 0; i < (size_t)N * S * N; ++i) lo[i] = hi[i] = -1;
    *dup = 0;
    // the launch grid: every unit of every rank, batch and head, as decode_unit hands them out
    const int grid = N * n_units * B * H;
    std::memset(coverage, 0, sizeof(int) * (size_t)grid);
    for (int blk = 0; blk < grid; ++blk) {
        const ra::UnitId u = ra::decode_unit(blk, bh_chunk, B, H, N, n_units, layout);
        if (u.b < 0 || u.b >= B || u.h < 0 || u.h >= H || u.qi < 0 || u.qi >= N || u.qt < 0 || u.qt >= n_units)
            return -1;
        ++coverage[((u.b * H + u.h) * N + u.qi) * n_units + u.qt];
        if (u.b != 0 || u.h != 0) continue;   // the walk does not depend on the pair
        const int row0 = u.qt * unit_rows;
        const int row_end = row0 + unit_rows < S ? row0 + unit_rows : S;
        std::fill(rc.seen.begin(), rc.seen.end(), 0);
        if (mode == 0) {
            record_unit(rc, layout, causal, cu, n_seqs, u.qi, -1, N, 0, row0, row_end, skip);
        } else if (mode == 1) {
            for (int s = 0; s < N; ++s) record_unit(rc, layout, causal, cu, n_seqs, u.qi, -1, 1, s, row0, row_end, skip);
        } else {
            for (int j = 0; j < N; ++j) record_unit(rc, layout, causal, cu, n_seqs, u.qi, j, 1, 0, row0, row_end, skip);
        }
    }
    return 0;
}

// The dK / dV pass over one (batch, key/value head) pair: every 128-key block
// of every rank, as decode_key_block hands them out, walks the query tiles of
// `heads` query heads.  For key row c of rank kj and query rank i:
// lo / hi the key's query bounds (-1 where shard i was never visited) and cnt
// the queries its tiles reach under the mask, per head -- [heads, N, S, N].
// coverage: [B * Hkv * N * n_blocks].  Returns 0, or -1 on a bad argument.
extern "C" int ra_test_key_walk(int layout, int N, int S, int causal, const int *cu, int n_seqs, int heads, int B,
                                int Hkv, int bh_chunk, int *lo, int *hi, int *cnt, int *coverage, int *dup) {
    if (N < 1 || S < 1 || heads < 1) return -1;
    const int n_blocks = (S + 127) / 128;
    const int64_t total = (int64_t)N * S;
    const size_t per_head = (size_t)N * S * N;
    for (size_t i = 0; i < per_head * heads; ++i) lo[i] = hi[i] = -1;
    *dup = 0;
    const int grid = N * n_blocks * B * Hkv;
    std::memset(coverage, 0, sizeof(int) * (size_t)grid);
    std::vector<unsigned char> seen((size_t)128 * heads * N * n_blocks);
    for (int blk = 0; blk < grid; ++blk) {
        const ra::UnitId u = ra::decode_key_block(blk, bh_chunk, B, Hkv, N, n_blocks, layout);
        if (u.b < 0 || u.b >= B || u.h < 0 || u.h >= Hkv || u.qi < 0 || u.qi >= N || u.qt < 0 || u.qt >= n_blocks)
            return -1;
        ++coverage[((u.b * Hkv + u.h) * N + u.qi) * n_blocks + u.qt];
        if (u.b != 0 || u.h != 0) continue;
        const int kj = u.qi, c0 = u.qt * 128, c_end = c0 + 128 < S ? c0 + 128 : S;
        std::fill(seen.begin(), seen.end(), 0);
        ra::QWalk w = ra::key_block_walk(layout, N, S, kj, heads, c0, c_end, causal, cu, n_seqs);
        for (w.start(); w.valid(); w.next()) {
            for (int c = c0; c < c_end; ++c) {
                int64_t lo_pos, hi_pos;
                ra::col_query_bounds(cu, n_seqs, total, ra::token_pos(layout, kj, c, N, S), causal, lo_pos, hi_pos);
                const int qlo = (int)ra::keys_upto(layout, w.i, lo_pos, N, S);
                const int qhi = (int)ra::keys_upto(layout, w.i, hi_pos, N, S);
                const size_t o = per_head * w.head + ((size_t)kj * S + c) * N + w.i;
                lo[o] = qlo;
                hi[o] = qhi;
                const int r0 = w.tile * 128 > qlo ? w.tile * 128 : qlo;
                const int r1 = w.tile * 128 + 128 < qhi ? w.tile * 128 + 128 : qhi;
                if (r1 > r0) {
                    cnt[o] += r1 - r0;
                    unsigned char &s = seen[(((size_t)(c - c0) * heads + w.head) * N + w.i) * n_blocks + w.tile];
                    if (s) *dup = 1;
                    s = 1;
                }
            }
        }
    }
    return 0;
}
