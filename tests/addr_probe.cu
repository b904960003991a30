// Test helper, not part of the library: evaluates the attention kernels'
// token-order tile addressing (tile_view on the host side, tile_coords on the
// device side; both are plain integer functions) on the host, so that a CPU
// test can compare every row's address with the layout's token position.
#include "ra_positions.cuh"

// For every rank r < N, batch b < B and local row s < S_pad (S rounded up to
// a whole 128-row tile): the element offset of row s of rank r's shard in the
// token-order tensor [B, L, cols], reached as tile (s - s % 128) plus s % 128
// rows along the view's row dimension, and whether every coordinate lies
// inside the view.  Results at index (r * B + b) * S_pad + s.
extern "C" int ra_test_token_offsets(int layout, int N, int64_t S, int B, int64_t cols, int64_t *off,
                                     unsigned char *inside) {
    const int64_t S_pad = (S + 127) / 128 * 128;
    const ra::TileView tv = ra::tile_view(true, layout, S, B, N, N, cols);
    for (int r = 0; r < N; ++r)
        for (int b = 0; b < B; ++b)
            for (int64_t s = 0; s < S_pad; ++s) {
                int c[3];
                const int row0 = (int)(s - s % 128);
                ra::tile_coords(1, layout, (int)S, N, r, b, row0, c[0], c[1], c[2]);
                c[tv.row_dim] += (int)(s % 128);
                int64_t o = 0;
                bool in = true;
                for (int i = 0; i < 3; ++i) {
                    o += (int64_t)c[i] * tv.st[i];
                    in = in && c[i] >= 0 && c[i] < tv.n[i];
                }
                off[((int64_t)r * B + b) * S_pad + s] = o;
                inside[((int64_t)r * B + b) * S_pad + s] = in ? 1 : 0;
            }
    return 0;
}
