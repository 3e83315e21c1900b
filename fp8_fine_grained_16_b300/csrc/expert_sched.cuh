// expert_sched.cuh -- per-expert tile lists of the grouped (MoE) GEMMs.
//
// Expert e owns rows [off[e], off[e+1]) of A and D (the jp-study.kr page: each token's
// rows are dispatched to its routed experts).  A tile covers tile_rows rows
// (256 for a CTA pair, 128 for one CTA), so expert e needs
// ceil(rows_e / tile_rows) row tiles, each crossed with every column tile of
// the output.  Tiles are numbered expert by expert, and within an expert
// column tile by column tile with the row tiles innermost, so the tiles that
// stream one weight tile run next to each other.
#pragma once
#include "common.cuh"

namespace fp8bs {

constexpr int kMaxExperts = 1024;

// Offsets into shared memory and the exclusive prefix of row-tile counts,
// pre_s[e] = row tiles of the experts before e (pre_s[E] = all).  Every
// thread of the CTA calls it (it synchronises the CTA twice).  An expert
// whose offsets are not 0 <= off[e] <= off[e+1] <= total_rows gets no rows;
// the result is true in every thread when any offset breaks the rules,
// including off[0] != 0 or off[E] != total_rows.
FP8_DEV bool expert_tile_prefix(const int32_t* off, int E, int64_t total_rows, int32_t* off_s, int32_t* pre_s,
                                int tile_rows) {
    __shared__ int bad_s;
    for (int i = threadIdx.x; i <= E; i += blockDim.x) off_s[i] = __ldg(off + i);
    if (threadIdx.x == 0) bad_s = 0;
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        bool bad = false;
        int carry = 0;
        if (lane == 0) pre_s[0] = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            int cnt = 0;
            if (e < E) {
                const int64_t lo = off_s[e], hi = off_s[e + 1];
                const bool ok = lo >= 0 && lo <= hi && hi <= total_rows;
                bad |= !ok;
                cnt = ok ? int((hi - lo + tile_rows - 1) / tile_rows) : 0;
            }
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            if (e < E) pre_s[e + 1] = carry + incl;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        bad |= (lane == 0) && (off_s[0] != 0 || int64_t(off_s[E]) != total_rows);
        if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) bad_s = 1;
    }
    __syncthreads();
    return bad_s != 0;
}

struct ExpertTile {
    int64_t row0;            // first row of the tile (global row index)
    int64_t row_end;         // rows >= row_end belong to the next expert: not stored
    int64_t col_tile;        // column tile index
    int e;                   // expert
};

// Tile w of the list above (num_n column tiles per row tile).
FP8_DEV ExpertTile expert_tile(const int32_t* off_s, const int32_t* pre_s, int E, int64_t num_n, int64_t w,
                               int tile_rows) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (int64_t(pre_s[mid]) * num_n <= w) lo = mid; else hi = mid;
    }
    const int64_t mt2 = pre_s[lo + 1] - pre_s[lo];
    const int64_t local = w - int64_t(pre_s[lo]) * num_n;
    ExpertTile t;
    t.e = lo;
    t.col_tile = local / mt2;
    t.row0 = int64_t(off_s[lo]) + (local % mt2) * tile_rows;
    t.row_end = off_s[lo + 1];
    return t;
}

}  // namespace fp8bs
