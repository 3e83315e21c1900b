// tail_split.cuh -- which work a CTA pair of the dense promoted GEMM does.
//
// The GEMM's 256 x 256 tiles go to the pairs round-robin, each over the whole
// K.  When that leaves a last wave of at most half the pairs, the tiles of
// that wave are cut along K instead: tail tile j is computed as `split`
// K ranges, range s by pair j * split + s, after that pair's whole tiles;
// each range's fp32 sum goes to workspace slab j * split + s, and a fix-up
// kernel adds a tile's slabs in K order.  When every tile is split (fewer
// tiles than pairs), exactly one pair per K range is launched.
//
// The same functions serve the kernel (device) and the host (launch
// planning and the library's plan queries), so the host can check the
// enumeration the kernel walks.
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define FP8_HD __host__ __device__ __forceinline__
#else
#define FP8_HD inline
#endif

namespace fp8bs {

constexpr int kSplitMinKBlocks = 16;          // below this a split saves less than the fix-up costs

struct SplitPlan {
    int64_t split;       // K ranges per tail tile; 0: no split
    int64_t tail0;       // first split tile (tiles below it run over the whole K)
    int64_t pairs;       // pairs to launch (at most the pairs offered)
};

// num_tiles tiles of nkb K blocks on `pairs` pairs; `slabs` workspace slabs
// available (0: no workspace).
FP8_HD SplitPlan plan_tail_split(int64_t num_tiles, int64_t nkb, int64_t pairs, int64_t slabs) {
    SplitPlan p{0, num_tiles, pairs};
    const int64_t n_tail = num_tiles % pairs;
    if (slabs > 0 && nkb >= kSplitMinKBlocks && n_tail > 0 && 2 * n_tail <= pairs) {
        int64_t sp = pairs / n_tail;
        if (sp > nkb / 2) sp = nkb / 2;
        if (n_tail * sp <= slabs) {
            p.split = sp;
            p.tail0 = num_tiles - n_tail;
            if (p.tail0 == 0) p.pairs = n_tail * sp;          // every tile split: one pair per K range
        }
    }
    if (p.split == 0 && num_tiles < p.pairs) p.pairs = num_tiles;   // at most one pair per tile
    return p;
}

struct WorkUnit {
    int64_t w;           // tile
    int64_t kb0, kb1;    // K blocks [kb0, kb1)
    int64_t slab;        // < 0: whole tile, stored to D; else its workspace slab
};

// Units of pair `c` of `np` launched pairs: its whole tiles c, c + np, ...
// below the split tiles, then (under a split) one K range of one tail tile.
FP8_HD int64_t pair_units(int64_t c, int64_t np, int64_t num_tiles, int64_t split, int64_t tail0) {
    const int64_t whole_end = split > 0 ? tail0 : num_tiles;
    const int64_t n_whole = whole_end > c ? (whole_end - c + np - 1) / np : 0;
    return n_whole + ((split > 0 && c < (num_tiles - tail0) * split) ? 1 : 0);
}

FP8_HD WorkUnit pair_unit(int64_t i, int64_t c, int64_t np, int64_t num_tiles, int64_t nkb, int64_t split,
                          int64_t tail0) {
    const int64_t whole_end = split > 0 ? tail0 : num_tiles;
    const int64_t n_whole = whole_end > c ? (whole_end - c + np - 1) / np : 0;
    if (i < n_whole) return WorkUnit{c + i * np, 0, nkb, -1};
    const int64_t j = c / split, s = c % split;
    return WorkUnit{tail0 + j, s * nkb / split, (s + 1) * nkb / split, c};
}

}  // namespace fp8bs
