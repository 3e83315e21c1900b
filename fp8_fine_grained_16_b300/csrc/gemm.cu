// gemm.cu -- block-scaled FP8 GEMMs on tcgen05 (dense and MoE grouped).
//
// What is computed (pages 2 and 3: partial sums are accumulated by the tensor
// cores over a K interval, then copied out, multiplied by the scaling
// factors and added into FP32; page 4: the interval is 128 elements):
//
//   D[m][n] = sum_kb  sA[kb][m] * sB(n, kb) * P_kb[m][n],
//   P_kb    = A[:, 128kb : 128kb+128] * B[:, 128kb : 128kb+128]^T   (E4M3 MMA)
//
// The pages' Hopper scheme overlaps promotion with WGMMA by ping-ponging two
// warpgroups.  Here the overlap comes from tensor memory instead.  One CTA
// per SM computes 128 x 256 output tiles:
//
//   warp 0        TMA producer.  Per K block one pipeline stage receives the
//                 A tile (128 x 128 B), the B tile (256 x 128 B), both with
//                 the 128-byte swizzle, and the scales the promotion needs:
//                 sA of the tile's 128 rows and sB of its columns.
//   warp 1        allocates TMEM and issues, per K block, four tcgen05.mma
//                 (K = 32 each) into one of two TMEM accumulators (256 fp32
//                 columns each), then commits to the stage's "empty" barrier
//                 and the accumulator's "full" barrier.
//   warps 2, 3    idle (they only give their registers to the promotion warps)
//   warps 4..11   promotion: two warpgroups, one per 128-column half.  Thread
//                 (warp w, lane l) owns tile row 32*(w%4)+l (TMEM lanes are
//                 tied to w%4).  Per K block it reads P_kb from TMEM in two
//                 64-column batches, frees the accumulator (one arrive per
//                 warp) as soon as the second batch is in registers, and adds
//                 P_kb * sA*sB into 128 fp32 registers with packed two-lane
//                 FMAs.  Meanwhile the MMA warp already fills the other
//                 accumulator with P_{kb+1}.  A stage is refilled only after
//                 the MMAs and all eight promotion warps are done with it.
//
// An mbarrier probe costs a couple of hundred cycles on this part even when
// the phase has completed, so each role tests the two barriers it needs per
// K block in one combined probe.
//
// The kernel is persistent: one CTA per SM walks a static list of output
// tiles; stage and accumulator indices run on across tile boundaries, so the
// epilogue of one tile overlaps the first MMAs of the next.
//
// Every pipeline wait is bounded (2 s).  A wait that expires records
// FP8_ERR_TIMEOUT in the device status word, raises a CTA-wide abort flag,
// and lets the CTA drain its copies in flight, release its tensor memory and
// exit.
#include <cudaTypedefs.h>

#include "common.cuh"

namespace fp8bs {

__device__ int g_gemm_status;

FP8_DEV void record_status(int code) { atomicCAS(&g_gemm_status, 0, code); }

constexpr int BM = 128;                 // tile rows (one tcgen05 M=128 MMA)
constexpr int BK = 128;                 // K block = promotion interval = scale block
constexpr int kThreads = 384;           // 12 warps = 3 warpgroups
constexpr int kPromoThreads = 256;      // warps 4..11
constexpr int kPromoWarps = kPromoThreads / 32;
// Register split: the block launches with 168 registers per thread (384 x 168
// = 64512); warpgroup 0 (TMA, MMA, idle) gives back down to 40 and the two
// promotion warpgroups grow to 232: 128*40 + 256*232 = 64512.
constexpr int kTmemCols = 512;
constexpr int kMaxExperts = 1024;
// Scales travel in the pipeline stage through rank-1 TMA maps.  A tensor
// copy starts on a 16-byte boundary of global memory, so the sA box
// (kSaBox floats) starts at the tile's first row rounded down to a multiple
// of 4 elements and the promotion indexes past that offset; each box lands
// on a 128-byte boundary of shared memory.
constexpr int kSaBox = BM + 4;                   // 132 floats = 528 bytes
constexpr int kSaRegion = 640;                   // bytes reserved for it in a stage
constexpr int kSbBox0 = 4;                       // BMODE 0: 16-byte box around one block scale
constexpr int kSbHalf0 = 32;                     // BMODE 0: floats between the two halves' boxes (128 bytes)
static_assert(kSaRegion % 128 == 0 && kSaRegion >= kSaBox * 4 && (kSbHalf0 * 4) % 128 == 0, "TMA box alignment");

template <int BN, int STAGES, int BMODE, bool GROUPED>
struct Layout {
    static constexpr int kABytes = BM * BK;
    static constexpr int kBBytes = BN * BK;
    static constexpr int kSaOff = kABytes + kBBytes;                        // in a stage
    static constexpr int kSbOff = kSaOff + kSaRegion;
    static constexpr int kSbRegion = BMODE == 1 ? BN * 4 : 2 * kSbHalf0 * 4;
    static constexpr int kStageBytes = (kSbOff + kSbRegion + 1023) & ~1023;
    static constexpr uint32_t kTxBytes = kABytes + kBBytes + kSaBox * 4 + (BMODE == 1 ? BN * 4 : 2 * kSbBox0 * 4);
    static constexpr int kStagesBytes = STAGES * kStageBytes;
    static constexpr int kBarOff = kStagesBytes;  // full[S], empty[S], tfull[2], tempty[2], done
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;       // tmem base, abort flag
    static constexpr int kGrpOff = (kMiscOff + 16 + 15) & ~15;    // grouped: off[E+1], tile prefix[E+1]
    static constexpr int kGrpBytes = GROUPED ? 2 * (kMaxExperts + 1) * 4 : 0;
    static constexpr int kBytes = kGrpOff + kGrpBytes;
    static constexpr int kDynSmem = kBytes + 1024;                // slack for 1024-byte alignment
    static_assert(kABytes % 1024 == 0 && kStageBytes % 1024 == 0, "operand tiles start on 1024-byte boundaries");
    static_assert(kSaOff % 128 == 0 && kSbOff % 128 == 0, "scale boxes start on 128-byte boundaries");
};

struct GemmArgs {
    const float* sa;
    const float* sb;
    void* d;
    const int32_t* off;      // grouped only
    int64_t M;               // dense: rows of A / D; grouped: total_rows
    int64_t N;
    int64_t K;
    int E;                   // grouped only
};

struct Tile {
    int64_t row0;            // first row of the tile (global row index)
    int64_t row_end;         // rows >= row_end are not stored
    int32_t n0;              // column tile index from a schedule; first column after tile_at
    int32_t e;               // expert (grouped)
};

// ---------------------------------------------------------------- schedules
// Dense: tile w -> m-tile w % num_m, n-tile w / num_m.  Consecutive tiles run
// on neighbouring SMs at the same time and share their B panel in L2.
struct DenseSched {
    int64_t num_m, num_n, M;
    FP8_DEV int64_t count() const { return num_m * num_n; }
    FP8_DEV Tile get(int64_t w) const {
        Tile t;
        const int64_t mt = w % num_m, nt = w / num_m;
        t.row0 = mt * BM;
        t.row_end = M;
        t.n0 = int32_t(nt);   // column tile index; the kernel scales it by BN
        t.e = 0;
        return t;
    }
};

// Grouped: expert e has mt_e = ceil(rows_e / 128) row tiles; the work list
// holds, for each expert in order, its num_n column tiles x mt_e row tiles
// with the row tile innermost, so that the row tiles of one (expert, column
// tile) run side by side and read the weight tile from HBM once.
struct GroupedSched {
    const int32_t* off_s;    // smem, offsets [E+1]
    const int32_t* pre_s;    // smem, prefix of row-tile counts [E+1]
    int E;
    int64_t num_n;
    FP8_DEV int64_t count() const { return int64_t(pre_s[E]) * num_n; }
    FP8_DEV Tile get(int64_t w) const {
        int lo = 0, hi = E;                 // find e: pre[e]*num_n <= w < pre[e+1]*num_n
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (int64_t(pre_s[mid]) * num_n <= w) lo = mid; else hi = mid;
        }
        const int e = lo;
        const int64_t mt = pre_s[e + 1] - pre_s[e];
        const int64_t local = w - int64_t(pre_s[e]) * num_n;
        Tile t;
        t.e = e;
        t.n0 = int32_t(local / mt);        // column tile index; the kernel scales it by BN
        t.row0 = int64_t(off_s[e]) + (local % mt) * BM;
        t.row_end = off_s[e + 1];
        return t;
    }
};

// ---------------------------------------------------------------- kernel
template <int BN, int STAGES, int BMODE, bool OUT_F32, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_blockscaled_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                            const GemmArgs args) {
    using L = Layout<BN, STAGES, BMODE, GROUPED>;
    static_assert(2 * BN <= kTmemCols, "two accumulators must fit in TMEM");
    static_assert(BN == 256, "one promotion half = 128 columns = one scale block and one column per warpgroup thread");
    constexpr int kHalf = BN / 2;          // columns per promotion warpgroup
    constexpr uint32_t kIdesc = idesc_e4m3_f32(BM, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = bars + 2 * STAGES + 2;
    uint64_t* done = bars + 2 * STAGES + 4;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_s = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t nkb = args.K / BK;

    // ---------------- set-up
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1 + kPromoWarps);          // MMA commit + every promotion warp
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kPromoWarps);             // one arrive per promotion warp
        }
        mbar_init(done, 1);
        *abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSA);
        tma_prefetch_desc(&tmSB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_base_s, kTmemCols);
        tmem_relinquish();
    }

    GroupedSched gs{};
    DenseSched ds{};
    if constexpr (GROUPED) {
        int32_t* off_s = reinterpret_cast<int32_t*>(smem + L::kGrpOff);
        int32_t* pre_s = off_s + (kMaxExperts + 1);
        const int E = args.E;
        bool bad = false;
        for (int i = threadIdx.x; i <= E; i += kThreads) off_s[i] = __ldg(args.off + i);
        __syncthreads();
        if (warp == 0) {
            // validate and build the prefix of row-tile counts, 32 experts per step
            int carry = 0;
            if (lane == 0) pre_s[0] = 0;
            for (int base = 0; base < E; base += 32) {
                const int e = base + lane;
                int cnt = 0;
                if (e < E) {
                    const int64_t lo = off_s[e], hi = off_s[e + 1];
                    const bool ok = lo >= 0 && lo <= hi && hi <= args.M;
                    bad |= !ok;
                    cnt = ok ? int((hi - lo + BM - 1) / BM) : 0;
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
            bad |= (lane == 0) && (off_s[0] != 0 || int64_t(off_s[E]) != args.M);
            if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && blockIdx.x == 0) record_status(FP8_ERR_OFFSETS);
        }
        gs = GroupedSched{off_s, pre_s, E, (args.N + BN - 1) / BN};
    } else {
        ds = DenseSched{(args.M + BM - 1) / BM, (args.N + BN - 1) / BN, args.M};
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_base_s;

    // Both schedules return the column-tile index in n0; scale it to a column.
    auto tile_at = [&](int64_t w) -> Tile {
        Tile t;
        if constexpr (GROUPED) t = gs.get(w); else t = ds.get(w);
        t.n0 *= BN;
        return t;
    };
    int64_t num_tiles;
    if constexpr (GROUPED) num_tiles = gs.count(); else num_tiles = ds.count();
    // BMODE 0: index in sb of K block 0 of the 128x128 block scales of column
    // half h of tile t (a half past N reads an in-bounds scale, never stored)
    auto sb_row = [&](const Tile& t, int h) -> int64_t {
        const int64_t c0 = int64_t(t.n0) + h * kHalf;
        return (int64_t(t.e) * (args.N / 128) + (c0 < args.N ? c0 : args.N - 1) / 128) * nkb;
    };

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 40;");
        if (warp == 0) {
            // ================= TMA producer
            if (lane == 0) {
                uint32_t it = 0;
                bool ok = true;
                for (int64_t w = blockIdx.x; ok && w < num_tiles; w += gridDim.x) {
                    const Tile t = tile_at(w);
                    int64_t sbr[2] = {0, 0};
                    if constexpr (BMODE == 0) {
                        sbr[0] = sb_row(t, 0);
                        sbr[1] = sb_row(t, 1);
                    }
                    for (int64_t kb = 0; kb < nkb; ++kb) {
                        const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
                        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_s)) {
                            ok = false;
                            break;
                        }
                        uint8_t* st = smem + stage * L::kStageBytes;
                        mbar_arrive_expect_tx(&full[stage], L::kTxBytes);
                        tma_load_2d(st, &tmA, &full[stage], int32_t(kb * BK), int32_t(t.row0));
                        if constexpr (GROUPED)
                            tma_load_3d(st + L::kABytes, &tmB, &full[stage], int32_t(kb * BK), t.n0, t.e);
                        else
                            tma_load_2d(st + L::kABytes, &tmB, &full[stage], int32_t(kb * BK), t.n0);
                        tma_load_1d(st + L::kSaOff, &tmSA, &full[stage], int32_t((kb * args.M + t.row0) & ~int64_t(3)));
                        if constexpr (BMODE == 0) {
                            tma_load_1d(st + L::kSbOff, &tmSB, &full[stage], int32_t((sbr[0] + kb) & ~int64_t(3)));
                            tma_load_1d(st + L::kSbOff + kSbHalf0 * 4, &tmSB, &full[stage],
                                        int32_t((sbr[1] + kb) & ~int64_t(3)));
                        } else {
                            tma_load_1d(st + L::kSbOff, &tmSB, &full[stage], int32_t(kb * args.N + t.n0));
                        }
                        ++it;
                    }
                }
                if (!ok) record_status(FP8_ERR_TIMEOUT);
                // Let every copy this thread issued land before the CTA can exit.
                // Only this thread arrives on full[], so the latest phase of each
                // stage is the one of its last issued load.
                int zero = 0;
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait_bounded(&full[j % STAGES], (j / STAGES) & 1u, reinterpret_cast<volatile int*>(&zero));
            }
            __syncwarp();
        } else if (warp == 1) {
            // ================= MMA issuer
            if (lane == 0) {
                uint32_t it = 0, g = 0;
                bool ok = true;
                for (int64_t w = blockIdx.x; ok && w < num_tiles; w += gridDim.x) {
                    for (int64_t kb = 0; kb < nkb; ++kb) {
                        const uint32_t buf = g & 1u, tphase = (g >> 1) & 1u;
                        const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
                        // the stage is usually loaded long before the accumulator frees up
                        if (!mbar_test_wait2(&full[stage], phase, &tempty[buf], tphase ^ 1u)) {
                            if (!mbar_wait_bounded(&full[stage], phase, abort_s)) { ok = false; break; }
                            if (!mbar_wait_bounded(&tempty[buf], tphase ^ 1u, abort_s)) { ok = false; break; }
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + stage * L::kStageBytes);
                        const uint32_t b_addr = a_addr + L::kABytes;
                        const uint64_t adesc = sw128_kmajor_desc(a_addr);
                        const uint64_t bdesc = sw128_kmajor_desc(b_addr);
                        const uint32_t d_tmem = tmem_base + buf * BN;
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k)      // K = 32 bytes per MMA: +2 in the >>4 address field
                            umma_e4m3(d_tmem, adesc + 2 * k, bdesc + 2 * k, kIdesc, k > 0 ? 1u : 0u);
                        umma_commit(&empty[stage]);
                        umma_commit(&tfull[buf]);
                        ++it;
                        ++g;
                    }
                }
                if (!ok) record_status(FP8_ERR_TIMEOUT);
                // all MMAs issued by this thread are complete once `done` flips
                umma_commit(done);
                int zero = 0;
                mbar_wait_bounded(done, 0, reinterpret_cast<volatile int*>(&zero));
            }
            __syncwarp();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
        // ================= promotion warpgroups
        const int wq = warp & 3;                       // TMEM lane quarter of this warp
        const int half = (warp - 4) >> 2;              // 0: columns [0, BN/2), 1: [BN/2, BN)
        const int r = wq * 32 + lane;                  // tile row
        const uint32_t t_lane = uint32_t(wq * 32) << 16;

        uint32_t g = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; ok && w < num_tiles; w += gridDim.x) {
            const Tile t = tile_at(w);
            const int64_t m = t.row0 + r;
            const int64_t ncol0 = int64_t(t.n0) + half * kHalf;   // first column of this thread's half
            // N % 128 == 0, so a half tile (128 columns) is either entirely
            // inside [0, N) or entirely past it (last tile of an N that is an
            // odd multiple of 128).
            const bool cols_ok = ncol0 < args.N;
            const int64_t sbr = BMODE == 0 ? sb_row(t, half) : 0;

            float2 acc[kHalf / 2];
#pragma unroll
            for (int i = 0; i < kHalf / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);

            for (int64_t kb = 0; kb < nkb; ++kb) {
                const uint32_t stage = g % STAGES, phase = (g / STAGES) & 1u;
                const uint32_t buf = g & 1u, tphase = (g >> 1) & 1u;
                // Lane 0 waits for this K block's stage (its scales) and
                // accumulator; __syncwarp passes the acquire on to the other
                // lanes, and the warp leaves the loop as a whole if a wait
                // gave up (the tcgen05 loads below are warp-collective).
                bool got = true;
                if (lane == 0 && !mbar_test_wait2(&full[stage], phase, &tfull[buf], tphase))
                    got = mbar_wait_bounded(&full[stage], phase, abort_s) &&
                          mbar_wait_bounded(&tfull[buf], tphase, abort_s);
                got = __shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) != 0;
                __syncwarp();
                if (!got) { ok = false; break; }
                tc_fence_after();

                const uint8_t* st = smem + stage * L::kStageBytes;
                // the sA box starts at (kb*M + row0) rounded down to 4 elements
                const float sa_cur = reinterpret_cast<const float*>(st + L::kSaOff)[int((kb * args.M + t.row0) & 3) + r];
                const float2 sa2 = make_float2(sa_cur, sa_cur);
                float2 sc2 = sa2;
                const float* sbk = reinterpret_cast<const float*>(st + L::kSbOff) + half * kHalf;   // BMODE 1
                if constexpr (BMODE == 0) {
                    const float sbv =
                        reinterpret_cast<const float*>(st + L::kSbOff)[half * kSbHalf0 + int((sbr + kb) & 3)];
                    const float sc = __fmul_rn(sa_cur, sbv);
                    sc2 = make_float2(sc, sc);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[stage]);      // this warp is done with the stage
                }

                auto scale_chunk = [&](int c, const uint32_t (&v)[32]) {
                    if constexpr (BMODE == 0) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            acc[c * 16 + i] = __ffma2_rn(
                                make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), sc2,
                                acc[c * 16 + i]);
                    } else {
                        const float4* sbv = reinterpret_cast<const float4*>(sbk + c * 32);
#pragma unroll
                        for (int i4 = 0; i4 < 8; ++i4) {
                            const float4 b4 = sbv[i4];
                            const float2 p0 = __fmul2_rn(
                                make_float2(__uint_as_float(v[4 * i4]), __uint_as_float(v[4 * i4 + 1])),
                                make_float2(b4.x, b4.y));
                            const float2 p1 = __fmul2_rn(
                                make_float2(__uint_as_float(v[4 * i4 + 2]), __uint_as_float(v[4 * i4 + 3])),
                                make_float2(b4.z, b4.w));
                            acc[c * 16 + 2 * i4] = __ffma2_rn(p0, sa2, acc[c * 16 + 2 * i4]);
                            acc[c * 16 + 2 * i4 + 1] = __ffma2_rn(p1, sa2, acc[c * 16 + 2 * i4 + 1]);
                        }
                    }
                };

                const uint32_t tcol = tmem_base + t_lane + buf * BN + half * kHalf;
                uint32_t va[32], vb[32];
                // columns [0, 64) of this half
                tmem_ld_32x32b_x32(tcol, va);
                tmem_ld_32x32b_x32(tcol + 32, vb);
                tmem_wait_ld_regs(va);
                regs_fence(vb);
                scale_chunk(0, va);
                scale_chunk(1, vb);
                // columns [64, 128); once they are in registers the accumulator
                // is free for the MMAs two K blocks ahead
                tmem_ld_32x32b_x32(tcol + 64, va);
                tmem_ld_32x32b_x32(tcol + 96, vb);
                tmem_wait_ld_regs(va);
                regs_fence(vb);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[buf]);
                scale_chunk(2, va);
                scale_chunk(3, vb);
                if constexpr (BMODE == 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[stage]);      // column scales no longer read
                }
                ++g;
            }
            if (!ok) break;

            // ---- epilogue: this thread's row, BN/2 consecutive columns
            if (cols_ok && m < t.row_end && m < args.M) {
                if constexpr (OUT_F32) {
                    float* dst = reinterpret_cast<float*>(args.d) + m * args.N + ncol0;
#pragma unroll
                    for (int i = 0; i < kHalf / 2; i += 2)
                        *reinterpret_cast<float4*>(dst + 2 * i) =
                            make_float4(acc[i].x, acc[i].y, acc[i + 1].x, acc[i + 1].y);
                } else {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(args.d) + m * args.N + ncol0;
#pragma unroll
                    for (int i = 0; i < kHalf / 2; i += 4) {
                        const uint4 o = make_uint4(cvt_bf16x2(acc[i].x, acc[i].y), cvt_bf16x2(acc[i + 1].x, acc[i + 1].y),
                                                   cvt_bf16x2(acc[i + 2].x, acc[i + 2].y),
                                                   cvt_bf16x2(acc[i + 3].x, acc[i + 3].y));
                        *reinterpret_cast<uint4*>(dst + 2 * i) = o;
                    }
                }
            }
        }
        if (!ok) record_status(FP8_ERR_TIMEOUT);
    }

    // ---------------- tear-down
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// K-major E4M3 operand [rows][K] (rank 2), or a stack [batch][rows][K]
// (rank 3, even when batch == 1), box = 128 (K) x box_rows (x 1), 128-byte
// swizzle, zero fill out of bounds.
static bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows,
                             int64_t batch, bool stacked) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cuuint64_t(K), cuuint64_t(rows), cuuint64_t(batch)};
    cuuint64_t strides[2] = {cuuint64_t(K), cuuint64_t(K) * cuuint64_t(rows)};
    cuuint32_t box[3] = {128u, cuuint32_t(box_rows), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    const cuuint32_t rank = stacked ? 3u : 2u;
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Rank-1 fp32 view of a scale tensor of n elements, box of `box` floats, no
// swizzle, zero fill past the end.
static bool make_scale_map(CUtensorMap* map, const float* base, int64_t n, int box) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[1] = {cuuint64_t(n)};
    cuuint64_t strides[1] = {0};
    cuuint32_t boxd[1] = {cuuint32_t(box)};
    cuuint32_t estr[1] = {1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1u, const_cast<float*>(base), dims, strides, boxd, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static int device_sms() {
    int dev = 0, n = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess || major != 10) return -1;
    return n;
}

template <int BN, int STAGES, int BMODE, bool OUT_F32, bool GROUPED>
static int launch(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msa, const CUtensorMap& msb,
                  const GemmArgs& args, int grid, cudaStream_t stream) {
    using L = Layout<BN, STAGES, BMODE, GROUPED>;
    auto kern = gemm_blockscaled_kernel<BN, STAGES, BMODE, OUT_F32, GROUPED>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynSmem) != cudaSuccess)
            return FP8_ERR_CUDA;
        attr_set = true;
    }
    kern<<<grid, kThreads, L::kDynSmem, stream>>>(ma, mb, msa, msb, args);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

constexpr int kBN = 256;
constexpr int kStages = 4;

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// will ever arrive on, gives up after timeout_ns and records FP8_ERR_TIMEOUT,
// exactly as a stalled GEMM pipeline stage would.
__global__ void wait_timeout_selftest_kernel(uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
        if (!mbar_wait_bounded(&bar, 0, &abort_flag, timeout_ns)) record_status(FP8_ERR_TIMEOUT);
    }
}

}  // namespace fp8bs

using namespace fp8bs;

extern "C" int fp8_gemm_blockscaled(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                                    int b_scale_mode, void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                                    fp8_stream_t stream) {
    if (!a || !sa || !b || !sb || !d || M <= 0 || N <= 0 || K <= 0) return FP8_ERR_ARG;
    if ((b_scale_mode != FP8_BSCALE_BLOCK128 && b_scale_mode != FP8_BSCALE_ROW) ||
        (d_dtype != FP8_OUT_BF16 && d_dtype != FP8_OUT_F32))
        return FP8_ERR_ARG;
    if (K % 128 || N % 128) return FP8_ERR_SHAPE;
    if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1) return FP8_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || !aligned16(sa) || !aligned16(sb)) return FP8_ERR_ALIGN;
    if (M * (K / 128) >= (int64_t(1) << 31) || (b_scale_mode == FP8_BSCALE_ROW && N * (K / 128) >= (int64_t(1) << 31)))
        return FP8_ERR_SHAPE;
    const int sms = device_sms();
    if (sms <= 0) return FP8_ERR_DEVICE;
    CUtensorMap ma, mb, msa, msb;
    const int64_t nsb = b_scale_mode == FP8_BSCALE_ROW ? N * (K / 128) : (N / 128) * (K / 128);
    if (!make_operand_map(&ma, a, M, K, BM, 1, false) || !make_operand_map(&mb, b, N, K, kBN, 1, false) ||
        !make_scale_map(&msa, sa, M * (K / 128), kSaBox) ||
        !make_scale_map(&msb, sb, nsb, b_scale_mode == FP8_BSCALE_ROW ? kBN : kSbBox0))
        return FP8_ERR_CUDA;
    GemmArgs args{sa, sb, d, nullptr, M, N, K, 0};
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + kBN - 1) / kBN);
    const int grid = int(tiles < sms ? tiles : sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (b_scale_mode == FP8_BSCALE_BLOCK128) {
        if (d_dtype == FP8_OUT_BF16) return launch<kBN, kStages, 0, false, false>(ma, mb, msa, msb, args, grid, s);
        return launch<kBN, kStages, 0, true, false>(ma, mb, msa, msb, args, grid, s);
    }
    if (d_dtype == FP8_OUT_BF16) return launch<kBN, kStages, 1, false, false>(ma, mb, msa, msb, args, grid, s);
    return launch<kBN, kStages, 1, true, false>(ma, mb, msa, msb, args, grid, s);
}

extern "C" int fp8_grouped_gemm_blockscaled(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                                            const int32_t* expert_offsets, int E, int64_t total_rows, int64_t N,
                                            int64_t K, uint16_t* d, fp8_stream_t stream) {
    if (!b || !sb || !expert_offsets || E <= 0 || E > kMaxExperts || total_rows < 0 || N <= 0 || K <= 0)
        return FP8_ERR_ARG;
    if (K % 128 || N % 128) return FP8_ERR_SHAPE;
    if (total_rows > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1)
        return FP8_ERR_SHAPE;
    if (total_rows == 0) return FP8_OK;
    if (!a || !sa || !d) return FP8_ERR_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || !aligned16(sa) || !aligned16(sb) ||
        (reinterpret_cast<uintptr_t>(expert_offsets) & 3u))
        return FP8_ERR_ALIGN;
    if (total_rows * (K / 128) >= (int64_t(1) << 31) || int64_t(E) * (N / 128) * (K / 128) >= (int64_t(1) << 31))
        return FP8_ERR_SHAPE;
    const int sms = device_sms();
    if (sms <= 0) return FP8_ERR_DEVICE;
    CUtensorMap ma, mb, msa, msb;
    if (!make_operand_map(&ma, a, total_rows, K, BM, 1, false) || !make_operand_map(&mb, b, N, K, kBN, E, true) ||
        !make_scale_map(&msa, sa, total_rows * (K / 128), kSaBox) ||
        !make_scale_map(&msb, sb, int64_t(E) * (N / 128) * (K / 128), kSbBox0))
        return FP8_ERR_CUDA;
    GemmArgs args{sa, sb, d, expert_offsets, total_rows, N, K, E};
    return launch<kBN, kStages, 0, false, true>(ma, mb, msa, msb, args, sms, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fp8_selftest_wait_timeout(uint64_t timeout_ns, fp8_stream_t stream) {
    if (timeout_ns == 0 || timeout_ns > kWaitTimeoutNs) return FP8_ERR_ARG;
    wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(timeout_ns);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// Status word of this translation unit: read and clear (synchronising).
extern "C" int fp8bs_gemm_take_status(cudaStream_t stream) {
    int v = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP8_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof v) != cudaSuccess) return FP8_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof zero) != cudaSuccess) return FP8_ERR_CUDA;
    return v;
}
