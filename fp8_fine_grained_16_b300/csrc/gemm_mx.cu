// gemm_mx.cu -- block-scaled FP8 GEMM with the scales applied by the tensor
// core, for power-of-two scales.
//
// The gnrental.net page notes that the fine-grained tiles match the idea of
// microscaling formats, which Blackwell tensor cores support; tmdrlife.com page
//  asks for tensor cores that take the scaling factors
// themselves, and fixes some activation scales to integral powers of two.
// With power-of-two scales (the quantisers' FP8_SCALE_POW2 mode) every scale
// s = 2^e is exactly a UE8M0 scale factor, so the block-scaled tcgen05 MMA
// (kind::mxf8f6f4, one scale per 32 K elements per row of A and of B) computes
//
//   D[m][n] = sum_kb sum_{k in kb} (sA[kb][m] qA[m][k]) (sB(n,kb) qB[n][k])
//
// with the 1x128 tile scale repeated in the four K = 32 MMAs of its K block
// and a 128x128 block scale repeated for every row n of the block.  The
// products 2^e * code are exact; the fp32 sum runs in tensor memory over the
// whole K, so no CUDA-core promotion is needed.  The result equals the
// block-promoted sum of the other GEMM up to fp32 rounding order.
//
// A cluster of two CTAs computes 256 x 224 output tiles with
// tcgen05.mma.cta_group::2 (M = 256): each CTA holds 128 rows of A and 112
// rows of B in shared memory.  224 columns leave room in the 512 TMEM columns
// for two accumulators (columns 0 and 256) and two 16-column scale slots
// (224..255); N = 7168 is 32 tiles of 224.  A scale slot serves four
// consecutive K blocks: byte b of each 32-bit word holds the scale of K
// block 4g + b, and the MMAs of that K block select byte b through the scale
// fields of the instruction descriptor.  Roles per CTA:
//
//   warp 0        TMA producer: A and the B half (128-byte swizzle) into a
//                 STAGES-deep ring.
//   warp 1        allocates TMEM; in the leader CTA, issues per K block four
//                 MMAs (K = 32) and commits them to both CTAs' barriers.
//   warps 2..5    scale warps (TMEM lane quarter = warp % 4): read the fp32
//                 scales of four K blocks from global memory, turn them into
//                 UE8M0 bytes and store them into a scale slot with
//                 tcgen05.st, one group ahead of the MMA.  A scale that is
//                 not a positive normal power of two records FP8_ERR_SCALE.
//   warps 6..9    epilogue (lane quarter = warp % 4): once per tile, read
//                 the accumulator, convert, store, free the accumulator.
//
// Barriers (S = STAGES; g = K-block counter / 4):
//   full[s]   leader: producer + both CTAs' operand bytes
//   empty[s]  each:   MMA commit (stage s may be reloaded)
//   sff[g%2]  leader: the 8 scale warps of the pair (group g is in TMEM)
//   sfe[g%2]  each:   MMA commit after the last K block of group g
//   accf[b]   each:   MMA commit after a tile's last K block
//   acce[b]   leader: the 8 epilogue warps of the pair
// Every wait is bounded (2 s); an expired wait records FP8_ERR_TIMEOUT, raises
// the CTA's abort flag, and the CTA drains and leaves as in the other GEMM.
#include "common.cuh"
#include "expert_sched.cuh"
#include "tensor_map.cuh"

namespace fp8bs {

__device__ int g_mx_status;

FP8_DEV void mx_record(int code) { atomicCAS(&g_mx_status, 0, code); }

namespace mx {

constexpr int BM = 128;                 // rows of A per CTA (M = 256 per pair)
constexpr int BN = 224;                 // columns per pair tile
constexpr int BK = 128;                 // K block = scale block
constexpr int kThreads = 320;           // 10 warps
constexpr int kTmemCols = 512;
constexpr int kAccStride = 256;         // accumulator b at TMEM column 256 * b
constexpr int kGroup = 4;               // K blocks per scale slot (one byte each)
constexpr int kSlotCols = 16;           // A scales at +0 .. +3, B scales at +8 .. +8 + BN/32
constexpr int kBCols = BN / 32;         // 7 B-scale columns
static_assert(BN + 2 * kSlotCols <= kAccStride && 8 + kBCols <= kSlotCols, "TMEM plan");
static_assert(BN % 32 == 0 && BN % 16 == 0 && BN <= 256, "MMA N");

// TMEM column of scale slot j (j = 0, 1), in the gap after accumulator 0.
FP8_DEV uint32_t slot_col(uint32_t j) { return BN + kSlotCols * j; }

struct Args {
    const float* sa;
    const float* sb;
    void* d;
    int64_t M, N, K;         // grouped: M = total rows of all experts
    const int32_t* off;      // grouped only: expert offsets [E+1]
    int E;                   // grouped only
};

template <bool PAIR, int STAGES, bool GROUPED>
struct Layout {
    static constexpr int kABytes = BM * BK;                     // 16 KB
    static constexpr int kBBytes = (PAIR ? BN / 2 : BN) * BK;   // 14 KB of a pair's B tile, 28 KB alone
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kPairTxBytes = (PAIR ? 2 : 1) * (kABytes + kBBytes);
    static constexpr int kXchgOff = STAGES * kStageBytes;       // packed B scale words, 2 x 8 x 32
    static constexpr int kBarOff = kXchgOff + 2 * 8 * 32 * 4;
    static constexpr int kNumBars = 2 * STAGES + 2 + 2 + 2 + 2 + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kGrpOff = kMiscOff + 16;                // grouped: offsets and row-pair prefix
    static constexpr int kGrpBytes = GROUPED ? 2 * (kMaxExperts + 1) * 4 : 0;
    static constexpr int kBytes = kGrpOff + kGrpBytes;
    static constexpr int kDynSmem = kBytes + 1024;
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "operand tiles on 1024-byte boundaries");
    static_assert(kDynSmem <= 232448, "shared memory per CTA");
};

template <bool PAIR, int STAGES, int BMODE, bool OUT_F32, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mx_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const Args args) {
    using L = Layout<PAIR, STAGES, GROUPED>;
    constexpr int kCtas = PAIR ? 2 : 1;
    constexpr int kTileRows = kCtas * BM;
    constexpr uint32_t kIdesc = idesc_mx_e4m3(kTileRows, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* sff = bars + 2 * STAGES;
    uint64_t* sfe = sff + 2;
    uint64_t* accf = sfe + 2;
    uint64_t* acce = accf + 2;
    uint64_t* done = acce + 2;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_s = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int64_t nkb = args.K / BK;
    const int64_t num_m2 = (args.M + kTileRows - 1) / kTileRows;
    const int64_t num_n = (args.N + BN - 1) / BN;
    // a "cluster" is the pair, or the CTA itself
    const int64_t cluster = PAIR ? blockIdx.x >> 1 : blockIdx.x, nclusters = PAIR ? gridDim.x >> 1 : gridDim.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&sff[j], 4 * kCtas);
            mbar_init(&sfe[j], 1);
            mbar_init(&accf[j], 1);
            mbar_init(&acce[j], 4 * kCtas);
        }
        mbar_init(done, 1);
        *abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(tmem_base_s, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_base_s, kTmemCols);
            tmem_relinquish();
        }
    }
    // Launched as a programmatic dependent launch, the kernel may have started
    // while the one before it on the stream is still running: everything
    // above touches only this CTA's own shared memory, TMEM and the kernel
    // parameters; from here on it reads and writes global memory.
    pdl_wait();

    // grouped: the per-expert tile list (offsets and row-pair prefix in shared memory)
    int32_t* off_s = reinterpret_cast<int32_t*>(smem + L::kGrpOff);
    int32_t* pre_s = off_s + (kMaxExperts + 1);
    int64_t num_tiles = num_m2 * num_n;
    if constexpr (GROUPED) {
        if (expert_tile_prefix(args.off, args.E, args.M, off_s, pre_s, kTileRows) && threadIdx.x == 0 && blockIdx.x == 0)
            mx_record(FP8_ERR_OFFSETS);
        num_tiles = int64_t(pre_s[args.E]) * num_n;
    }
    tc_fence_before();
    if constexpr (PAIR) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_base_s;

    // Tile w.  Dense: row pair w % num_m2, column tile w / num_m2.  Grouped:
    // the expert list.  row0 is this CTA's first row; rows >= row_end are
    // computed but not stored.
    struct TileAt {
        int64_t row0, row_end, n0;
        int e;
    };
    auto tile_at = [&](int64_t w) {
        TileAt t;
        if constexpr (GROUPED) {
            const ExpertTile x = expert_tile(off_s, pre_s, args.E, num_n, w, kTileRows);
            t.row0 = x.row0 + int64_t(rank) * BM;
            t.row_end = x.row_end;
            t.n0 = x.col_tile * BN;
            t.e = x.e;
        } else {
            t.row0 = (w % num_m2) * kTileRows + int64_t(rank) * BM;
            t.row_end = args.M;
            t.n0 = (w / num_m2) * BN;
            t.e = 0;
        }
        return t;
    };
    // K blocks this cluster walks in all (every tile has nkb)
    const int64_t my_tiles = cluster < num_tiles ? (num_tiles - 1 - cluster) / nclusters + 1 : 0;
    const int64_t my_iters = my_tiles * nkb;

    if (warp == 0) {
        // ================= TMA producer (each CTA)
        if (lane == 0) {
            const uint32_t full0 = PAIR ? mapa_shared(&full[0], 0) : 0u;
            uint32_t it = 0;
            bool ok = true;
            for (int64_t w = cluster; ok && w < num_tiles; w += nclusters) {
                const TileAt t = tile_at(w);
                for (int64_t kb = 0; kb < nkb; ++kb) {
                    const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_s)) { ok = false; break; }
                    uint8_t* st = smem + stage * L::kStageBytes;
                    const uint32_t fbar = full0 + stage * 8;
                    if (leader) mbar_arrive_expect_tx(&full[stage], L::kPairTxBytes);
                    if constexpr (PAIR) {
                        tma_load_2d_pair(st, &tmA, fbar, int32_t(kb * BK), int32_t(t.row0));
                        if constexpr (GROUPED)
                            tma_load_3d_pair(st + L::kABytes, &tmB, fbar, int32_t(kb * BK),
                                             int32_t(t.n0 + rank * (BN / 2)), t.e);
                        else
                            tma_load_2d_pair(st + L::kABytes, &tmB, fbar, int32_t(kb * BK),
                                             int32_t(t.n0 + rank * (BN / 2)));
                    } else {
                        tma_load_2d(st, &tmA, &full[stage], int32_t(kb * BK), int32_t(t.row0));
                        if constexpr (GROUPED)
                            tma_load_3d(st + L::kABytes, &tmB, &full[stage], int32_t(kb * BK), int32_t(t.n0), t.e);
                        else
                            tma_load_2d(st + L::kABytes, &tmB, &full[stage], int32_t(kb * BK), int32_t(t.n0));
                    }
                    ++it;
                }
            }
            if (!ok) mx_record(FP8_ERR_TIMEOUT);
            // the leader's full[] counts both CTAs' bytes: let the last copies land
            if (leader) {
                int zero = 0;
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait_bounded(&full[j % STAGES], (j / STAGES) & 1u, reinterpret_cast<volatile int*>(&zero));
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer (leader only): the whole warp runs the
        // loop in step; lane 0 waits on barriers, one elected lane issues.
        if (leader) {
            uint32_t it = 0, tc = 0;
            bool ok = true;
            bool ready = false;     // barriers of K block `it` already seen complete
            // commit to a barrier of both CTAs of a pair (or of the CTA alone)
            auto commit = [&](uint64_t* bar) {
                if constexpr (PAIR) umma_commit_pair_elect(bar, 0x3); else umma_commit_elect(bar);
            };
            auto wait_all = [&](uint64_t* bar, uint32_t parity) {
                bool got = true;
                if (lane == 0) got = mbar_wait_bounded(bar, parity, abort_s);
                return __shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) != 0;
            };
            for (int64_t w = cluster; ok && w < num_tiles; w += nclusters, ++tc) {
                const uint32_t buf = tc & 1u;
                // the epilogue of tile tc - 2 has read this accumulator
                if (!wait_all(&acce[buf], ((tc >> 1) & 1u) ^ 1u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * kAccStride;
                for (int64_t kb = 0; kb < nkb; ++kb) {
                    const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
                    const uint32_t g = it / kGroup, b = it % kGroup;
                    if (!ready) {
                        // scales of group g are in slot g % 2 (both CTAs)
                        if (b == 0 && !wait_all(&sff[g & 1u], (g >> 1) & 1u)) { ok = false; break; }
                        // operands of both CTAs landed
                        if (!wait_all(&full[stage], phase)) { ok = false; break; }
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * L::kStageBytes);
                    const uint64_t adesc = sw128_kmajor_desc(a_addr);
                    const uint64_t bdesc = sw128_kmajor_desc(a_addr + L::kABytes);
                    const uint32_t sf = tmem_base + slot_col(g & 1u);
                    const uint32_t idesc = kIdesc | (b << 4) | (b << 29);      // scale byte b of A and B
#pragma unroll
                    for (int k = 0; k < BK / 32 - 1; ++k)
                        umma_mx_e4m3_elect<PAIR>(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, sf, sf + 8,
                                                (kb > 0 || k > 0) ? 1u : 0u);
                    // The last MMA goes out together with a probe of the next K
                    // block's barriers: the probe's latency overlaps the issue of
                    // the MMA, which waits for the tensor core to take it.
                    {
                        const uint32_t nit = it + 1, ns = nit % STAGES, np = (nit / STAGES) & 1u;
                        const uint32_t ng = nit / kGroup;
                        ready = umma_mx_e4m3_probe_elect<PAIR>(
                            d_tmem, adesc + 2 * (BK / 32 - 1), bdesc + 2 * (BK / 32 - 1), idesc, sf, sf + 8,
                            smem_u32(&full[ns]), np, nit % kGroup == 0 ? smem_u32(&sff[ng & 1u]) : 0u, (ng >> 1) & 1u);
                        ready = __all_sync(0xFFFFFFFFu, ready);
                    }
                    commit(&empty[stage]);
                    if (b == kGroup - 1) commit(&sfe[g & 1u]);
                    ++it;
                }
                if (!ok) break;
                commit(&accf[buf]);
            }
            if (!ok && lane == 0) mx_record(FP8_ERR_TIMEOUT);
            // commits track the issuing thread's MMAs: the same elected lane
            if constexpr (PAIR) umma_commit_pair_elect(done, 0x1); else umma_commit_elect(done);
            if (lane == 0) {
                int zero = 0;
                mbar_wait_bounded(done, 0, reinterpret_cast<volatile int*>(&zero));
            }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ================= scale warps (each CTA): row r of the CTA's 128 and
        // tile columns 32j + lane, for TMEM lane quarter q.  The fp32 scales of
        // group g + 1 are loaded while group g is converted and stored, so one
        // load latency overlaps a whole group of MMAs.
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t t_lane = uint32_t(32 * q) << 16;
        const uint32_t sff0 = PAIR ? mapa_shared(&sff[0], 0) : 0u;
        const int nblk = int(args.N / 128);
        const uint32_t unkb = uint32_t(nkb);
        // Position of a K block in this cluster's walk, advanced one K block at
        // a time (tile coordinates change once per tile: no per-K-block division).
        struct Pos {
            uint32_t kb, w;
            int64_t m;          // this thread's row
            int32_t n0;         // first column of the tile
            int64_t sb0;        // grouped: the expert's first B-scale row block (e * N/128)
        };
        auto set_tile = [&](Pos& p) {
            const TileAt t = tile_at(p.w);
            p.m = t.row0 + r;
            p.n0 = int32_t(t.n0);
            p.sb0 = int64_t(t.e) * nblk;
        };
        Pos pl{0, uint32_t(cluster), 0, 0, 0};
        set_tile(pl);
        // The four scale warps share the B scales: warp q loads and packs tile
        // column groups j = q and q + 4 (columns 32j + lane) and passes the
        // packed words to the others through shared memory.
        constexpr int kMyB = 2;
        uint32_t* xchg = reinterpret_cast<uint32_t*>(smem + L::kXchgOff);
        // Raw fp32 scales of one group: A of this thread's row, B of its column
        // groups (rows >= M, columns >= N and j >= BN/32 read as 1.0).
        auto load_group = [&](uint32_t it0, uint32_t (&ua)[kGroup], uint32_t (&ub)[kGroup][kMyB]) {
#pragma unroll
            for (int b = 0; b < kGroup; ++b) {
                const bool live = it0 + b < uint32_t(my_iters);
                ua[b] = __float_as_uint(live && pl.m < args.M ? __ldg(args.sa + int64_t(pl.kb) * args.M + pl.m) : 1.0f);
#pragma unroll
                for (int jj = 0; jj < kMyB; ++jj) {
                    const int j = q + 4 * jj;
                    const int n = pl.n0 + 32 * j + lane;
                    float v = 1.0f;
                    if (live && j < kBCols && n < args.N) {
                        if constexpr (BMODE == 0)
                            v = __ldg(args.sb + (pl.sb0 + min(n >> 7, nblk - 1)) * nkb + pl.kb);
                        else v = __ldg(args.sb + int64_t(pl.kb) * args.N + n);
                    }
                    ub[b][jj] = __float_as_uint(v);
                }
                if (live && ++pl.kb == unkb) {
                    pl.kb = 0;
                    pl.w += uint32_t(nclusters);
                    set_tile(pl);
                }
            }
        };
        // UE8M0 bytes of four K blocks in one word (byte b = K block 4g + b).
        // The biased exponent of a positive fp32 is bits 23..30.
        auto pack4 = [](uint32_t u0, uint32_t u1, uint32_t u2, uint32_t u3) {
            return (u0 >> 23) | ((u1 >> 15) & 0xFF00u) | ((u2 >> 7) & 0xFF0000u) | ((u3 << 1) & 0xFF000000u);
        };
        // A scale is a positive normal power of two iff its mantissa is zero and
        // u - 2^23 < 0x7F000000 (excludes zero/subnormal, Inf/NaN and negatives).
        uint32_t chk_max = 0, chk_mant = 0;
        auto check = [&](uint32_t u) {
            chk_max = max(chk_max, u - 0x00800000u);
            chk_mant |= u & 0x007FFFFFu;
        };
        uint32_t na[kGroup], nbv[kGroup][kMyB];
        if (my_iters > 0) load_group(0, na, nbv);
        bool ok = true;
        for (uint32_t it0 = 0; it0 < uint32_t(my_iters); it0 += kGroup) {
            const uint32_t g = it0 / kGroup;
            uint32_t ca[kGroup], cbv[kGroup][kMyB];
#pragma unroll
            for (int b = 0; b < kGroup; ++b) {
                ca[b] = na[b];
#pragma unroll
                for (int jj = 0; jj < kMyB; ++jj) cbv[b][jj] = nbv[b][jj];
            }
            if (it0 + kGroup < uint32_t(my_iters)) load_group(it0 + kGroup, na, nbv);
            const uint32_t wa = pack4(ca[0], ca[1], ca[2], ca[3]);
            uint32_t* xb = xchg + (g & 1u) * (8 * 32);
#pragma unroll
            for (int jj = 0; jj < kMyB; ++jj) xb[(q + 4 * jj) * 32 + lane] = pack4(cbv[0][jj], cbv[1][jj], cbv[2][jj], cbv[3][jj]);
#pragma unroll
            for (int b = 0; b < kGroup; ++b) {
                check(ca[b]);
#pragma unroll
                for (int jj = 0; jj < kMyB; ++jj) check(cbv[b][jj]);
            }
            // the four scale warps (128 threads) have written this group's words
            asm volatile("bar.sync 1, 128;" ::: "memory");
            uint32_t wb[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) wb[j] = xb[j * 32 + lane];
            // The MMAs of group g - 2 are done with slot g % 2.  A warp whose
            // wait expired keeps looping (without waiting or storing) so that
            // the four warps meet at every named barrier the same number of
            // times; the raised abort flag ends the others' waits quickly.
            bool got = ok;
            if (ok && lane == 0) got = mbar_wait_bounded(&sfe[g & 1u], ((g >> 1) & 1u) ^ 1u, abort_s);
            ok = __shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) != 0;
            if (ok) {
                tc_fence_after();
                const uint32_t sf = tmem_base + t_lane + slot_col(g & 1u);
                tmem_st_32x32b_x4(sf, wa, wa, wa, wa);
                tmem_st_32x32b_x8(sf + 8, wb);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR) mbar_arrive_cluster(sff0 + (g & 1u) * 8); else mbar_arrive(&sff[g & 1u]);
                }
            }
        }
        const bool bad = chk_max >= 0x7F000000u || chk_mant != 0;
        if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) mx_record(FP8_ERR_SCALE);
        if (!ok && lane == 0) mx_record(FP8_ERR_TIMEOUT);
    } else {
        // ================= epilogue warps (each CTA): row r of the CTA's 128
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t t_lane = uint32_t(32 * q) << 16;
        const uint32_t acce0 = PAIR ? mapa_shared(&acce[0], 0) : 0u;
        uint32_t tc = 0;
        bool ok = true;
        for (int64_t w = cluster; ok && w < num_tiles; w += nclusters, ++tc) {
            const uint32_t buf = tc & 1u;
            const TileAt t = tile_at(w);
            const int64_t m = t.row0 + r, n0 = t.n0;
            bool got = true;
            if (lane == 0) got = mbar_wait_bounded(&accf[buf], (tc >> 1) & 1u, abort_s);
            got = __shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) != 0;
            if (!got) { ok = false; break; }
            tc_fence_after();
            const uint32_t tcol = tmem_base + t_lane + buf * kAccStride;
#pragma unroll 1
            for (int c = 0; c < kBCols; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tcol + 32 * c, v);
                tmem_wait_ld_regs(v);
                const int64_t n = n0 + 32 * c;
                if (m < t.row_end && m < args.M && n < args.N) {
                    if constexpr (OUT_F32) {
                        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(args.d) + m * args.N + n);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(args.d) + m * args.N + n);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(
                                cvt_bf16x2(__uint_as_float(v[8 * i]), __uint_as_float(v[8 * i + 1])),
                                cvt_bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                                cvt_bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                                cvt_bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_cluster(acce0 + buf * 8); else mbar_arrive(&acce[buf]);
            }
        }
        if (!ok && lane == 0) mx_record(FP8_ERR_TIMEOUT);
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, kTmemCols); else tmem_dealloc(tmem_base, kTmemCols);
    }
}

constexpr int kStages = 7;           // a pair: 30 KB of operands per stage and CTA
constexpr int kSingleStages = 4;     // one CTA: 44 KB per stage

template <bool PAIR, int BMODE, bool OUT_F32, bool GROUPED>
static int launch(const CUtensorMap& ma, const CUtensorMap& mb, const Args& args, int sms, cudaStream_t stream) {
    constexpr int S = PAIR ? kStages : kSingleStages;
    using Lay = Layout<PAIR, S, GROUPED>;
    auto kern = gemm_mx_pair_kernel<PAIR, S, BMODE, OUT_F32, GROUPED>;
    static unsigned char smem_opted_in[kMaxDevices] = {};
    if (!opt_in_dynamic_smem(kern, Lay::kDynSmem, smem_opted_in)) return FP8_ERR_CUDA;
    // a programmatic dependent launch (the kernel waits before its first
    // global access), as the promoted GEMMs
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay::kDynSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    if constexpr (!PAIR) {
        // one CTA per SM (shared memory and launch bounds allow no more)
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(sms);
        if (cudaLaunchKernelEx(&cfg, kern, ma, mb, args) != cudaSuccess) return FP8_ERR_CUDA;
        return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
    }
    cfg.numAttrs = 2;
    int max_clusters = 0;
    cfg.gridDim = dim3(2 * (sms / 2));
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess || max_clusters <= 0)
        return FP8_ERR_CUDA;
    const int clusters = max_clusters < sms / 2 ? max_clusters : sms / 2;
    cfg.gridDim = dim3(2 * clusters);
    if (cudaLaunchKernelEx(&cfg, kern, ma, mb, args) != cudaSuccess) return FP8_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace mx
}  // namespace fp8bs

using namespace fp8bs;

extern "C" int fp8_gemm_blockscaled_pow2(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                                         int b_scale_mode, void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                                         fp8_stream_t stream) {
    if (!a || !sa || !b || !sb || !d || M <= 0 || N <= 0 || K <= 0) return FP8_ERR_ARG;
    if ((b_scale_mode != FP8_BSCALE_BLOCK128 && b_scale_mode != FP8_BSCALE_ROW) ||
        (d_dtype != FP8_OUT_BF16 && d_dtype != FP8_OUT_F32))
        return FP8_ERR_ARG;
    if (K % 128 || N % 128) return FP8_ERR_SHAPE;
    if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1) return FP8_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || !aligned16(sa) || !aligned16(sb)) return FP8_ERR_ALIGN;
    const int sms = device_sms();
    if (sms <= 0) return FP8_ERR_DEVICE;
    CUtensorMap ma, mb;
    if (!make_operand_map(&ma, a, M, K, mx::BM, 1, false) || !make_operand_map(&mb, b, N, K, mx::BN / 2, 1, false))
        return FP8_ERR_CUDA;
    const mx::Args args{sa, sb, d, M, N, K, nullptr, 0};
    const int64_t pair_tiles = ((M + 2 * mx::BM - 1) / (2 * mx::BM)) * ((N + mx::BN - 1) / mx::BN);
    if (pair_tiles * (K / 128) >= (int64_t(1) << 31) || N + mx::BN >= (int64_t(1) << 31)) return FP8_ERR_SHAPE;
    const int grid_sms = int(2 * pair_tiles < sms ? 2 * pair_tiles : sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (b_scale_mode == FP8_BSCALE_BLOCK128) {
        if (d_dtype == FP8_OUT_BF16) return mx::launch<true, 0, false, false>(ma, mb, args, grid_sms, s);
        return mx::launch<true, 0, true, false>(ma, mb, args, grid_sms, s);
    }
    if (d_dtype == FP8_OUT_BF16) return mx::launch<true, 1, false, false>(ma, mb, args, grid_sms, s);
    return mx::launch<true, 1, true, false>(ma, mb, args, grid_sms, s);
}

extern "C" int fp8_grouped_gemm_blockscaled_pow2(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
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
    // at most total_rows/128 + E row tiles, each with ceil(N/224) column tiles of K/128 blocks
    const int64_t max_tiles = (total_rows / mx::BM + E) * ((N + mx::BN - 1) / mx::BN);
    if (max_tiles * (K / 128) >= (int64_t(1) << 31) || int64_t(E) * (N / 128) * (K / 128) >= (int64_t(1) << 31) ||
        N + mx::BN >= (int64_t(1) << 31))
        return FP8_ERR_SHAPE;
    const int sms = device_sms();
    if (sms <= 0) return FP8_ERR_DEVICE;
    CUtensorMap ma, mb;
    if (!make_operand_map(&ma, a, total_rows, K, mx::BM, 1, false) ||
        !make_operand_map(&mb, b, N, K, mx::BN, E, true))
        return FP8_ERR_CUDA;
    const mx::Args args{sa, sb, d, total_rows, N, K, expert_offsets, E};
    // one CTA per 128 x 224 tile: experts hold ~128 rows on average, so a
    // 256-row pair tile would spend half its MMAs on padding rows
    return mx::launch<false, 0, false, true>(ma, mb, args, sms, reinterpret_cast<cudaStream_t>(stream));
}

// Status word of this translation unit: read and clear (synchronising).
extern "C" int fp8bs_gemm_mx_take_status(cudaStream_t stream) {
    int v = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP8_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_mx_status, sizeof v) != cudaSuccess) return FP8_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_mx_status, &zero, sizeof zero) != cudaSuccess) return FP8_ERR_CUDA;
    return v;
}
