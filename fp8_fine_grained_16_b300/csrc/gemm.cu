// gemm.cu -- block-scaled FP8 GEMMs on tcgen05 (dense, Wgrad and MoE grouped).
//
// What is computed (the tmdrlife.com and gnrental.net pages: partial sums are accumulated by the tensor
// cores over a K interval, then copied out, multiplied by the scaling
// factors and added into FP32; the jp-study.kr page: the interval is 128 elements):
//
//   D[m][n] = sum_kb  sA[kb][m] * sB(n, kb) * P_kb[m][n],
//   P_kb    = A[:, 128kb : 128kb+128] * B[:, 128kb : 128kb+128]^T   (E4M3 MMA)
//
// The pages' Hopper scheme overlaps promotion with WGMMA by ping-ponging two
// warpgroups.  Here the overlap comes from tensor memory: the MMAs of K block
// kb+1 fill one TMEM accumulator while the CUDA cores promote P_kb out of the
// other.
//
// One persistent kernel serves every form.  A cluster of two CTAs on
// neighbouring SMs computes 256 x 256 output tiles with
// tcgen05.mma.cta_group::2 (M = 256): each CTA holds its 128 rows of A and
// half of the B tile in its own shared memory, and each CTA's TMEM receives
// its 128 rows of D.  Per K block a CTA moves 32 KB of operands through
// shared memory for 128 x 256 x 128 multiply-adds (a one-CTA 128 x 256 tile
// moves 48 KB for the same work).  The grouped (MoE) form runs the same code
// with one CTA per 128 x 256 tile (PAIR = false, tcgen05.mma.cta_group::1,
// a 4-stage ring): experts hold ~128 rows each, so a 256-row pair tile would
// spend half its MMAs on padding.  Roles, per CTA:
//
//   warp 0        TMA producer: A and B halves (128-byte swizzle) and the
//                 scales the promotion needs (sA of the CTA's 128 rows, sB of
//                 the tile's columns) into a 4-stage ring.
//   warp 1        allocates the pair's TMEM (two 256-column fp32
//                 accumulators); in the leader CTA it issues four MMAs
//                 (K = 32 each) per K block and commits them to both CTAs'
//                 barriers.
//   warps 2, 3    idle (they only give their registers to the promotion warps)
//   warps 4..11   promotion: two warpgroups, one per 128-column half.  Thread
//                 (warp w, lane l) owns row 32*(w%4)+l of its CTA's 128 rows
//                 (TMEM lanes are tied to w%4).  Per K block it reads P_kb
//                 from TMEM in two 64-column loads, frees the accumulator once
//                 all of it is in registers, and adds P_kb * sA*sB into 128
//                 fp32 registers with packed two-lane FMAs.  It frees a stage
//                 as soon as the scales it needs are in its own shared-memory
//                 slots.
//
// The kernel is persistent: each cluster walks a static list of pair tiles;
// stage and accumulator indices run on across tile boundaries, so the
// epilogue of one tile overlaps the first MMAs of the next.
//
// Tail split (dense forms).  When the tiles leave a last wave of
// at most half the clusters, those tail tiles are cut along K instead: each
// cluster, after its whole-K tiles, promotes one K range of one tail tile
// and writes that fp32 partial sum to a workspace slab.  A second kernel on
// the same stream adds a tile's slabs in K order and stores D (or quantises
// it, for the E4M3 output).  The result is the same sum of promoted K blocks,
// regrouped into per-range fp32 sums.
//
// Every pipeline wait is bounded (2 s).  A wait that expires records
// FP8_ERR_TIMEOUT in the device status word, raises the CTA's abort flag,
// and lets the CTA drain its copies in flight, release its tensor memory and
// exit (both CTAs meet at a final cluster barrier first).
#include "common.cuh"
#include "expert_sched.cuh"
#include "tail_split.cuh"
#include "tensor_map.cuh"

namespace fp8bs {

__device__ int g_gemm_status;

FP8_DEV void record_status(int code) { atomicCAS(&g_gemm_status, 0, code); }

constexpr int BM = 128;                 // tile rows (one tcgen05 M=128 MMA)
constexpr int BK = 128;                 // K block = promotion interval = scale block
constexpr int kThreads = 384;           // 12 warps = 3 warpgroups
constexpr int kPromoThreads = 256;      // warps 4..11
constexpr int kPromoWarps = kPromoThreads / 32;
constexpr int kTmemCols = 512;
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

struct GemmArgs {
    const float* sa;
    const float* sb;
    void* d;                 // bf16 / fp32 output, or the E4M3 codes of D
    const int32_t* off;      // grouped only
    int64_t M;               // dense: rows of A / D; grouped: total_rows
    int64_t N;
    int64_t K;
    int E;                   // grouped only
    float* s_out;            // E4M3 output: 1x128 scales of D, [N/128][M]
    uint32_t flags;          // E4M3 output: FP8_SCALE_POW2
    float* ws = nullptr;     // tail split: [tail tiles * split][256][256] fp32 partial sums
    int64_t tail0 = 0;       // tail split: first split tile; tiles below it run over the whole K
    int32_t split = 0;       // tail split: K ranges per tail tile (0: no split)
};

// Output forms of the GEMM.
constexpr int kOutBF16 = 0, kOutF32 = 1, kOutE4M3 = 2;

// With per-column B scales (the Wgrad form, BMODE 1) every element of P_kb
// takes its own product of a row and a column scale, and a thread that owns
// one row x 128 columns must receive 128 column scales per K block from
// shared memory (the warp's 32 threads all need the same ones).  That
// broadcast, 128 KB per CTA per K block, is what bounds the promotion.  The
// two-row promotion reads P_kb with the 16-lane TMEM load (tcgen05.ld.16x256b),
// which gives each thread two rows x 64 columns: half the column scales per
// thread for the same number of elements.  The E4M3 output keeps the
// one-row layout, whose thread holds a whole 1x128 output tile.
__host__ __device__ constexpr bool two_row_promotion(int bmode, int out) { return bmode == 1 && out != kOutE4M3; }

struct Tile {
    int64_t row0;            // first row of the tile (global row index)
    int64_t row_end;         // rows >= row_end are not stored
    int32_t n0;              // column tile index from a schedule; first column after tile_at
    int32_t e;               // expert (grouped)
};

// ================================================================ kernel
// The leader (rank 0) issues tcgen05.mma.cta_group::2; both CTAs keep their
// A rows and B half at the same shared-memory offsets.
//
//   producer (warp 0, each CTA)  TMA-loads its A and B halves, counted on the
//                                leader's full[s] (the leader expects both
//                                CTAs' bytes), and its own scales, counted on
//                                its own sfull[s].
//   MMA (warp 1, leader only)    waits full[s], issues four MMAs, and commits
//                                to empty[s] and sfull[s] of both CTAs
//                                (multicast).
//   promotion (warps 4..11)      on the CTA's own TMEM rows.
//
// Every role waits on one barrier per K block (a probe costs ~190 cycles):
//   full[s]  (leader)  = producer's arrival + both CTAs' operand bytes + the
//                        16 promotion warps that freed the TMEM accumulator
//                        this K block will overwrite (K block g uses buffer
//                        g % 2, freed by the promotion of K block g - 2; the
//                        first two K blocks find their buffers free: every
//                        promotion warp pre-arrives on full[0] and full[1]).
//   sfull[s] (each)    = producer's arrival + this CTA's scale bytes + the
//                        MMA commit of that K block (its accumulator is ready).
//   empty[s] (each)    = MMA commit + this CTA's 8 promotion warps (each
//                        arrives once it has copied the scales it reads).
constexpr int kPairStages = 4;
constexpr int kSingleStages = 4;     // one CTA holds all 256 B rows: 48 KB of operands per stage
// Register split (launched with 168 per thread, 64512 in all): warpgroup 0
// keeps 64 (the producer's per-K-block state spills at 40), the promotion
// warpgroups get 216 (128 accumulators + one 32-column TMEM batch +
// addressing):
// 128*64 + 256*216 = 63488 <= 64512.
constexpr int kPairRegsWG0 = 64, kPairRegsPromo = 216;
static_assert(128 * kPairRegsWG0 + 256 * kPairRegsPromo <= kThreads * 168, "register split");

constexpr int kOutStageChunk = 32 * 64;                 // one staging tile: 32 rows x 64 bytes

template <bool PAIR, int BN, int STAGES, int BMODE, bool GROUPED, bool TWO_ROW = false>
struct PairLayout {
    static constexpr int kABytes = BM * BK;                      // this CTA's 128 rows
    static constexpr int kBBytes = (PAIR ? BN / 2 : BN) * BK;    // this CTA's half of B (all of it alone)
    static constexpr int kSaOff = kABytes + kBBytes;
    static constexpr int kSbOff = kSaOff + kSaRegion;
    static constexpr int kSbRegion = BMODE == 1 ? BN * 4 : 2 * kSbHalf0 * 4;
    static constexpr int kStageBytes = (kSbOff + kSbRegion + 1023) & ~1023;
    static constexpr uint32_t kPairTxBytes = (PAIR ? 2 : 1) * (kABytes + kBBytes);   // leader's full[s]: both CTAs
    static constexpr uint32_t kScaleTxBytes = kSaBox * 4 + (BMODE == 1 ? BN * 4 : 2 * kSbBox0 * 4);
    static constexpr int kStagesBytes = STAGES * kStageBytes;
    static constexpr int kBarOff = kStagesBytes;  // full[S], sfull[S], empty[S], done
    static constexpr int kNumBars = 3 * STAGES + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;       // tmem base, abort flag
    // Promotion warps' own copies of the scales they read from a stage (so the
    // stage can be freed at once): per warp, a slot per lane for its row scale
    // or scale product, and in BMODE 1 two buffers of its half's 128 column
    // scales (alternating K blocks).
    static constexpr int kPrivOff = (kMiscOff + 16 + 15) & ~15;
    static constexpr int kPrivRowBytes = kPromoWarps * 32 * 4;
    static constexpr int kPrivColOff = kPrivOff + kPrivRowBytes;
    // (with the two-row promotion every warp holds all BN column scales)
    static constexpr int kPrivColBytes = BMODE == 1 ? 2 * kPromoWarps * (TWO_ROW ? BN : BN / 2) * 4 : 0;
    static constexpr int kGrpOff = kPrivColOff + kPrivColBytes;
    static constexpr int kGrpBytes = GROUPED ? 2 * (kMaxExperts + 1) * 4 : 0;
    // one-row promotion: each warp's output staging tile (32 rows x 64 bytes);
    // not with per-column B scales, whose scale buffers leave no room for it
    static constexpr int kOutStageOff = (kGrpOff + kGrpBytes + 1023) & ~1023;
    // two staging tiles per warp (alternating by chunk) where they fit, else one
    static constexpr int kOutStageBufs =
        (TWO_ROW || BMODE == 1) ? 0 : (kOutStageOff + 2 * kPromoWarps * kOutStageChunk + 1024 <= 232448 ? 2 : 1);
    static constexpr int kOutStageWarpBytes = kOutStageBufs * kOutStageChunk;
    static constexpr int kOutStageBytes = kPromoWarps * kOutStageWarpBytes;
    static constexpr int kBytes = kOutStageOff + kOutStageBytes;
    static constexpr int kDynSmem = kBytes + 1024;
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0 && kStageBytes % 1024 == 0,
                  "operand tiles start on 1024-byte boundaries");
    static_assert(kSaOff % 128 == 0 && kSbOff % 128 == 0, "scale boxes start on 128-byte boundaries");
    static_assert(kDynSmem <= 232448, "shared memory per CTA");
};

// Dense tiles of `rows` rows (256 for a CTA pair, 128 for one CTA):
// w -> row tile w % num_m2, column tile w / num_m2.
struct DensePairSched {
    int64_t num_m2, num_n, M;
    int rows;
    FP8_DEV int64_t count() const { return num_m2 * num_n; }
    FP8_DEV Tile get(int64_t w) const {
        Tile t;
        t.row0 = (w % num_m2) * rows;
        t.row_end = M;
        t.n0 = int32_t(w / num_m2);
        t.e = 0;
        return t;
    }
};

// Grouped tiles: the per-expert list of expert_sched.cuh.
struct GroupedPairSched {
    const int32_t* off_s;
    const int32_t* pre_s;    // prefix of row-tile counts [E+1]
    int E;
    int64_t num_n;
    int rows;
    FP8_DEV int64_t count() const { return int64_t(pre_s[E]) * num_n; }
    FP8_DEV Tile get(int64_t w) const {
        const ExpertTile x = expert_tile(off_s, pre_s, E, num_n, w, rows);
        Tile t;
        t.e = x.e;
        t.n0 = int32_t(x.col_tile);
        t.row0 = x.row0;
        t.row_end = x.row_end;
        return t;
    }
};

template <bool PAIR, int BN, int STAGES, int BMODE, int OUT, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                     const __grid_constant__ CUtensorMap tmD, const GemmArgs args) {
    // Per-column B scales (BMODE 1, bf16/fp32 out): the two-row promotion
    constexpr bool kTwoRow = two_row_promotion(BMODE, OUT);
    using L = PairLayout<PAIR, BN, STAGES, BMODE, GROUPED, kTwoRow>;
    static_assert(2 * BN <= kTmemCols, "two accumulators must fit in TMEM");
    static_assert(BN == 256, "one promotion half = 128 columns = one scale block and one column per warpgroup thread");
    constexpr int kHalf = BN / 2;
    constexpr int kCtas = PAIR ? 2 : 1;
    constexpr int kTileRows = kCtas * BM;
    constexpr uint32_t kIdesc = idesc_e4m3_f32(kTileRows, BN);  // M = 256 across a pair, 128 alone

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* full = bars;                       // leader: operands of both CTAs + accumulator free
    uint64_t* sfull = bars + STAGES;             // own scales + accumulator ready
    uint64_t* empty = bars + 2 * STAGES;         // MMA commit + own promotion warps
    uint64_t* done = bars + 3 * STAGES;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_s = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int64_t nkb = args.K / BK;
    // a "cluster" is the pair, or the CTA itself
    const int64_t cluster = PAIR ? blockIdx.x >> 1 : blockIdx.x, nclusters = PAIR ? gridDim.x >> 1 : gridDim.x;

    // ---------------- set-up
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1 + kCtas * kPromoWarps);
            mbar_init(&sfull[i], 2);
            mbar_init(&empty[i], 1 + kPromoWarps);
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

    GroupedPairSched gs{};
    DensePairSched ds{};
    if constexpr (GROUPED) {
        int32_t* off_s = reinterpret_cast<int32_t*>(smem + L::kGrpOff);
        int32_t* pre_s = off_s + (kMaxExperts + 1);
        const int E = args.E;
        if (expert_tile_prefix(args.off, E, args.M, off_s, pre_s, kTileRows) && threadIdx.x == 0 && blockIdx.x == 0)
            record_status(FP8_ERR_OFFSETS);
        gs = GroupedPairSched{off_s, pre_s, E, (args.N + BN - 1) / BN, kTileRows};
    } else {
        ds = DensePairSched{(args.M + kTileRows - 1) / kTileRows, (args.N + BN - 1) / BN, args.M, kTileRows};
    }
    tc_fence_before();
    // Both CTAs' barriers are initialised and the TMEM is allocated before
    // either CTA touches the other's shared memory.
    if constexpr (PAIR) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_base_s;

    auto tile_at = [&](int64_t w) -> Tile {
        Tile t;
        if constexpr (GROUPED) t = gs.get(w); else t = ds.get(w);
        t.n0 *= BN;
        t.row0 += int64_t(rank) * BM;            // this CTA's 128 rows of the pair tile
        return t;
    };
    int64_t num_tiles;
    if constexpr (GROUPED) num_tiles = gs.count(); else num_tiles = ds.count();
    // This cluster's work units (tail_split.cuh): whole tiles, then under a
    // tail split one K range of one tail tile.
    const int64_t split = GROUPED ? 0 : int64_t(args.split);
    const int64_t n_units = pair_units(cluster, nclusters, num_tiles, split, args.tail0);
    auto unit_at = [&](int64_t i) -> WorkUnit {
        return pair_unit(i, cluster, nclusters, num_tiles, nkb, split, args.tail0);
    };
    auto sb_row = [&](const Tile& t, int h) -> int64_t {
        const int64_t c0 = int64_t(t.n0) + h * kHalf;
        return (int64_t(t.e) * (args.N / 128) + (c0 < args.N ? c0 : args.N - 1) / 128) * nkb;
    };

    // The two-row promotion (per-column B scales, bf16/fp32 out).  Warp
    // (w%4 = q, (w-4)/4 = hh) reads TMEM lanes 32q + 16hh .. +15 across all BN
    // columns with the 16x256b shape: thread t owns rows ra = 32q + 16hh + t/4
    // and ra + 8 of the CTA's 128 and, in every group of 8 columns, columns
    // 2(t%4) and 2(t%4) + 1 (64 columns of the 256).  Per K block it copies the
    // BN column scales into its own buffer (two 16-byte pieces per lane), frees
    // the stage, loads P_kb in two 128-column halves (64 registers each),
    // frees the accumulator after the second, and adds P * sB(column) * sA(row)
    // into 2 x 64 fp32 registers with packed two-lane operations.
    auto promote_two_rows = [&]() {
        const int wq = warp & 3, hh = (warp - 4) >> 2;
        const int lb = 32 * wq + 16 * hh;                  // first TMEM lane of this warp
        const int ra = lb + (lane >> 2), rb = ra + 8;      // the thread's two rows (of the CTA's 128)
        const int cp = 2 * (lane & 3);                      // its column pair in each group of 8
        const uint32_t t_lane = uint32_t(lb) << 16;
        const uint32_t full0 = PAIR ? mapa_shared(&full[0], 0) : smem_u32(&full[0]);
        auto release = [&](uint32_t stage_i) {
            if constexpr (PAIR) mbar_arrive_cluster(full0 + stage_i * 8); else mbar_arrive(&full[stage_i]);
        };
        __syncwarp();
        if (lane == 0) {
            release(0);
            release(1);
        }
        uint32_t g = 0;
        bool ok = true;
        for (int64_t ui = 0; ok && ui < n_units; ++ui) {
            const WorkUnit u = unit_at(ui);
            const Tile t = tile_at(u.w);
            const int sa_off0 = int(t.row0 & 3), m_step = int(args.M & 3);
            float2 acc_a[BN / 8], acc_b[BN / 8];
#pragma unroll
            for (int i = 0; i < BN / 8; ++i) acc_a[i] = acc_b[i] = make_float2(0.0f, 0.0f);

            for (int kb = int(u.kb0); kb < int(u.kb1); ++kb) {
                const uint32_t stage = g % STAGES, phase = (g / STAGES) & 1u;
                const uint32_t buf = g & 1u;
                bool got = true;
                if (lane == 0) got = mbar_wait_bounded(&sfull[stage], phase, abort_s);
                got = __shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) != 0;
                __syncwarp();
                if (!got) { ok = false; break; }
                tc_fence_after();

                const uint8_t* st = smem + stage * L::kStageBytes;
                const float* sab = reinterpret_cast<const float*>(st + L::kSaOff) + ((sa_off0 + kb * m_step) & 3);
                const float sa0 = sab[ra], sa1 = sab[rb];
                // this K block's copy of the BN column scales (buffer g % 2, last
                // read two K blocks ago); each value read from the stage goes into
                // a store of this warp before the stage is freed
                float* sbk = reinterpret_cast<float*>(smem + L::kPrivColOff) + ((g & 1u) * kPromoWarps + (warp - 4)) * BN;
#pragma unroll
                for (int i = 0; i < BN / 128; ++i)
                    reinterpret_cast<float4*>(sbk)[lane + 32 * i] =
                        reinterpret_cast<const float4*>(st + L::kSbOff)[lane + 32 * i];
                float* row_slot = reinterpret_cast<float*>(smem + L::kPrivOff) + (warp - 4) * 32 + lane;
                *row_slot = sa0 + sa1;
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);

                const float2 s0 = make_float2(sa0, sa0), s1 = make_float2(sa1, sa1);
                auto scale_half = [&](int hc, const uint32_t (&v)[64]) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int grp = 16 * hc + k;
                        const float2 sb = *reinterpret_cast<const float2*>(sbk + 8 * grp + cp);
                        const float2 pa = __fmul2_rn(make_float2(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1])), sb);
                        const float2 pb =
                            __fmul2_rn(make_float2(__uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3])), sb);
                        acc_a[grp] = __ffma2_rn(pa, s0, acc_a[grp]);
                        acc_b[grp] = __ffma2_rn(pb, s1, acc_b[grp]);
                    }
                };
                const uint32_t tcol = tmem_base + t_lane + buf * BN;
                uint32_t v[64];
                tmem_ld_16x256b_x16(tcol, v);
                tmem_wait_ld_regs64(v);
                scale_half(0, v);
                tmem_ld_16x256b_x16(tcol + 128, v);
                tmem_wait_ld_regs64(v);
                tc_fence_before();
                __syncwarp();
                // all of P_kb for this warp's 16 lanes is in registers:
                // accumulator `buf` is free for K block g + 2
                if (lane == 0) release((g + 2) % STAGES);
                scale_half(1, v);
                ++g;
            }
            if (!ok) break;

            if constexpr (!GROUPED) {
                if (u.slab >= 0) {
                    // K range of a split tile: the whole 256 x BN partial goes
                    // to its slab; the fix-up kernel adds the slabs
                    float* dst_a = args.ws + (u.slab * kTileRows + int64_t(rank) * BM + ra) * BN + cp;
                    float* dst_b = dst_a + 8 * BN;
#pragma unroll
                    for (int grp = 0; grp < BN / 8; ++grp) {
                        *reinterpret_cast<float2*>(dst_a + 8 * grp) = acc_a[grp];
                        *reinterpret_cast<float2*>(dst_b + 8 * grp) = acc_b[grp];
                    }
                    continue;
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int64_t m = t.row0 + (rr ? rb : ra);
                if (m >= t.row_end || m >= args.M) continue;
                const float2* acc = rr ? acc_b : acc_a;
#pragma unroll
                for (int grp = 0; grp < BN / 8; ++grp) {
                    const int64_t n = int64_t(t.n0) + 8 * grp + cp;
                    if (n >= args.N) break;
                    if constexpr (OUT == kOutF32)
                        *reinterpret_cast<float2*>(reinterpret_cast<float*>(args.d) + m * args.N + n) = acc[grp];
                    else
                        *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(args.d) + m * args.N + n) =
                            cvt_bf16x2(acc[grp].x, acc[grp].y);
                }
            }
        }
        if (!ok) record_status(FP8_ERR_TIMEOUT);
    };

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPairRegsWG0));
        if (warp == 0) {
            // ================= TMA producer (each CTA)
            if (lane == 0) {
                const uint32_t full0 = PAIR ? mapa_shared(&full[0], 0) : 0u;   // leader's full[0], cluster address
                uint32_t it = 0;
                bool ok = true;
                for (int64_t ui = 0; ok && ui < n_units; ++ui) {
                    const WorkUnit u = unit_at(ui);
                    const Tile t = tile_at(u.w);
                    int64_t sbr[2] = {0, 0};
                    if constexpr (BMODE == 0) {
                        sbr[0] = sb_row(t, 0);
                        sbr[1] = sb_row(t, 1);
                    }
                    for (int64_t kb = u.kb0; kb < u.kb1; ++kb) {
                        const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
                        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_s)) {
                            ok = false;
                            break;
                        }
                        uint8_t* st = smem + stage * L::kStageBytes;
                        const uint32_t fbar = full0 + stage * 8;
                        if (leader) mbar_arrive_expect_tx(&full[stage], L::kPairTxBytes);
                        if constexpr (PAIR) {
                            tma_load_2d_pair(st, &tmA, fbar, int32_t(kb * BK), int32_t(t.row0));
                            if constexpr (GROUPED)
                                tma_load_3d_pair(st + L::kABytes, &tmB, fbar, int32_t(kb * BK),
                                                 t.n0 + int32_t(rank) * (BN / 2), t.e);
                            else
                                tma_load_2d_pair(st + L::kABytes, &tmB, fbar, int32_t(kb * BK),
                                                 t.n0 + int32_t(rank) * (BN / 2));
                        } else {
                            tma_load_2d(st, &tmA, &full[stage], int32_t(kb * BK), int32_t(t.row0));
                            if constexpr (GROUPED)
                                tma_load_3d(st + L::kABytes, &tmB, &full[stage], int32_t(kb * BK), t.n0, t.e);
                            else
                                tma_load_2d(st + L::kABytes, &tmB, &full[stage], int32_t(kb * BK), t.n0);
                        }
                        mbar_arrive_expect_tx(&sfull[stage], L::kScaleTxBytes);
                        tma_load_1d(st + L::kSaOff, &tmSA, &sfull[stage], int32_t((kb * args.M + t.row0) & ~int64_t(3)));
                        if constexpr (BMODE == 0) {
                            tma_load_1d(st + L::kSbOff, &tmSB, &sfull[stage], int32_t((sbr[0] + kb) & ~int64_t(3)));
                            tma_load_1d(st + L::kSbOff + kSbHalf0 * 4, &tmSB, &sfull[stage],
                                        int32_t((sbr[1] + kb) & ~int64_t(3)));
                        } else {
                            tma_load_1d(st + L::kSbOff, &tmSB, &sfull[stage], int32_t(kb * args.N + t.n0));
                        }
                        ++it;
                    }
                }
                if (!ok) record_status(FP8_ERR_TIMEOUT);
                // Let this CTA's copies land before it can leave: its scales on
                // its own sfull[]; both CTAs' operand tiles on the leader's full[]
                // (the final cluster barrier holds the other CTA until then).
                int zero = 0;
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t j = first; j < it; ++j) {
                    mbar_wait_bounded(&sfull[j % STAGES], (j / STAGES) & 1u, reinterpret_cast<volatile int*>(&zero));
                    if (leader)
                        mbar_wait_bounded(&full[j % STAGES], (j / STAGES) & 1u, reinterpret_cast<volatile int*>(&zero));
                }
            }
            __syncwarp();
        } else if (warp == 1) {
            // ================= MMA issuer (leader only)
            if (leader && lane == 0) {
                uint32_t it = 0, g = 0;
                bool ok = true;
                for (int64_t ui = 0; ok && ui < n_units; ++ui) {
                    const WorkUnit u = unit_at(ui);
                    for (int64_t kb = u.kb0; kb < u.kb1; ++kb) {
                        const uint32_t buf = g & 1u;
                        const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
                        // operands of both CTAs landed and accumulator `buf` is free
                        if (!mbar_wait_bounded(&full[stage], phase, abort_s)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + stage * L::kStageBytes);
                        const uint32_t b_addr = a_addr + L::kABytes;
                        const uint64_t adesc = sw128_kmajor_desc(a_addr);
                        const uint64_t bdesc = sw128_kmajor_desc(b_addr);
                        const uint32_t d_tmem = tmem_base + buf * BN;
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            if constexpr (PAIR)
                                umma_e4m3_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, kIdesc, k > 0 ? 1u : 0u);
                            else
                                umma_e4m3(d_tmem, adesc + 2 * k, bdesc + 2 * k, kIdesc, k > 0 ? 1u : 0u);
                        }
                        if constexpr (PAIR) {
                            umma_commit_pair(&empty[stage], 0x3);
                            umma_commit_pair(&sfull[stage], 0x3);  // accumulator ready, in both CTAs
                        } else {
                            umma_commit(&empty[stage]);
                            umma_commit(&sfull[stage]);
                        }
                        ++it;
                        ++g;
                    }
                }
                if (!ok) record_status(FP8_ERR_TIMEOUT);
                if constexpr (PAIR) umma_commit_pair(done, 0x1); else umma_commit(done);
                int zero = 0;
                mbar_wait_bounded(done, 0, reinterpret_cast<volatile int*>(&zero));
            }
            __syncwarp();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPairRegsPromo));
        // ================= promotion warpgroups (each CTA, its own 128 rows)
        if constexpr (kTwoRow) {
            promote_two_rows();
        } else {
        const int wq = warp & 3;
        const int half = (warp - 4) >> 2;
        const int r = wq * 32 + lane;
        const uint32_t t_lane = uint32_t(wq * 32) << 16;
        // release on the leader's full[] (the CTA's own alone)
        const uint32_t full0 = PAIR ? mapa_shared(&full[0], 0) : smem_u32(&full[0]);
        auto release = [&](uint32_t stage_i) {
            if constexpr (PAIR) mbar_arrive_cluster(full0 + stage_i * 8); else mbar_arrive(&full[stage_i]);
        };
        // the two accumulators start out free: release them to K blocks 0 and 1
        __syncwarp();
        if (lane == 0) {
            release(0);
            release(1);
        }

        uint32_t g = 0;
        bool ok = true;
        for (int64_t ui = 0; ok && ui < n_units; ++ui) {
            const WorkUnit u = unit_at(ui);
            const Tile t = tile_at(u.w);
            // Where this K block's scales sit in the stage's boxes: the sA box
            // starts at (kb*M + row0) rounded down to 4 elements, the BMODE-0 sB
            // box at (sb_row + kb) rounded down to 4.  Both offsets advance by a
            // constant per K block (mod 4).
            const int sa_off0 = int(t.row0 & 3), m_step = int(args.M & 3);
            const int sb_off0 = BMODE == 0 ? int(sb_row(t, half) & 3) : 0;

            float2 acc[kHalf / 2];
#pragma unroll
            for (int i = 0; i < kHalf / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);

            for (int kb = int(u.kb0); kb < int(u.kb1); ++kb) {
                const uint32_t stage = g % STAGES, phase = (g / STAGES) & 1u;
                const uint32_t buf = g & 1u;
                // scales landed and the MMAs of this K block are done
                bool got = true;
                if (lane == 0) got = mbar_wait_bounded(&sfull[stage], phase, abort_s);
                got = __shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) != 0;
                __syncwarp();
                if (!got) { ok = false; break; }
                tc_fence_after();

                const uint8_t* st = smem + stage * L::kStageBytes;
                const float sa_cur = reinterpret_cast<const float*>(st + L::kSaOff)[((sa_off0 + kb * m_step) & 3) + r];
                const float2 sa2 = make_float2(sa_cur, sa_cur);
                float2 sc2 = sa2;
                // The warp frees the stage as soon as it has its scales.  Every
                // value it read from the stage first goes into a shared-memory
                // store of its own (a store cannot be made before its load
                // completes, and the release arrive orders it), so the stage's
                // next TMA refill cannot overtake a read.  Freeing the stage
                // while a read was still only feeding later FMAs let the refill
                // overwrite column scales not yet read: results varied from
                // run to run.
                float* row_slot = reinterpret_cast<float*>(smem + L::kPrivOff) + (warp - 4) * 32 + lane;
                const float* sbk = reinterpret_cast<const float*>(smem + L::kPrivColOff) +
                                   ((g & 1u) * kPromoWarps + (warp - 4)) * kHalf;
                if constexpr (BMODE == 0) {
                    const float sbv =
                        reinterpret_cast<const float*>(st + L::kSbOff)[half * kSbHalf0 + ((sb_off0 + kb) & 3)];
                    const float sc = __fmul_rn(sa_cur, sbv);
                    sc2 = make_float2(sc, sc);
                    *row_slot = sc;
                } else {
                    // this K block's copy of the half's column scales (buffer g % 2,
                    // last read two K blocks ago): one 16-byte piece per lane
                    const float4 b4 =
                        reinterpret_cast<const float4*>(reinterpret_cast<const float*>(st + L::kSbOff) + half * kHalf)[lane];
                    reinterpret_cast<float4*>(const_cast<float*>(sbk))[lane] = b4;
                    *row_slot = sa_cur;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);

                auto scale_chunk = [&](int c, const uint32_t* v) {
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

                // 64 columns at a time (two loads per K block): the second load's
                // wait frees the accumulator, and one 64-register batch beside
                // the 128 accumulators fits the promotion's register share
                const uint32_t tcol = tmem_base + t_lane + buf * BN + half * kHalf;
                uint32_t v[64];
                tmem_ld_32x32b_x64(tcol, v);
                tmem_wait_ld_regs64(v);
                scale_chunk(0, v);
                scale_chunk(1, v + 32);
                tmem_ld_32x32b_x64(tcol + 64, v);
                tmem_wait_ld_regs64(v);
                tc_fence_before();
                __syncwarp();
                // all of P_kb is in registers: accumulator `buf` is free for K
                // block g + 2 (on the leader's full[])
                if (lane == 0) release((g + 2) % STAGES);
                scale_chunk(2, v);
                scale_chunk(3, v + 32);
                ++g;
            }
            if (!ok) break;

            if constexpr (!GROUPED) {
                if (u.slab >= 0) {
                    // K range of a split tile: the whole 256 x 256 partial goes
                    // to its slab (rows and columns past D included); the
                    // fix-up kernel adds the slabs and applies the bounds
                    float* dst = args.ws + (u.slab * kTileRows + int64_t(rank) * BM + r) * BN + half * kHalf;
#pragma unroll
                    for (int i = 0; i < kHalf / 2; i += 2)
                        *reinterpret_cast<float4*>(dst + 2 * i) =
                            make_float4(acc[i].x, acc[i].y, acc[i + 1].x, acc[i + 1].y);
                    continue;
                }
            }
            const int64_t m = t.row0 + r;
            const int64_t ncol0 = int64_t(t.n0) + half * kHalf;
            if (ncol0 < args.N) {                  // N % 128 == 0: the whole half is inside D or outside it
                const bool row_ok = m < t.row_end && m < args.M;
                float inv = 1.0f;
                if constexpr (OUT == kOutE4M3) {
                    // The thread holds row m, columns ncol0 .. ncol0+127 of D in
                    // fp32: exactly one 1x128 activation tile of the next GEMM
                    // (its K runs along this GEMM's N).  Quantise it as the
                    // 1x128 quantiser does: fp32 amax, scale, x*inv, E4M3.
                    float amax = 0.0f;
#pragma unroll
                    for (int i = 0; i < kHalf / 2; ++i) amax = fmaxf(amax, fmaxf(fabsf(acc[i].x), fabsf(acc[i].y)));
                    const float sc = tile_scale(amax, (args.flags & FP8_SCALE_POW2) != 0, inv);
                    if (row_ok) args.s_out[(ncol0 / 128) * args.M + m] = sc;
                }
                if constexpr (L::kOutStageBytes == 0) {
                    // (per-column B scales, E4M3 out) the thread stores its own row
                    if (row_ok) {
                        uint8_t* dst = reinterpret_cast<uint8_t*>(args.d) + m * args.N + ncol0;
#pragma unroll
                        for (int i = 0; i < kHalf / 2; i += 8) {
                            uint32_t w[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                w[j] = cvt_e4m3x2(__fmul_rn(acc[i + 2 * j].x, inv), __fmul_rn(acc[i + 2 * j].y, inv)) |
                                       (cvt_e4m3x2(__fmul_rn(acc[i + 2 * j + 1].x, inv),
                                                   __fmul_rn(acc[i + 2 * j + 1].y, inv))
                                        << 16);
                            *reinterpret_cast<uint4*>(dst + 2 * i) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                } else {
                // The stores go through this warp's staging tile, 64 bytes of
                // each of its 32 rows at a time (16-byte piece j of row i at
                // piece j ^ ((i / 2) % 4), the 64-byte swizzle of the tensor
                // map of D: conflict-free both ways).  A warp whose 32 rows all
                // belong to the tile hands each chunk to one TMA tensor store;
                // at the end of an expert or of D the lanes store the rows that
                // belong, 64-byte segments of 8 rows per instruction.
                uint8_t* const stg_warp = smem + L::kOutStageOff + (warp - 4) * L::kOutStageWarpBytes;
                const int64_t m_warp = t.row0 + 32 * wq;
                const bool whole = m_warp + 32 <= t.row_end && m_warp + 32 <= args.M;     // warp-uniform
                constexpr int kElem = OUT == kOutF32 ? 4 : (OUT == kOutBF16 ? 2 : 1);
                constexpr int kChunkCols = 64 / kElem;
                const int swz = (lane >> 1) & 3;
#pragma unroll
                for (int c = 0; c < kHalf / kChunkCols; ++c) {
                    uint8_t* stg = stg_warp + (c % L::kOutStageBufs) * kOutStageChunk;
                    uint32_t w[16];
                    if constexpr (OUT == kOutBF16) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = cvt_bf16x2(acc[c * 16 + i].x, acc[c * 16 + i].y);
                    } else if constexpr (OUT == kOutF32) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            w[2 * i] = __float_as_uint(acc[c * 8 + i].x);
                            w[2 * i + 1] = __float_as_uint(acc[c * 8 + i].y);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 p0 = acc[c * 32 + 2 * i], p1 = acc[c * 32 + 2 * i + 1];
                            w[i] = cvt_e4m3x2(__fmul_rn(p0.x, inv), __fmul_rn(p0.y, inv)) |
                                   (cvt_e4m3x2(__fmul_rn(p1.x, inv), __fmul_rn(p1.y, inv)) << 16);
                        }
                    }
                    // the tensor store that last used this staging tile has read it
                    // (with two tiles, the most recent store may still be reading the other)
                    if (lane == 0) {
                        if constexpr (L::kOutStageBufs == 2) bulk_wait_group_read1(); else bulk_wait_group_read0();
                    }
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ swz) << 4)) =
                            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    if (whole) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmD, stg, int32_t(ncol0 + c * kChunkCols), int32_t(m_warp));
                            bulk_commit_group();
                        }
                    } else {
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int rr = 8 * i + (lane >> 2), pc = lane & 3;
                            const uint4 v =
                                *reinterpret_cast<const uint4*>(stg + rr * 64 + ((pc ^ ((rr >> 1) & 3)) << 4));
                            const int64_t mm = m_warp + rr;
                            if (mm < t.row_end && mm < args.M)
                                *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(args.d) +
                                                          (mm * args.N + ncol0 + c * kChunkCols) * kElem + pc * 16) = v;
                        }
                        __syncwarp();
                    }
                }
                }
            }
        }
        // this warp's tensor stores are complete before the CTA can leave
        if constexpr (L::kOutStageBytes > 0) {
            if (lane == 0) bulk_wait_group0();
            __syncwarp();
        }
        if (!ok) record_status(FP8_ERR_TIMEOUT);
        }
    }

    // ---------------- tear-down: neither CTA leaves (or frees TMEM) while the
    // other may still use its shared memory or tensor memory
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, kTmemCols); else tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Tail split fix-up: D over the split tiles = the sum of each tile's slabs,
// added in K order in fp32, then stored as the GEMM stores it.  Block b
// covers rows 4 * (b % 64) .. +3 of split tile b / 64; a thread adds four
// columns, so a warp holds one row x 128 columns: for the E4M3 output that
// is one 1x128 tile, quantised as the GEMM's epilogue does (amax over the
// warp, the same scale rule and conversion).
constexpr int kFixRowsPerBlock = 4;
template <int OUT>
__global__ void __launch_bounds__(256) splitk_fixup_kernel(const float* __restrict__ ws, void* __restrict__ d,
                                                          int64_t M, int64_t N, int64_t tail0, int split,
                                                          int64_t num_m2, float* __restrict__ s_out,
                                                          uint32_t flags) {
    constexpr int kTile = 256;
    const int64_t j = blockIdx.x / (kTile / kFixRowsPerBlock);
    const int row = int(blockIdx.x % (kTile / kFixRowsPerBlock)) * kFixRowsPerBlock + int(threadIdx.x >> 6);
    const int c = int(threadIdx.x & 63) * 4;
    const int64_t w = tail0 + j;
    const int64_t m = (w % num_m2) * kTile + row, n = (w / num_m2) * kTile + c;
    // a warp's 32 threads share m and the 128-column block of n: they leave together
    if (m >= M || n >= N) return;
    const float4* p = reinterpret_cast<const float4*>(ws + (j * split * kTile + row) * kTile + c);
    constexpr int64_t kSlab = int64_t(kTile) * kTile / 4;      // float4s per slab
    float4 acc = p[0];
#pragma unroll 4
    for (int sp = 1; sp < split; ++sp) {
        const float4 v = p[sp * kSlab];
        acc = make_float4(__fadd_rn(acc.x, v.x), __fadd_rn(acc.y, v.y), __fadd_rn(acc.z, v.z), __fadd_rn(acc.w, v.w));
    }
    if constexpr (OUT == kOutE4M3) {
        float amax = fmaxf(fmaxf(fabsf(acc.x), fabsf(acc.y)), fmaxf(fabsf(acc.z), fabsf(acc.w)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        float inv;
        const float sc = tile_scale(amax, (flags & FP8_SCALE_POW2) != 0, inv);
        *reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(d) + m * N + n) =
            cvt_e4m3x2(__fmul_rn(acc.x, inv), __fmul_rn(acc.y, inv)) |
            (cvt_e4m3x2(__fmul_rn(acc.z, inv), __fmul_rn(acc.w, inv)) << 16);
        if ((threadIdx.x & 31) == 0) s_out[(n / 128) * M + m] = sc;
    } else if constexpr (OUT == kOutF32) {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(d) + m * N + n) = acc;
    } else {
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(d) + m * N + n) =
            make_uint2(cvt_bf16x2(acc.x, acc.y), cvt_bf16x2(acc.z, acc.w));
    }
}

// ---------------------------------------------------------------- host side
constexpr int kBN = 256;
constexpr int64_t kSlabBytes = int64_t(2 * BM) * kBN * 4;     // one pair tile of fp32 K-range sums

// Workspace the tail split may use on this device: one slab per cluster.
static int64_t split_workspace_bytes(int sms, int64_t K) {
    return K / 128 >= kSplitMinKBlocks ? int64_t(sms / 2) * kSlabBytes : 0;
}

// D [rows][N] as boxes of 32 rows x 64 bytes with the 64-byte swizzle: the
// epilogue's tensor stores from its staging tiles.
static bool make_out_map(CUtensorMap* map, void* d, int64_t rows, int64_t N, int out) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int elem = out == kOutF32 ? 4 : (out == kOutBF16 ? 2 : 1);
    const CUtensorMapDataType dt = out == kOutF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                  : (out == kOutBF16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT8);
    cuuint64_t dims[2] = {cuuint64_t(N), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(N) * cuuint64_t(elem)};
    cuuint32_t box[2] = {cuuint32_t(64 / elem), 32u};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(map, dt, 2u, d, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool PAIR, int BN, int STAGES, int BMODE, int OUT, bool GROUPED>
static int launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msa, const CUtensorMap& msb,
                       GemmArgs args, int sms, cudaStream_t stream, int64_t ws_bytes = 0) {
    using L = PairLayout<PAIR, BN, STAGES, BMODE, GROUPED, two_row_promotion(BMODE, OUT)>;
    auto kern = gemm_pair_kernel<PAIR, BN, STAGES, BMODE, OUT, GROUPED>;
    CUtensorMap md;
    if (!make_out_map(&md, args.d, args.M, args.N, OUT)) return FP8_ERR_CUDA;
    static unsigned char smem_opted_in[kMaxDevices] = {};
    if (!opt_in_dynamic_smem(kern, L::kDynSmem, smem_opted_in)) return FP8_ERR_CUDA;
    // A programmatic dependent launch: the CTAs may start (barriers, TMEM,
    // descriptor prefetch) while the kernel before them on the stream drains,
    // and wait (griddepcontrol.wait) before their first global access.
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kDynSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    if constexpr (!PAIR) {
        // one CTA per SM (shared memory and launch bounds allow no more)
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(sms);
        if (cudaLaunchKernelEx(&cfg, kern, ma, mb, msa, msb, md, args) != cudaSuccess) return FP8_ERR_CUDA;
        return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
    }
    cfg.numAttrs = 2;
    int max_clusters = 0;
    cfg.gridDim = dim3(2 * (sms / 2));
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess || max_clusters <= 0)
        return FP8_ERR_CUDA;
    int clusters = max_clusters < sms / 2 ? max_clusters : sms / 2;
    // Tail split and the number of pairs to launch (tail_split.cuh): every
    // launched pair gets work, and the slabs never exceed one per pair.
    args.split = 0;
    int64_t num_m2 = 0, n_tail = 0;
    if constexpr (PAIR && !GROUPED) {
        num_m2 = (args.M + 2 * BM - 1) / (2 * BM);
        const int64_t num_tiles = num_m2 * ((args.N + BN - 1) / BN);
        const SplitPlan plan = plan_tail_split(num_tiles, args.K / BK, clusters, args.ws ? ws_bytes / kSlabBytes : 0);
        args.split = int32_t(plan.split);
        args.tail0 = plan.tail0;
        n_tail = num_tiles - plan.tail0;
        clusters = int(plan.pairs);
    }
    cfg.gridDim = dim3(2 * clusters);
    if (cudaLaunchKernelEx(&cfg, kern, ma, mb, msa, msb, md, args) != cudaSuccess) return FP8_ERR_CUDA;
    if constexpr (PAIR && !GROUPED) {
        if (args.split > 0) {
            const unsigned blocks = unsigned(n_tail * (2 * BM / kFixRowsPerBlock));
            splitk_fixup_kernel<OUT><<<blocks, 256, 0, stream>>>(args.ws, args.d, args.M, args.N, args.tail0,
                                                                  args.split, num_m2, args.s_out, args.flags);
        }
    }
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

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

static int gemm_blockscaled_impl(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                                 int b_scale_mode, void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                                 float* ws, int64_t ws_bytes, fp8_stream_t stream) {
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
    if (!make_operand_map(&ma, a, M, K, BM, 1, false) || !make_operand_map(&mb, b, N, K, kBN / 2, 1, false) ||
        !make_scale_map(&msa, sa, M * (K / 128), kSaBox) ||
        !make_scale_map(&msb, sb, nsb, b_scale_mode == FP8_BSCALE_ROW ? kBN : kSbBox0))
        return FP8_ERR_CUDA;
    GemmArgs args{sa, sb, d, nullptr, M, N, K, 0, nullptr, 0u};
    args.ws = ws;
    const int64_t pair_tiles = ((M + 2 * BM - 1) / (2 * BM)) * ((N + kBN - 1) / kBN);
    // with a workspace, fewer tiles than clusters are split along K over the
    // whole GPU; without one, a cluster per tile
    const bool may_split = ws && K / 128 >= kSplitMinKBlocks;
    const int grid_sms = int(may_split || 2 * pair_tiles >= sms ? sms : 2 * pair_tiles);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (b_scale_mode == FP8_BSCALE_BLOCK128) {
        if (d_dtype == FP8_OUT_BF16)
            return launch_pair<true, kBN, kPairStages, 0, kOutBF16, false>(ma, mb, msa, msb, args, grid_sms, s, ws_bytes);
        return launch_pair<true, kBN, kPairStages, 0, kOutF32, false>(ma, mb, msa, msb, args, grid_sms, s, ws_bytes);
    }
    if (d_dtype == FP8_OUT_BF16)
        return launch_pair<true, kBN, kPairStages, 1, kOutBF16, false>(ma, mb, msa, msb, args, grid_sms, s, ws_bytes);
    return launch_pair<true, kBN, kPairStages, 1, kOutF32, false>(ma, mb, msa, msb, args, grid_sms, s, ws_bytes);
}

extern "C" int fp8_gemm_blockscaled(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                                    int b_scale_mode, void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                                    fp8_stream_t stream) {
    return gemm_blockscaled_impl(a, sa, b, sb, b_scale_mode, d, d_dtype, M, N, K, nullptr, 0, stream);
}

// Columns of one 256-row pair tile of a GEMM form: every form uses 256 x 256
// tiles (the grouped form runs them as 128 x 256 single-CTA tiles).
extern "C" int fp8_gemm_tile_cols(int form) {
    return form == FP8_GEMM_FORM_DENSE || form == FP8_GEMM_FORM_Q8 || form == FP8_GEMM_FORM_GROUPED ? kBN
                                                                                                  : FP8_ERR_ARG;
}

extern "C" int fp8_gemm_split_plan(int form, int64_t M, int64_t N, int64_t K, int pairs, int64_t workspace_bytes,
                                   int64_t* split, int64_t* tail0, int64_t* launched_pairs) {
    if (form != FP8_GEMM_FORM_DENSE && form != FP8_GEMM_FORM_Q8) return FP8_ERR_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || pairs <= 0 || workspace_bytes < 0 || !split || !tail0 || !launched_pairs)
        return FP8_ERR_ARG;
    if (K % 128 || N % 128) return FP8_ERR_SHAPE;
    const int64_t num_tiles = ((M + 2 * BM - 1) / (2 * BM)) * ((N + kBN - 1) / kBN);
    const SplitPlan p = plan_tail_split(num_tiles, K / BK, pairs, workspace_bytes / kSlabBytes);
    *split = p.split;
    *tail0 = p.tail0;
    *launched_pairs = p.pairs;
    return FP8_OK;
}

extern "C" int64_t fp8_gemm_split_units(int form, int64_t M, int64_t N, int64_t K, int pairs,
                                        int64_t workspace_bytes, int64_t pair, int64_t* units, int64_t max_units) {
    int64_t split, tail0, np;
    const int rc = fp8_gemm_split_plan(form, M, N, K, pairs, workspace_bytes, &split, &tail0, &np);
    if (rc != FP8_OK) return rc;
    if (pair < 0 || pair >= np || max_units < 0 || (max_units > 0 && !units)) return FP8_ERR_ARG;
    const int64_t num_tiles = ((M + 2 * BM - 1) / (2 * BM)) * ((N + kBN - 1) / kBN);
    const int64_t n = pair_units(pair, np, num_tiles, split, tail0);
    for (int64_t i = 0; i < n && i < max_units; ++i) {
        const WorkUnit u = pair_unit(i, pair, np, num_tiles, K / BK, split, tail0);
        units[4 * i] = u.w;
        units[4 * i + 1] = u.kb0;
        units[4 * i + 2] = u.kb1;
        units[4 * i + 3] = u.slab;
    }
    return n;
}

extern "C" int64_t fp8_gemm_blockscaled_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return FP8_ERR_ARG;
    const int sms = device_sms();
    if (sms <= 0) return FP8_ERR_DEVICE;
    return split_workspace_bytes(sms, K);
}

extern "C" int fp8_gemm_blockscaled_ws(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                                       int b_scale_mode, void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                                       void* workspace, int64_t workspace_bytes, fp8_stream_t stream) {
    if (workspace_bytes < 0 || (workspace_bytes > 0 && !workspace)) return FP8_ERR_ARG;
    if (workspace && !aligned16(workspace)) return FP8_ERR_ALIGN;
    return gemm_blockscaled_impl(a, sa, b, sb, b_scale_mode, d, d_dtype, M, N, K,
                                 workspace_bytes > 0 ? static_cast<float*>(workspace) : nullptr, workspace_bytes,
                                 stream);
}

static int gemm_blockscaled_q8_impl(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                                    int b_scale_mode, uint8_t* q_out, float* s_out, uint32_t flags, int64_t M,
                                    int64_t N, int64_t K, float* ws, int64_t ws_bytes, fp8_stream_t stream) {
    if (!a || !sa || !b || !sb || !q_out || !s_out || M <= 0 || N <= 0 || K <= 0) return FP8_ERR_ARG;
    if ((b_scale_mode != FP8_BSCALE_BLOCK128 && b_scale_mode != FP8_BSCALE_ROW) || (flags & ~FP8_SCALE_POW2))
        return FP8_ERR_ARG;
    if (K % 128 || N % 128) return FP8_ERR_SHAPE;
    if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1) return FP8_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(q_out) || !aligned16(sa) || !aligned16(sb) ||
        (reinterpret_cast<uintptr_t>(s_out) & 3u))
        return FP8_ERR_ALIGN;
    if (M * (K / 128) >= (int64_t(1) << 31) || M * (N / 128) >= (int64_t(1) << 31) ||
        (b_scale_mode == FP8_BSCALE_ROW && N * (K / 128) >= (int64_t(1) << 31)))
        return FP8_ERR_SHAPE;
    const int sms = device_sms();
    if (sms <= 0) return FP8_ERR_DEVICE;
    CUtensorMap ma, mb, msa, msb;
    const int64_t nsb = b_scale_mode == FP8_BSCALE_ROW ? N * (K / 128) : (N / 128) * (K / 128);
    if (!make_operand_map(&ma, a, M, K, BM, 1, false) || !make_operand_map(&mb, b, N, K, kBN / 2, 1, false) ||
        !make_scale_map(&msa, sa, M * (K / 128), kSaBox) ||
        !make_scale_map(&msb, sb, nsb, b_scale_mode == FP8_BSCALE_ROW ? kBN : kSbBox0))
        return FP8_ERR_CUDA;
    GemmArgs args{sa, sb, q_out, nullptr, M, N, K, 0, s_out, flags};
    args.ws = ws;
    const int64_t pair_tiles = ((M + 2 * BM - 1) / (2 * BM)) * ((N + kBN - 1) / kBN);
    const bool may_split = ws && K / 128 >= kSplitMinKBlocks;
    const int grid_sms = int(may_split || 2 * pair_tiles >= sms ? sms : 2 * pair_tiles);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (b_scale_mode == FP8_BSCALE_BLOCK128)
        return launch_pair<true, kBN, kPairStages, 0, kOutE4M3, false>(ma, mb, msa, msb, args, grid_sms, s, ws_bytes);
    return launch_pair<true, kBN, kPairStages, 1, kOutE4M3, false>(ma, mb, msa, msb, args, grid_sms, s, ws_bytes);
}

extern "C" int fp8_gemm_blockscaled_q8(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                                       int b_scale_mode, uint8_t* q_out, float* s_out, uint32_t flags, int64_t M,
                                       int64_t N, int64_t K, fp8_stream_t stream) {
    return gemm_blockscaled_q8_impl(a, sa, b, sb, b_scale_mode, q_out, s_out, flags, M, N, K, nullptr, 0, stream);
}

extern "C" int fp8_gemm_blockscaled_q8_ws(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                                          int b_scale_mode, uint8_t* q_out, float* s_out, uint32_t flags, int64_t M,
                                          int64_t N, int64_t K, void* workspace, int64_t workspace_bytes,
                                          fp8_stream_t stream) {
    if (workspace_bytes < 0 || (workspace_bytes > 0 && !workspace)) return FP8_ERR_ARG;
    if (workspace && !aligned16(workspace)) return FP8_ERR_ALIGN;
    return gemm_blockscaled_q8_impl(a, sa, b, sb, b_scale_mode, q_out, s_out, flags, M, N, K,
                                    workspace_bytes > 0 ? static_cast<float*>(workspace) : nullptr,
                                    workspace_bytes, stream);
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
    GemmArgs args{sa, sb, d, expert_offsets, total_rows, N, K, E, nullptr, 0u};
    // one CTA per tile: experts hold ~128 rows on average, and each CTA streams
    // its own weight tiles, so twice as many tiles are in flight as with pairs
    return launch_pair<false, kBN, kSingleStages, 0, kOutBF16, true>(ma, mb, msa, msb, args, sms,
                                                                    reinterpret_cast<cudaStream_t>(stream));
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
