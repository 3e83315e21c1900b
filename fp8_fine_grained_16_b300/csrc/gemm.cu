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
// warpgroups.  Here the overlap comes from tensor memory instead:
//
//   warp 0        TMA producer: A (128 x 128 B) and B (BN x 128 B) tiles of
//                 one K block per pipeline stage, 128-byte swizzle.
//   warp 1        allocates TMEM and issues, per K block, four
//                 tcgen05.mma (K = 32 each) into one of two TMEM
//                 accumulators (BN fp32 columns each), then commits to the
//                 stage's "empty" barrier and the accumulator's "full"
//                 barrier.
//   warps 2, 3    idle (they only give their registers to the promotion warps)
//   warps 4..11   promotion: two warpgroups, one per half of the BN columns.
//                 Thread (warp w, lane l) owns tile row 32*(w%4)+l (TMEM
//                 lanes are tied to w%4).  Per K block it reads P_kb from
//                 TMEM, frees the accumulator, and adds P_kb * sA*sB into
//                 BN/2 fp32 registers.  While it does so the MMA warp is
//                 already filling the other accumulator with P_{kb+1}.
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
// Register split: the block launches with 168 registers per thread (384 x 168
// = 64512); warpgroup 0 (TMA, MMA, idle) gives back down to 40 and the two
// promotion warpgroups grow to 232: 128*40 + 256*232 = 64512.
constexpr int kTmemCols = 512;
constexpr int kMaxExperts = 1024;

template <int BN, int STAGES, int BMODE, bool GROUPED>
struct Layout {
    static constexpr int kABytes = BM * BK;
    static constexpr int kBBytes = BN * BK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStagesBytes = STAGES * kStageBytes;
    static constexpr int kBarOff = kStagesBytes;  // full[S], empty[S], tfull[2], tempty[2], done, sbar[2][2]
    static constexpr int kNumBars = 2 * STAGES + 9;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;       // tmem base, abort flag
    static constexpr int kSbOff = (kMiscOff + 16 + 15) & ~15;     // row-scale buffers [2][BN] (BMODE 1)
    static constexpr int kSbBytes = BMODE == 1 ? 2 * BN * 4 : 0;
    static constexpr int kGrpOff = kSbOff + kSbBytes;             // grouped: off[E+1], tile prefix[E+1]
    static constexpr int kGrpBytes = GROUPED ? 2 * (kMaxExperts + 1) * 4 : 0;
    static constexpr int kBytes = kGrpOff + kGrpBytes;
    static constexpr int kDynSmem = kBytes + 1024;                // slack for 1024-byte alignment
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
                            const GemmArgs args) {
    using L = Layout<BN, STAGES, BMODE, GROUPED>;
    static_assert(2 * BN <= kTmemCols, "two accumulators must fit in TMEM");
    static_assert(BN == 256, "one promotion half = 128 columns = one scale block and one column per warpgroup thread");
    constexpr int kHalf = BN / 2;          // columns per promotion warpgroup
    constexpr int kChunks = kHalf / 32;
    constexpr uint32_t kIdesc = idesc_e4m3_f32(BM, BN);
    constexpr uint32_t kTxBytes = L::kABytes + L::kBBytes;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = bars + 2 * STAGES + 2;
    uint64_t* done = bars + 2 * STAGES + 4;
    uint64_t* sbar = bars + 2 * STAGES + 5;      // row-scale buffer barriers [half][buffer] (BMODE 1)
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_s = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t nkb = args.K / BK;

    // ---------------- set-up
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kPromoThreads);
        }
        mbar_init(done, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&sbar[i], 128);
        *abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
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

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 40;");
        if (warp == 0) {
            // ================= TMA producer
            if (lane == 0) {
                uint32_t it = 0;
                bool ok = true;
                for (int64_t w = blockIdx.x; ok && w < num_tiles; w += gridDim.x) {
                    const Tile t = tile_at(w);
                    for (int64_t kb = 0; kb < nkb; ++kb) {
                        const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
                        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_s)) {
                            ok = false;
                            break;
                        }
                        uint8_t* sa_tile = smem + stage * L::kStageBytes;
                        uint8_t* sb_tile = sa_tile + L::kABytes;
                        mbar_arrive_expect_tx(&full[stage], kTxBytes);
                        tma_load_2d(sa_tile, &tmA, &full[stage], int32_t(kb * BK), int32_t(t.row0));
                        if constexpr (GROUPED)
                            tma_load_3d(sb_tile, &tmB, &full[stage], int32_t(kb * BK), t.n0, t.e);
                        else
                            tma_load_2d(sb_tile, &tmB, &full[stage], int32_t(kb * BK), t.n0);
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
        } else if (warp == 1) {
            // ================= MMA issuer
            if (lane == 0) {
                uint32_t it = 0, g = 0;
                bool ok = true;
                for (int64_t w = blockIdx.x; ok && w < num_tiles; w += gridDim.x) {
                    for (int64_t kb = 0; kb < nkb; ++kb) {
                        const uint32_t buf = g & 1u, tphase = (g >> 1) & 1u;
                        if (!mbar_wait_bounded(&tempty[buf], tphase ^ 1u, abort_s)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
                        if (!mbar_wait_bounded(&full[stage], phase, abort_s)) { ok = false; break; }
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
        float* sbuf = reinterpret_cast<float*>(smem + L::kSbOff);   // [2][BN], BMODE 1
        const int wg_tid = threadIdx.x - 128 - half * 128;          // 0..127 within the warpgroup
        uint32_t g = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; ok && w < num_tiles; w += gridDim.x) {
            const Tile t = tile_at(w);
            const int64_t m = t.row0 + r;
            const int64_t m_ld = m < args.M ? m : args.M - 1;     // in-bounds row for scale loads
            const int64_t ncol0 = int64_t(t.n0) + half * kHalf;   // first column of this thread's half
            // N % 128 == 0, so a half tile (128 columns) is either entirely
            // inside [0, N) or entirely past it (last tile of an N that is an
            // odd multiple of 128); a half past N loads in-bounds scales and
            // stores nothing.
            const bool cols_ok = ncol0 < args.N;
            const int64_t ncol_ld = cols_ok ? ncol0 : args.N - kHalf;
            const float* sb_e = args.sb;
            if constexpr (GROUPED) sb_e += int64_t(t.e) * (args.N / 128) * nkb;

            auto load_sa = [&](int64_t kb) { return __ldg(args.sa + kb * args.M + m_ld); };
            auto load_sb = [&](int64_t kb) -> float {
                if constexpr (BMODE == 0) return __ldg(sb_e + (ncol_ld / 128) * nkb + kb);
                else return __ldg(sb_e + kb * args.N + ncol_ld + wg_tid);
            };

            float acc[kHalf];
#pragma unroll
            for (int i = 0; i < kHalf; ++i) acc[i] = 0.0f;
            float sa_next = load_sa(0), sb_next = load_sb(0);

            for (int64_t kb = 0; kb < nkb; ++kb) {
                const float sa_cur = sa_next, sb_cur = sb_next;
                if (kb + 1 < nkb) {
                    sa_next = load_sa(kb + 1);
                    sb_next = load_sb(kb + 1);
                }
                const uint32_t buf = g & 1u, tphase = (g >> 1) & 1u;
                if constexpr (BMODE == 1) {
                    // publish this K block's column scales to the warpgroup (double-buffered;
                    // a buffer is rewritten two blocks later, after every thread of the
                    // warpgroup has arrived on the next block's barrier)
                    sbuf[buf * BN + half * kHalf + wg_tid] = sb_cur;
                    mbar_arrive(&sbar[half * 2 + buf]);
                    if (!mbar_wait_bounded(&sbar[half * 2 + buf], tphase, abort_s)) { ok = false; break; }
                }
                if (!mbar_wait_bounded(&tfull[buf], tphase, abort_s)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tcol = tmem_base + t_lane + buf * BN + half * kHalf;
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tcol + c * 32, v);
                    tmem_wait_ld();
                    if (c == kChunks - 1) {
                        tc_fence_before();
                        mbar_arrive(&tempty[buf]);           // accumulator may be overwritten now
                    }
                    if constexpr (BMODE == 0) {
                        const float sc = __fmul_rn(sa_cur, sb_cur);
#pragma unroll
                        for (int i = 0; i < 32; ++i) acc[c * 32 + i] = fmaf(__uint_as_float(v[i]), sc, acc[c * 32 + i]);
                    } else {
                        const float4* sbv = reinterpret_cast<const float4*>(sbuf + buf * BN + half * kHalf + c * 32);
#pragma unroll
                        for (int i4 = 0; i4 < 8; ++i4) {
                            const float4 b4 = sbv[i4];
                            const float bs[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int i = i4 * 4 + j;
                                acc[c * 32 + i] = fmaf(__uint_as_float(v[i]), __fmul_rn(sa_cur, bs[j]), acc[c * 32 + i]);
                            }
                        }
                    }
                }
                ++g;
            }
            if (!ok) break;

            // ---- epilogue: this thread's row, BN/2 consecutive columns
            if (cols_ok && m < t.row_end && m < args.M) {
                if constexpr (OUT_F32) {
                    float* dst = reinterpret_cast<float*>(args.d) + m * args.N + ncol0;
#pragma unroll
                    for (int i = 0; i < kHalf; i += 4)
                        *reinterpret_cast<float4*>(dst + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
                } else {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(args.d) + m * args.N + ncol0;
#pragma unroll
                    for (int i = 0; i < kHalf; i += 8) {
                        const uint4 o = make_uint4(cvt_bf16x2(acc[i], acc[i + 1]), cvt_bf16x2(acc[i + 2], acc[i + 3]),
                                                   cvt_bf16x2(acc[i + 4], acc[i + 5]),
                                                   cvt_bf16x2(acc[i + 6], acc[i + 7]));
                        *reinterpret_cast<uint4*>(dst + i) = o;
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

static int device_sms() {
    int dev = 0, n = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess || major != 10) return -1;
    return n;
}

template <int BN, int STAGES, int BMODE, bool OUT_F32, bool GROUPED>
static int launch(const CUtensorMap& ma, const CUtensorMap& mb, const GemmArgs& args, int grid, cudaStream_t stream) {
    using L = Layout<BN, STAGES, BMODE, GROUPED>;
    auto kern = gemm_blockscaled_kernel<BN, STAGES, BMODE, OUT_F32, GROUPED>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynSmem) != cudaSuccess)
            return FP8_ERR_CUDA;
        attr_set = true;
    }
    kern<<<grid, kThreads, L::kDynSmem, stream>>>(ma, mb, args);
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
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || (reinterpret_cast<uintptr_t>(sa) & 3u) ||
        !aligned16(sb))
        return FP8_ERR_ALIGN;
    const int sms = device_sms();
    if (sms <= 0) return FP8_ERR_DEVICE;
    CUtensorMap ma, mb;
    if (!make_operand_map(&ma, a, M, K, BM, 1, false) || !make_operand_map(&mb, b, N, K, kBN, 1, false))
        return FP8_ERR_CUDA;
    GemmArgs args{sa, sb, d, nullptr, M, N, K, 0};
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + kBN - 1) / kBN);
    const int grid = int(tiles < sms ? tiles : sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (b_scale_mode == FP8_BSCALE_BLOCK128) {
        if (d_dtype == FP8_OUT_BF16) return launch<kBN, kStages, 0, false, false>(ma, mb, args, grid, s);
        return launch<kBN, kStages, 0, true, false>(ma, mb, args, grid, s);
    }
    if (d_dtype == FP8_OUT_BF16) return launch<kBN, kStages, 1, false, false>(ma, mb, args, grid, s);
    return launch<kBN, kStages, 1, true, false>(ma, mb, args, grid, s);
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
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || (reinterpret_cast<uintptr_t>(sa) & 3u) ||
        (reinterpret_cast<uintptr_t>(sb) & 3u) || (reinterpret_cast<uintptr_t>(expert_offsets) & 3u))
        return FP8_ERR_ALIGN;
    const int sms = device_sms();
    if (sms <= 0) return FP8_ERR_DEVICE;
    CUtensorMap ma, mb;
    if (!make_operand_map(&ma, a, total_rows, K, BM, 1, false) || !make_operand_map(&mb, b, N, K, kBN, E, true))
        return FP8_ERR_CUDA;
    GemmArgs args{sa, sb, d, expert_offsets, total_rows, N, K, E};
    return launch<kBN, kStages, 0, false, true>(ma, mb, args, sms, reinterpret_cast<cudaStream_t>(stream));
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
