// transpose.cu -- transposed copy of a 128x128-block-quantised E4M3 matrix,
// for FP8 Dgrad (the why-be.why-be.co.kr (wr_id 35533) page: E4M3 for every
// tensor, in Fprop, Dgrad and Wgrad; the jp-study.kr page: weights are
// quantised per 128x128 block).
//
// The amax of a 128x128 block does not change when the block is transposed,
// so quantising W^T per 128x128 block gives exactly the transposed codes and
// the transposed grid of block scales of quantising W.  Dgrad,
// dX = dY * W, is then the block-scaled GEMM with A = dY (1x128 tiles) and
// B = W^T from this copy.
//
// A persistent kernel, one CTA per SM.  Warp 0 (one lane) streams the CTA's
// 128x128-byte blocks into an 8-stage ring with TMA tensor loads (128-byte
// swizzle: 16-byte piece j of tile row r sits at piece j ^ (r % 8)), so that
// 128 KB of loads per SM stay in flight while the blocks before them are
// transposed.  Each of four worker warps takes every fourth block: a thread
// transposes two 16x16-byte sub-blocks (sixteen 16-byte shared loads, 4x4 byte
// transposes in registers, sixteen 16-byte shared stores), writes them into the
// warp's own output tile in the same swizzled layout, and one lane stores that
// tile to W^T with a TMA tensor store (the warp copies its tiles' block
// scales up front, one tile per lane).  Thread (lane l) of sub-block pass b
// takes input piece column sx = l % 8 and input row group p = sx ^ (l / 8 + 4b):
// the eight threads of each 16-byte access phase then have distinct sx and
// distinct p, so both the swizzled loads (piece sx ^ (row % 8)) and stores
// (piece p ^ (row % 8)) hit eight different 16-byte bank groups.
//
// Every wait is bounded; an expired wait records FP8_ERR_TIMEOUT, the warps
// stop, and the producer lets its copies in flight land before the CTA exits.
#include "common.cuh"
#include "tensor_map.cuh"

namespace fp8bs {

__device__ int g_tr_status;
FP8_DEV void tr_record(int code) { atomicCAS(&g_tr_status, 0, code); }

constexpr int kTrStages = 8;                            // input ring depth (128x128-byte tiles)
constexpr int kTrWorkers = 4;                           // transposing warps
constexpr int kTrTile = 128 * 128;                      // bytes per tile
constexpr int kTrThreads = 32 * (1 + kTrWorkers);
constexpr int kTrBarOff = (kTrStages + kTrWorkers) * kTrTile;
constexpr int kTrSmem = kTrBarOff + 2 * kTrStages * 8 + 16 + 1024;   // + barriers, abort flag, 1024-byte alignment

// 4x4 byte transpose: in[r] holds bytes (r,0..3) little-endian; out[c] gets
// bytes (0..3,c).
FP8_DEV void transpose4x4(const uint32_t (&in)[4], uint32_t (&out)[4]) {
    const uint32_t t0 = __byte_perm(in[0], in[1], 0x5140);   // a0 b0 a1 b1
    const uint32_t t1 = __byte_perm(in[2], in[3], 0x5140);   // c0 d0 c1 d1
    const uint32_t t2 = __byte_perm(in[0], in[1], 0x7362);   // a2 b2 a3 b3
    const uint32_t t3 = __byte_perm(in[2], in[3], 0x7362);   // c2 d2 c3 d3
    out[0] = __byte_perm(t0, t1, 0x5410);                    // a0 b0 c0 d0
    out[1] = __byte_perm(t0, t1, 0x7632);                    // a1 b1 c1 d1
    out[2] = __byte_perm(t2, t3, 0x5410);                    // a2 b2 c2 d2
    out[3] = __byte_perm(t2, t3, 0x7632);                    // a3 b3 c3 d3
}

// Tile t of the CTA's list: block (nb, kb) of the [N/128][K/128] grid, kb fastest.
__global__ void __launch_bounds__(kTrThreads, 1) transpose_128x128_kernel(const __grid_constant__ CUtensorMap tmIn,
                                                                          const __grid_constant__ CUtensorMap tmOut,
                                                                          const float* __restrict__ s,
                                                                          float* __restrict__ sT, int64_t nnb,
                                                                          int64_t nkb) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* in_tiles = smem;
    uint8_t* out_tiles = smem + kTrStages * kTrTile;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTrBarOff);
    uint64_t* empty = full + kTrStages;
    volatile int* abort_s = reinterpret_cast<volatile int*>(empty + kTrStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = nnb * nkb;
    const int64_t my_tiles = int64_t(blockIdx.x) < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTrStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        *abort_s = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ================= TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmIn);
            bool ok = true;
            int64_t i = 0;
            for (; i < my_tiles; ++i) {
                const uint32_t st = uint32_t(i % kTrStages), ph = uint32_t(i / kTrStages) & 1u;
                if (!mbar_wait_bounded(&empty[st], ph ^ 1u, abort_s)) { ok = false; break; }
                const int64_t t = blockIdx.x + i * gridDim.x;
                const int64_t nb = t / nkb, kb = t - nb * nkb;
                mbar_arrive_expect_tx(&full[st], kTrTile);
                tma_load_2d(in_tiles + st * kTrTile, &tmIn, &full[st], int32_t(kb * 128), int32_t(nb * 128));
            }
            if (!ok) {
                tr_record(FP8_ERR_TIMEOUT);
                // the copies already issued land before the CTA's shared memory goes away
                int zero = 0;
                for (int64_t j = i > kTrStages ? i - kTrStages : 0; j < i; ++j)
                    mbar_wait_bounded(&full[j % kTrStages], uint32_t(j / kTrStages) & 1u,
                                      reinterpret_cast<volatile int*>(&zero));
            }
        }
        __syncwarp();
        return;
    }

    // ================= worker warps
    const int wk = warp - 1;
    uint8_t* out = out_tiles + wk * kTrTile;
    const int sx = lane & 7, tq = lane >> 3;
    // the block scales of this warp's tiles first, one tile per lane: the
    // loads are independent, so their latency is paid once per 32 tiles and
    // overlaps the first tile's copy instead of stalling every tile
    for (int64_t i = wk + int64_t(kTrWorkers) * lane; i < my_tiles; i += int64_t(kTrWorkers) * 32) {
        const int64_t t = blockIdx.x + i * gridDim.x;
        const int64_t nb = t / nkb, kb = t - nb * nkb;
        sT[kb * nnb + nb] = s[nb * nkb + kb];
    }
    bool ok = true;
    for (int64_t i = wk; i < my_tiles; i += kTrWorkers) {
        const uint32_t st = uint32_t(i % kTrStages), ph = uint32_t(i / kTrStages) & 1u;
        // every lane waits (acquiring the tile); the warp leaves together if any lane gave up
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[st], ph, abort_s))) { ok = false; break; }
        const uint8_t* in = in_tiles + st * kTrTile;
        // the previous store out of this warp's output tile has finished reading it
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int p = sx ^ (tq + 4 * b);                  // input rows 16p .. 16p+15
            uint4 v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = *reinterpret_cast<const uint4*>(in + (16 * p + j) * 128 + ((sx ^ (j & 7)) << 4));
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                // word w of the piece: input columns 16sx + 4w .. +3 = output rows c
                uint32_t o[4][4];                             // o[i][g]: output row 16sx+4w+i, word g of piece p
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint32_t a[4] = {(&v[4 * g].x)[w], (&v[4 * g + 1].x)[w], (&v[4 * g + 2].x)[w],
                                           (&v[4 * g + 3].x)[w]};
                    uint32_t r[4];
                    transpose4x4(a, r);
#pragma unroll
                    for (int c = 0; c < 4; ++c) o[c][g] = r[c];
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int row = 16 * sx + 4 * w + c;
                    *reinterpret_cast<uint4*>(out + row * 128 + ((p ^ (row & 7)) << 4)) =
                        make_uint4(o[c][0], o[c][1], o[c][2], o[c][3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);               // every lane's loads of the stage are consumed
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const int64_t t = blockIdx.x + i * gridDim.x;
            const int64_t nb = t / nkb, kb = t - nb * nkb;
            tma_store_2d(&tmOut, out, int32_t(nb * 128), int32_t(kb * 128));
            bulk_commit_group();
        }
    }
    if (!ok && lane == 0) tr_record(FP8_ERR_TIMEOUT);
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
}

// [rows][cols] bytes as 128x128-byte boxes with the 128-byte swizzle.
inline bool make_tile_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(cols)};
    cuuint32_t box[2] = {128u, 128u};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2u, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fp8bs

using namespace fp8bs;

extern "C" int fp8_transpose_128x128(const uint8_t* q, const float* s, int64_t N, int64_t K, uint8_t* qT, float* sT,
                                     fp8_stream_t stream) {
    if (!q || !s || !qT || !sT || N <= 0 || K <= 0) return FP8_ERR_ARG;
    if (N % 128 || K % 128) return FP8_ERR_SHAPE;
    if (N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1) return FP8_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(qT) || ((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(sT)) & 3u))
        return FP8_ERR_ALIGN;
    const int sms = device_sms();
    if (sms <= 0) return FP8_ERR_DEVICE;
    CUtensorMap mi, mo;
    if (!make_tile_map(&mi, q, N, K) || !make_tile_map(&mo, qT, K, N)) return FP8_ERR_CUDA;
    static unsigned char opted[kMaxDevices];
    if (!opt_in_dynamic_smem(transpose_128x128_kernel, kTrSmem, opted)) return FP8_ERR_CUDA;
    const int64_t tiles = (N / 128) * (K / 128);
    const int grid = int(tiles < sms ? tiles : sms);
    transpose_128x128_kernel<<<grid, kTrThreads, kTrSmem, reinterpret_cast<cudaStream_t>(stream)>>>(
        mi, mo, s, sT, N / 128, K / 128);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" int fp8bs_transpose_take_status(cudaStream_t stream) {
    int v = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP8_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_tr_status, sizeof v) != cudaSuccess) return FP8_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_tr_status, &zero, sizeof zero) != cudaSuccess) return FP8_ERR_CUDA;
    return v;
}
