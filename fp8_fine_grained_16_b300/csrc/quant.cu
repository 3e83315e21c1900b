// quant.cu -- online max-abs E4M3 quantisers (the jp-study.kr page: the max-abs value is
// computed online for each 1x128 activation tile and each 128x128 weight
// block; the tmdrlife.com page: each quantiser reads the BF16 values once and writes FP8
// codes plus scales back in the same pass).
//
// All three kernels are HBM-bound streaming passes: 2 bytes read + 1 byte
// written per element (+4 bytes of scale per tile).  Loads are 16-byte
// vector loads through the read-only path, the tile amax is reduced with
// warp shuffles, and the codes leave as coalesced 8/16-byte stores.
#include "common.cuh"

namespace fp8bs {

// ------------------------------------------------------------------ cast
__global__ void __launch_bounds__(256) cast_e4m3_kernel(const float* __restrict__ x, int64_t n,
                                                        uint8_t* __restrict__ q) {
    const int64_t n8 = n >> 3;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(x) + 2 * i);
        const float4 b = __ldg(reinterpret_cast<const float4*>(x) + 2 * i + 1);
        uint2 o;
        o.x = cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(a.z, a.w) << 16);
        o.y = cvt_e4m3x2(b.x, b.y) | (cvt_e4m3x2(b.z, b.w) << 16);
        reinterpret_cast<uint2*>(q)[i] = o;
    }
    // tail (n % 8 elements), one thread each
    const int64_t t = (n8 << 3) + int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t < n) q[t] = uint8_t(cvt_e4m3x2(x[t], 0.0f) & 0xFFu);
}

// ------------------------------------------------------------------ 1x128
// One warp per row; a half-warp owns one tile (lane l of the half holds
// elements [8l, 8l+8) of it), so a warp step covers two adjacent K blocks and
// kU steps are unrolled to keep kU 16-byte loads per thread in flight.  All
// lanes run every shuffle; loads and stores past the row's last K block are
// skipped.  A CTA of 8 warps covers 8 consecutive rows, so the 8 scales of
// one K block leave as one 32-byte segment.
constexpr int kQ1Rows = 8;      // rows (warps) per CTA
constexpr int kQ1U = 4;         // warp steps (tile pairs) unrolled per iteration

template <bool POW2>
FP8_DEV void quant_act_1x128_rows(const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t* __restrict__ q, float* __restrict__ s, int64_t cta) {
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;
    const int l16 = lane & 15;
    const int64_t m = cta * kQ1Rows + (threadIdx.x >> 5);
    if (m >= M) return;                                   // warp-uniform
    const int nkb = int(K >> 7);
    const uint4* xr = reinterpret_cast<const uint4*>(x + m * ldx) + l16;   // + 16 * kb per tile
    uint2* qr = reinterpret_cast<uint2*>(q + m * K) + l16;                  // + 16 * kb per tile

    for (int kb0 = 0; kb0 < nkb; kb0 += 2 * kQ1U) {
        uint4 v[kQ1U];
#pragma unroll
        for (int u = 0; u < kQ1U; ++u) {
            const int kb = kb0 + 2 * u + half;
            v[u] = kb < nkb ? __ldg(xr + 16 * kb) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kQ1U; ++u) {
            const int kb = kb0 + 2 * u + half;
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            float f[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = bf16_lo(w[i]);
                f[2 * i + 1] = bf16_hi(w[i]);
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            float inv;
            const float sc = tile_scale(amax, POW2, inv);
            if (kb < nkb) {
                uint2 o;
                o.x = cvt_e4m3x2(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv)) |
                      (cvt_e4m3x2(__fmul_rn(f[2], inv), __fmul_rn(f[3], inv)) << 16);
                o.y = cvt_e4m3x2(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv)) |
                      (cvt_e4m3x2(__fmul_rn(f[6], inv), __fmul_rn(f[7], inv)) << 16);
                qr[16 * kb] = o;
                if (l16 == 0) s[int64_t(kb) * M + m] = sc;
            }
        }
    }
}

template <bool POW2>
__global__ void __launch_bounds__(256) quant_act_1x128_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                              int64_t ldx, uint8_t* __restrict__ q,
                                                              float* __restrict__ s) {
    pdl_launch_dependents();
    quant_act_1x128_rows<POW2>(x, M, K, ldx, q, s, blockIdx.x);
}

// ------------------------------------------------------------------ 128x128
// One CTA (256 threads) per 128x128 block.  Thread t covers rows
// t/16 + 16*i (i < 8) and columns 8*(t%16) .. +7 of the block: each
// 16-thread group reads one 256-byte row segment per step.
template <bool POW2>
FP8_DEV void quant_weight_block(const uint16_t* __restrict__ w, int64_t N, int64_t K, int64_t ldw,
                                uint8_t* __restrict__ q, float* __restrict__ s, int64_t blk) {
    __shared__ float red[8];
    const int64_t nkb = K >> 7;
    const int64_t nb = blk / nkb, kb = blk - nb * nkb;
    const int t = threadIdx.x;
    const int r0 = t >> 4, c = (t & 15) * 8;
    const uint16_t* base = w + (nb * 128) * ldw + kb * 128 + c;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(base + (r0 + 16 * i) * ldw));
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t ww[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(ww[j])), fabsf(bf16_hi(ww[j]))));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((t & 31) == 0) red[t >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    float inv;
    const float sc = tile_scale(amax, POW2, inv);
    if (t == 0) s[nb * nkb + kb] = sc;

    uint8_t* qb = q + (nb * 128) * K + kb * 128 + c;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t ww[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint2 o;
        o.x = cvt_e4m3x2(__fmul_rn(bf16_lo(ww[0]), inv), __fmul_rn(bf16_hi(ww[0]), inv)) |
              (cvt_e4m3x2(__fmul_rn(bf16_lo(ww[1]), inv), __fmul_rn(bf16_hi(ww[1]), inv)) << 16);
        o.y = cvt_e4m3x2(__fmul_rn(bf16_lo(ww[2]), inv), __fmul_rn(bf16_hi(ww[2]), inv)) |
              (cvt_e4m3x2(__fmul_rn(bf16_lo(ww[3]), inv), __fmul_rn(bf16_hi(ww[3]), inv)) << 16);
        *reinterpret_cast<uint2*>(qb + (r0 + 16 * i) * K) = o;
    }
}

template <bool POW2>
__global__ void __launch_bounds__(256) quant_weight_128x128_kernel(const uint16_t* __restrict__ w, int64_t N,
                                                                   int64_t K, int64_t ldw, uint8_t* __restrict__ q,
                                                                   float* __restrict__ s) {
    pdl_launch_dependents();
    quant_weight_block<POW2>(w, N, K, ldw, q, s, blockIdx.x);
}

// ------------------------------------------------------------------ X and W in one launch
// The two operands of a linear layer Y = X W^T: CTAs [0, nx) quantise 8 rows
// of X each (1x128 tiles), the rest one 128x128 block of W each.  The X CTAs,
// about 3.5 times the work of a W block at K = 7168, come first, so the last
// wave is made of the short ones.  Both passes read disjoint inputs and write
// disjoint outputs; one launch lets them share the GPU without a second
// stream, and the GEMM after it can start early (programmatic launch).
// Capped at 80 registers (three CTAs per SM, as the weight pass alone): the
// compiler's own choice for the joined kernel, 87, allows only two.
template <bool POW2>
__global__ void __launch_bounds__(256, 3) quant_act_weight_kernel(const uint16_t* __restrict__ x, int64_t M,
                                                               int64_t ldx, uint8_t* __restrict__ qx,
                                                               float* __restrict__ sx, int64_t nx,
                                                               const uint16_t* __restrict__ w, int64_t N,
                                                               int64_t ldw, uint8_t* __restrict__ qw,
                                                               float* __restrict__ sw, int64_t K) {
    pdl_launch_dependents();
    if (int64_t(blockIdx.x) < nx)
        quant_act_1x128_rows<POW2>(x, M, K, ldx, qx, sx, blockIdx.x);
    else
        quant_weight_block<POW2>(w, N, K, ldw, qw, sw, int64_t(blockIdx.x) - nx);
}

// ------------------------------------------------------------------ 128x1, transposed
// One CTA (256 threads) per 128-token x 64-column tile.  Thread t reads the
// 4 consecutive rows 4*(t/8) .. +3 at columns 8*(t%8) .. +7 (8 threads per
// 128-byte row segment).  Column amax: thread-local over its 4 rows, then a
// shuffle over the 4 lanes of the warp sharing t%8, then across the 8 warps
// through shared memory.  The codes of 4 consecutive tokens of one column
// form one 32-bit word, so they go into the transposed shared tile with one
// store; the tile then leaves as 128-byte rows of qT.
constexpr int kT1Cols = 64;
constexpr int kT1Stride = 33;   // words per transposed row (128 B + 4 B pad)

template <bool POW2>
__global__ void __launch_bounds__(256) quant_act_128x1_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t H,
                                                              int64_t ldx, uint8_t* __restrict__ qT,
                                                              float* __restrict__ s) {
    __shared__ float red[8][kT1Cols];
    __shared__ float inv_s[kT1Cols];
    __shared__ uint32_t tile[kT1Cols * kT1Stride];

    const int64_t nhb = (H + kT1Cols - 1) / kT1Cols;
    const int64_t tb = blockIdx.x / nhb, hb = blockIdx.x - tb * nhb;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int rg = t >> 3;              // row group: rows 4rg .. 4rg+3
    const int c8 = (t & 7) * 8;         // first of 8 columns
    const int64_t h0 = hb * kT1Cols;
    const bool col_ok = h0 + c8 < H;    // H % 8 == 0: a group of 8 is all in or all out

    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[j] = make_uint4(0, 0, 0, 0);
        if (col_ok) v[j] = __ldg(reinterpret_cast<const uint4*>(x + (tb * 128 + 4 * rg + j) * ldx + h0 + c8));
    }
    float f[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[j][2 * i] = bf16_lo(w[i]);
            f[j][2 * i + 1] = bf16_hi(w[i]);
        }
    }
    float cmax[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float a = fmaxf(fmaxf(fabsf(f[0][i]), fabsf(f[1][i])), fmaxf(fabsf(f[2][i]), fabsf(f[3][i])));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 8));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 16));
        cmax[i] = a;
    }
    if (lane < 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) red[wid][c8 + i] = cmax[i];
    }
    __syncthreads();
    if (t < kT1Cols) {
        float a = red[0][t];
#pragma unroll
        for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w][t]);
        float inv;
        const float sc = tile_scale(a, POW2, inv);
        inv_s[t] = inv;
        if (h0 + t < H) s[tb * H + h0 + t] = sc;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float inv = inv_s[c8 + i];
        const uint32_t word = cvt_e4m3x2(__fmul_rn(f[0][i], inv), __fmul_rn(f[1][i], inv)) |
                              (cvt_e4m3x2(__fmul_rn(f[2][i], inv), __fmul_rn(f[3][i], inv)) << 16);
        tile[(c8 + i) * kT1Stride + rg] = word;
    }
    __syncthreads();
    // 64 rows of 128 bytes: 8 threads per row, 16 bytes each, two passes
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int row = pass * 32 + (t >> 3);
        const int w0 = (t & 7) * 4;
        if (h0 + row < H) {
            const uint32_t* src = tile + row * kT1Stride + w0;
            const uint4 o = make_uint4(src[0], src[1], src[2], src[3]);
            *reinterpret_cast<uint4*>(qT + (h0 + row) * T + tb * 128 + w0 * 4) = o;
        }
    }
}

static int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

static int launch_status() { return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA; }

}  // namespace fp8bs

using namespace fp8bs;

extern "C" int fp8_cast_e4m3(const float* x, int64_t n, uint8_t* q, fp8_stream_t stream) {
    if (n < 0 || (n > 0 && (!x || !q))) return FP8_ERR_ARG;
    if (n == 0) return FP8_OK;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(q) & 7u)) return FP8_ERR_ALIGN;
    const int64_t work = (n >> 3) + 8;
    const int64_t blocks = (work + 255) / 256;
    const int64_t cap = int64_t(num_sms()) * 8;
    const int grid = int(blocks < cap ? blocks : cap);
    cast_e4m3_kernel<<<grid, 256, 0, stream>>>(x, n, q);
    return launch_status();
}

extern "C" int fp8_quant_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, float* s,
                                   uint32_t flags, fp8_stream_t stream) {
    if (!x || !q || !s || M <= 0 || K <= 0 || ldx < K || (flags & ~FP8_SCALE_POW2)) return FP8_ERR_ARG;
    if (K % 128) return FP8_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || (ldx % 8) || (reinterpret_cast<uintptr_t>(s) & 3u)) return FP8_ERR_ALIGN;
    const int64_t blocks = (M + kQ1Rows - 1) / kQ1Rows;
    if (blocks > 0x7FFFFFFFll) return FP8_ERR_SHAPE;
    const unsigned grid = unsigned(blocks);
    if (flags & FP8_SCALE_POW2)
        quant_act_1x128_kernel<true><<<grid, 256, 0, stream>>>(x, M, K, ldx, q, s);
    else
        quant_act_1x128_kernel<false><<<grid, 256, 0, stream>>>(x, M, K, ldx, q, s);
    return launch_status();
}

extern "C" int fp8_quant_weight_128x128(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, float* s,
                                        uint32_t flags, fp8_stream_t stream) {
    if (!w || !q || !s || N <= 0 || K <= 0 || ldw < K || (flags & ~FP8_SCALE_POW2)) return FP8_ERR_ARG;
    if (N % 128 || K % 128) return FP8_ERR_SHAPE;
    if (!aligned16(w) || !aligned16(q) || (ldw % 8) || (reinterpret_cast<uintptr_t>(s) & 3u)) return FP8_ERR_ALIGN;
    const int64_t blocks = (N / 128) * (K / 128);
    if (blocks > 0x7FFFFFFFll) return FP8_ERR_SHAPE;
    if (flags & FP8_SCALE_POW2)
        quant_weight_128x128_kernel<true><<<unsigned(blocks), 256, 0, stream>>>(w, N, K, ldw, q, s);
    else
        quant_weight_128x128_kernel<false><<<unsigned(blocks), 256, 0, stream>>>(w, N, K, ldw, q, s);
    return launch_status();
}

extern "C" int fp8_quant_act_128x1(const uint16_t* x, int64_t T, int64_t H, int64_t ldx, uint8_t* qT, float* s,
                                   uint32_t flags, fp8_stream_t stream) {
    if (!x || !qT || !s || T <= 0 || H <= 0 || ldx < H || (flags & ~FP8_SCALE_POW2)) return FP8_ERR_ARG;
    if (T % 128 || H % 8) return FP8_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(qT) || (ldx % 8) || (reinterpret_cast<uintptr_t>(s) & 3u)) return FP8_ERR_ALIGN;
    const int64_t blocks = (T / 128) * ((H + kT1Cols - 1) / kT1Cols);
    if (blocks > 0x7FFFFFFFll) return FP8_ERR_SHAPE;
    if (flags & FP8_SCALE_POW2)
        quant_act_128x1_kernel<true><<<unsigned(blocks), 256, 0, stream>>>(x, T, H, ldx, qT, s);
    else
        quant_act_128x1_kernel<false><<<unsigned(blocks), 256, 0, stream>>>(x, T, H, ldx, qT, s);
    return launch_status();
}

extern "C" int fp8_quant_act_weight(const uint16_t* x, int64_t M, int64_t ldx, uint8_t* qx, float* sx,
                                    const uint16_t* w, int64_t N, int64_t ldw, uint8_t* qw, float* sw, int64_t K,
                                    uint32_t flags, fp8_stream_t stream) {
    if (!x || !qx || !sx || !w || !qw || !sw || M <= 0 || N <= 0 || K <= 0 || ldx < K || ldw < K ||
        (flags & ~FP8_SCALE_POW2))
        return FP8_ERR_ARG;
    if (K % 128 || N % 128) return FP8_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(qx) || !aligned16(w) || !aligned16(qw) || (ldx % 8) || (ldw % 8) ||
        (reinterpret_cast<uintptr_t>(sx) & 3u) || (reinterpret_cast<uintptr_t>(sw) & 3u))
        return FP8_ERR_ALIGN;
    const int64_t nx = (M + kQ1Rows - 1) / kQ1Rows;
    const int64_t blocks = nx + (N / 128) * (K / 128);
    if (blocks > 0x7FFFFFFFll) return FP8_ERR_SHAPE;
    if (flags & FP8_SCALE_POW2)
        quant_act_weight_kernel<true><<<unsigned(blocks), 256, 0, stream>>>(x, M, ldx, qx, sx, nx, w, N, ldw, qw, sw, K);
    else
        quant_act_weight_kernel<false><<<unsigned(blocks), 256, 0, stream>>>(x, M, ldx, qx, sx, nx, w, N, ldw, qw, sw, K);
    return launch_status();
}
