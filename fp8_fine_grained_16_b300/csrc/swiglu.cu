// swiglu.cu -- SwiGLU fused with 1x128 quantisation of its output, the input
// of the MoE down-projection (page 2: the scaling factors of this activation
// are integral powers of 2; page 4: quantisation is per 1x128 tile).
//
//   h[r][j] = SiLU(g) * u,  g = y[r][j], u = y[r][I + j],  SiLU(g) = g / (1 + e^-g)
//
// then the 1x128 tile rule on the fp32 h: amax, scale (power of two or
// amax/448 by flag), codes E4M3(fp32(h * inv)).  h never goes to HBM.
//
// Every step of h is one IEEE fp32 operation, e^x included: it is computed by
// the published Cody-Waite method (x = n*ln2 + r with ln2 split into a part
// exact in 17 bits and a remainder, e^r by its degree-7 Taylor polynomial in
// Horner form with fused multiply-adds, one multiply by 2^n), not by the
// library expf, so h is a fixed function of (g, u) and the codes can be
// checked bit for bit.  That e^x is within 1 ulp of the exact value.
//
// One warp per row; each half-warp quantises one 128-column tile (16 lanes x
// 8 values, 16-byte loads of gate and up), its amax reduced with shuffles.
#include "common.cuh"

namespace fp8bs {

// e^x for the fp32 SwiGLU above.  x > 88 gives +inf and x < -87 gives 0:
// only 1 + e^x is formed, where both are exact.
FP8_DEV float exp_cody_waite(float x) {
    if (x > 88.0f) return __int_as_float(0x7F800000);
    if (x < -87.0f) return 0.0f;
    const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));     // x * log2(e), to the nearest integer
    float r = __fmaf_rn(-n, 0x1.62e4p-1f, x);                 // ln2, high part (n * it is exact)
    r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);                    // ln2, low part
    float p = 0x1.a01a02p-13f;                                // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);                     // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);                      // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);                      // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);                      // 1/3!
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __int_as_float((int(n) + 127) << 23));   // 2^n, n in [-126, 127]
}

// (g * sigma(g)) * u with sigma(g) = 1 / (1 + e^-g); the reciprocal is the
// correctly rounded one, equal to the IEEE quotient 1 / (1 + e^-g).
FP8_DEV float swiglu_fp32(float g, float u) {
    const float sig = __frcp_rn(__fadd_rn(1.0f, exp_cody_waite(-g)));
    return __fmul_rn(__fmul_rn(g, sig), u);
}

constexpr int kSgRows = 8;          // rows (warps) per CTA

template <bool POW2>
__global__ void __launch_bounds__(256) swiglu_quant_1x128_kernel(const uint16_t* __restrict__ y, int64_t R, int64_t I,
                                                                  int64_t ldy, uint8_t* __restrict__ q,
                                                                  float* __restrict__ s) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * kSgRows + warp;
    if (row >= R) return;                                     // whole warp leaves together
    const int half = lane >> 4, l16 = lane & 15;
    const int ntiles = int(I >> 7);
    const uint16_t* yr = y + row * ldy;
    for (int t0 = 0; t0 < ntiles; t0 += 2) {
        const int tile = t0 + half;
        const bool live = tile < ntiles;                     // an odd last tile leaves half-warp 1 idle
        const int64_t col = int64_t(tile) * 128 + l16 * 8;
        float h[8];
        float amax = 0.0f;
        if (live) {
            const uint4 gv = __ldg(reinterpret_cast<const uint4*>(yr + col));
            const uint4 uv = __ldg(reinterpret_cast<const uint4*>(yr + I + col));
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                h[2 * j] = swiglu_fp32(bf16_lo(gw[j]), bf16_lo(uw[j]));
                h[2 * j + 1] = swiglu_fp32(bf16_hi(gw[j]), bf16_hi(uw[j]));
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(h[i]));
        }
        // amax of the tile: xor offsets below 16 stay inside the half-warp
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        if (live) {
            float inv;
            const float sc = tile_scale(amax, POW2, inv);
            uint2 o;
            o.x = cvt_e4m3x2(__fmul_rn(h[0], inv), __fmul_rn(h[1], inv)) |
                  (cvt_e4m3x2(__fmul_rn(h[2], inv), __fmul_rn(h[3], inv)) << 16);
            o.y = cvt_e4m3x2(__fmul_rn(h[4], inv), __fmul_rn(h[5], inv)) |
                  (cvt_e4m3x2(__fmul_rn(h[6], inv), __fmul_rn(h[7], inv)) << 16);
            *reinterpret_cast<uint2*>(q + row * I + col) = o;
            if (l16 == 0) s[int64_t(tile) * R + row] = sc;
        }
    }
}

}  // namespace fp8bs

using namespace fp8bs;

extern "C" int fp8_swiglu_quant_1x128(const uint16_t* y, int64_t R, int64_t I, int64_t ldy, uint8_t* q, float* s,
                                      uint32_t flags, fp8_stream_t stream) {
    if (!y || !q || !s || R <= 0 || I <= 0 || ldy < 2 * I || (flags & ~FP8_SCALE_POW2)) return FP8_ERR_ARG;
    if (I % 128) return FP8_ERR_SHAPE;
    if (!aligned16(y) || !aligned16(q) || (ldy % 8) || (reinterpret_cast<uintptr_t>(s) & 3u)) return FP8_ERR_ALIGN;
    const int64_t blocks = (R + kSgRows - 1) / kSgRows;
    if (blocks > 0x7FFFFFFFll) return FP8_ERR_SHAPE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (flags & FP8_SCALE_POW2)
        swiglu_quant_1x128_kernel<true><<<unsigned(blocks), 256, 0, st>>>(y, R, I, ldy, q, s);
    else
        swiglu_quant_1x128_kernel<false><<<unsigned(blocks), 256, 0, st>>>(y, R, I, ldy, q, s);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}
