// swiglu.cu -- SwiGLU fused with 1x128 quantisation of its output, the input
// of the MoE down-projection (the tmdrlife.com page: the scaling factors of this activation
// are integral powers of 2; the jp-study.kr page: quantisation is per 1x128 tile).
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
// checked bit for bit.  That e^x is within 1 ulp of the exact value.  The
// reciprocal in sigma is the correctly rounded one, formed by Markstein's
// correction of the hardware approximation (below).
//
// One warp per row; each half-warp quantises 128-column tiles (16 lanes x 8
// values, 16-byte loads of gate and up; two tiles' loads in flight), the
// amax reduced with shuffles.  Pairs of elements go through two-lane packed
// fp32 operations, lane by lane the same IEEE operations.  A lane whose 8
// gates all satisfy |g| <= 87 skips the range handling (the clamps, the +inf
// select and the reciprocal's fallback test), which cannot change any value
// there; the rest take the full steps.
#include "common.cuh"

namespace fp8bs {

// The reduction and polynomial steps of e^x for two values already in
// [-87, 88]: returns 2^n * P(r), with n = rint(x * log2 e), r = x - n*ln2 (ln2
// in two parts) and P the degree-7 Taylor polynomial of e^r in Horner form.
FP8_DEV float2 exp_steps(float2 xc) {
    const float2 t = __fmul2_rn(xc, make_float2(0x1.715476p+0f, 0x1.715476p+0f));   // x * log2(e)
    // t to the nearest integer (ties to even, as rint): adding 1.5 * 2^23 leaves
    // the rounded integer in the low mantissa bits of the sum (|t| < 128), and
    // subtracting it again gives n exactly -- full-rate adds instead of
    // float -> integer conversions.
    const float2 big = __fadd2_rn(t, make_float2(0x1.8p23f, 0x1.8p23f));
    const float2 n = __fadd2_rn(big, make_float2(-0x1.8p23f, -0x1.8p23f));
    // r = x - n*ln2 in two steps; n * (-c) is exactly -(n * c), so each fused
    // step rounds the same value as with -n
    float2 r = __ffma2_rn(n, make_float2(-0x1.62e4p-1f, -0x1.62e4p-1f), xc);      // ln2, high part (exact product)
    r = __ffma2_rn(n, make_float2(-0x1.7f7d1cp-20f, -0x1.7f7d1cp-20f), r);        // ln2, low part
    float2 p = make_float2(0x1.a01a02p-13f, 0x1.a01a02p-13f);                      // 1/7!
    p = __ffma2_rn(p, r, make_float2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));            // 1/6!
    p = __ffma2_rn(p, r, make_float2(0x1.111112p-7f, 0x1.111112p-7f));              // 1/5!
    p = __ffma2_rn(p, r, make_float2(0x1.555556p-5f, 0x1.555556p-5f));              // 1/4!
    p = __ffma2_rn(p, r, make_float2(0x1.555556p-3f, 0x1.555556p-3f));              // 1/3!
    p = __ffma2_rn(p, r, make_float2(0.5f, 0.5f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    // 2^n, n in [-126, 127]: the sum's bits are 0x4B400000 + n, so its bits
    // shifted up by 23 (0x4B400000 << 23 vanishes mod 2^32) plus 127 << 23
    // are those of 2^n
    return __fmul2_rn(p, make_float2(__int_as_float((__float_as_int(big.x) << 23) + (127 << 23)),
                                     __int_as_float((__float_as_int(big.y) << 23) + (127 << 23))));
}

// d = 1 + e^x of two values, for sigma = 1/d in the fp32 SwiGLU above, with
// two-lane packed fp32 operations (each lane is the same IEEE operation as
// its scalar form).  The definition takes e^x = +inf above 88 and 0 below
// -87.  Inputs in [-87, 88] take the steps unchanged.  An input below -87 is
// computed at -87: e^-87 ~ 1.6e-38 is far below half an ulp of 1, so 1 + e
// rounds to exactly 1, the d that e = 0 gives, and no select is needed for
// it.  An input above 88 is computed at 88 and its e replaced by +inf.
FP8_DEV float2 one_plus_exp(float2 x) {
    const float2 xc = make_float2(fminf(fmaxf(x.x, -87.0f), 88.0f), fminf(fmaxf(x.y, -87.0f), 88.0f));
    const float2 e = exp_steps(xc);
    const float inf = __int_as_float(0x7F800000);
    return __fadd2_rn(make_float2(1.0f, 1.0f), make_float2(x.x > 88.0f ? inf : e.x, x.y > 88.0f ? inf : e.y));
}

// 1/d correctly rounded for two values d in [1, 2^126) (the IEEE quotient),
// by Markstein's method (P. Markstein, "Computation of elementary functions
// on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990):
// from an approximation y within one ulp of 1/d, the residual r = 1 - d*y is
// exact in one fused multiply-add and y + r*y, rounded once, is the correctly
// rounded 1/d.  The approximation is the hardware's rcp.approx.ftz.f32 (at
// most one ulp off).
FP8_DEV float2 rcp_rn_markstein(float2 d) {
    float2 y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y.x) : "f"(d.x));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y.y) : "f"(d.y));
    const float2 r = __ffma2_rn(make_float2(-d.x, -d.y), y, make_float2(1.0f, 1.0f));
    return __ffma2_rn(r, y, y);
}

// 1/d correctly rounded for two values d >= 1: Markstein's method where the
// reciprocal is normal; d >= 2^126 (results below the normal range), +inf and
// NaN take __frcp_rn, which every other d matches bit for bit (checked for all
// d >= 1 by fp8_selftest_reciprocal).
FP8_DEV float2 rcp_rn_from_one(float2 d) {
    if (!(d.x < 0x1p126f && d.y < 0x1p126f)) return make_float2(__frcp_rn(d.x), __frcp_rn(d.y));
    return rcp_rn_markstein(d);
}

// (g * sigma(g)) * u for two elements, sigma(g) = 1 / (1 + e^-g); the
// reciprocal is the correctly rounded one, equal to the IEEE quotient.
FP8_DEV float2 swiglu2_fp32(float2 g, float2 u) {
    const float2 d = one_plus_exp(make_float2(-g.x, -g.y));
    const float2 sig = rcp_rn_from_one(d);
    return __fmul2_rn(__fmul2_rn(g, sig), u);
}

// The same h for two gates with |g| <= 87, without the range handling, which
// cannot change anything there: x = -g lies in [-87, 87], so the clamps leave
// it as it is and the +inf select does not fire, and d <= 1 + e^87 < 2^126,
// so Markstein's reciprocal needs no fallback.
FP8_DEV float2 swiglu2_fp32_in_range(float2 g, float2 u) {
    const float2 d = __fadd2_rn(make_float2(1.0f, 1.0f), exp_steps(make_float2(-g.x, -g.y)));
    const float2 sig = rcp_rn_markstein(d);
    return __fmul2_rn(__fmul2_rn(g, sig), u);
}

// Every float d with bits in [lo, hi] (d >= 1): rcp_rn_from_one(d) against
// __frcp_rn(d), bit for bit; the count of differences is added to *bad.
__global__ void __launch_bounds__(256) reciprocal_selftest_kernel(uint32_t lo, uint32_t hi,
                                                                  unsigned long long* bad) {
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x * 2;
    unsigned long long n = 0;
    for (uint64_t b = uint64_t(lo) + (uint64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 2; b <= hi; b += stride) {
        const bool two = b + 1 <= hi;
        const float2 d = make_float2(__uint_as_float(uint32_t(b)), __uint_as_float(uint32_t(two ? b + 1 : b)));
        const float2 r = rcp_rn_from_one(d);
        n += __float_as_uint(r.x) != __float_as_uint(__frcp_rn(d.x));
        if (two) n += __float_as_uint(r.y) != __float_as_uint(__frcp_rn(d.y));
    }
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, o);
    if ((threadIdx.x & 31) == 0 && n) atomicAdd(bad, n);
}

constexpr int kSgRows = 8;          // rows (warps) per CTA
constexpr int kSgTiles = 2;         // tiles per half-warp per iteration (loads in flight)

// At most 48 registers, so five CTAs (40 warps) share an SM: the kernel is
// bound by issue and load latency, and more resident warps hide more of both
// (four CTAs at the compiler's own 51 registers ran 6% slower).
template <bool POW2>
__global__ void __launch_bounds__(256, 5) swiglu_quant_1x128_kernel(const uint16_t* __restrict__ y, int64_t R, int64_t I,
                                                                  int64_t ldy, uint8_t* __restrict__ q,
                                                                  float* __restrict__ s) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * kSgRows + warp;
    if (row >= R) return;                                     // whole warp leaves together
    const int half = lane >> 4, l16 = lane & 15;
    const int ntiles = int(I >> 7);
    const uint16_t* yr = y + row * ldy;
    for (int t0 = 0; t0 < ntiles; t0 += 2 * kSgTiles) {
        // half-warp `half` takes tiles t0 + half + 2u, u < kSgTiles
        uint4 gv[kSgTiles], uv[kSgTiles];
#pragma unroll
        for (int u = 0; u < kSgTiles; ++u) {
            const int tile = t0 + half + 2 * u;
            if (tile < ntiles) {
                const int64_t col = int64_t(tile) * 128 + l16 * 8;
                gv[u] = __ldg(reinterpret_cast<const uint4*>(yr + col));
                uv[u] = __ldg(reinterpret_cast<const uint4*>(yr + I + col));
            }
        }
#pragma unroll
        for (int u = 0; u < kSgTiles; ++u) {
            const int tile = t0 + half + 2 * u;
            const bool live = tile < ntiles;                 // the last tiles may leave a half-warp idle
            float2 h[4];
            float amax = 0.0f;
            if (live) {
                const uint32_t gw[4] = {gv[u].x, gv[u].y, gv[u].z, gv[u].w};
                const uint32_t uw[4] = {uv[u].x, uv[u].y, uv[u].z, uv[u].w};
                float2 g[4], uu[4];
                bool in_range = true;          // |g| <= 87 for all 8 gates (false for NaN)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    g[j] = make_float2(bf16_lo(gw[j]), bf16_hi(gw[j]));
                    uu[j] = make_float2(bf16_lo(uw[j]), bf16_hi(uw[j]));
                    in_range &= (fabsf(g[j].x) <= 87.0f) & (fabsf(g[j].y) <= 87.0f);
                }
                if (in_range) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) h[j] = swiglu2_fp32_in_range(g[j], uu[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) h[j] = swiglu2_fp32(g[j], uu[j]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(h[j].x), fabsf(h[j].y)));
            }
            // amax of the tile: xor offsets below 16 stay inside the half-warp
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            if (live) {
                float inv;
                const float sc = tile_scale(amax, POW2, inv);
                const float2 inv2 = make_float2(inv, inv);
                float2 c[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) c[j] = __fmul2_rn(h[j], inv2);
                uint2 o;
                o.x = cvt_e4m3x2(c[0].x, c[0].y) | (cvt_e4m3x2(c[1].x, c[1].y) << 16);
                o.y = cvt_e4m3x2(c[2].x, c[2].y) | (cvt_e4m3x2(c[3].x, c[3].y) << 16);
                *reinterpret_cast<uint2*>(q + row * I + int64_t(tile) * 128 + l16 * 8) = o;
                if (l16 == 0) s[int64_t(tile) * R + row] = sc;
            }
        }
    }
}

}  // namespace fp8bs

using namespace fp8bs;

extern "C" int fp8_selftest_reciprocal(uint32_t first_bits, uint32_t last_bits, unsigned long long* mismatches,
                                       fp8_stream_t stream) {
    if (!mismatches || first_bits < 0x3F800000u || last_bits < first_bits) return FP8_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(mismatches) & 7u) return FP8_ERR_ALIGN;
    const uint64_t n = uint64_t(last_bits) - first_bits + 1;
    const uint64_t blocks = (n / 2 + 255) / 256;
    const unsigned grid = unsigned(blocks < 148 * 16 ? (blocks ? blocks : 1) : 148 * 16);
    reciprocal_selftest_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(first_bits, last_bits,
                                                                                          mismatches);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

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
