/*
 * fp8_oracle.c -- plain, slow CPU oracle for the fine-grained FP8 path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  Only the test suite, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * Sources: the five scraped web pages on DeepSeek-V3's FP8 training.  They
 * have no titles; each is cited by its host, then by the passage's subject:
 *   why-be.why-be.co.kr (wr_id 35533) page -- the format passage (E4M3 for
 *                                            every tensor)
 *   tmdrlife.com page (wr_id 13334)        -- accumulation / promotion
 *                                            passages, the power-of-2
 *                                            scaling passage
 *   gnrental.net page (wr_id 40936)        -- BF16 combine, promotion
 *                                            ("Figure 7 (b)")
 *   jp-study.kr page (document_srl 258368) -- online max-abs per 1x128 /
 *                                            128x128, quantise before MoE
 *                                            dispatch, 256 routed experts /
 *                                            top-8, 128-element accumulation
 *                                            interval, FP8 Wgrad
 *
 * Every routine is the plain definition written out; loops run in the
 * obvious order.  Floating point: fp32 where the method fixes fp32 (scales,
 * the x*inv product), fp64 everywhere else.  Build with -ffp-contract=off
 * and without fast-math so that every fp32 operation rounds once.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   R1 E4M3 is the OCP "E4M3FN" format: bias 7, no infinities, NaN = S.1111.111,
 *      largest finite 448.  Conversion rounds to nearest, ties to even, and
 *      saturates to +-448 (inf included).  A negative value that rounds to
 *      zero keeps its sign (code 0x80).
 *   R2 Tile scale: amax is floored at 2^-64 so an all-zero tile stays finite.
 *      Default mode: inv = 448/amax and s = amax/448, both fp32 divisions.
 *      Power-of-two mode: s = 2^e with e the smallest integer such that
 *      448 * 2^e >= amax; inv = 2^-e.
 *   R3 Codes are E4M3(fp32(x * inv)): one fp32 multiply, then the E4M3 cast.
 *   R4 Promotion interval = scale block = 128 elements of K.
 *   R5 Routing: top-k by logit value, ties to the lower expert index; the
 *      dispatch order is a stable sort of (token, slot) by expert; gates are
 *      a softmax over the k selected logits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <fenv.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* bf16 <-> float                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the top half of an fp32 word, so widening is exact. */
static float bf16_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a double to bf16 once, to nearest with ties to even.  bf16 has an
 * 8-bit significand, exponent range of fp32 (normal >= 2^-126, subnormal
 * quantum 2^-133).  Values past the bf16 range become +-inf. */
static uint16_t double_to_bf16(double d) {
    if (isnan(d)) return 0x7FC0;
    double a = fabs(d);
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
    int E = e - 1;                /* unbiased exponent */
    if (E < -126) E = -126;       /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, E - 7);
    double n = nearbyint(a / quantum);   /* exact division by a power of two */
    double v = n * quantum;
    if (v >= 0x1p128) return sign | 0x7F80;   /* rounded past the largest bf16 */
    float f = (float)v;           /* v has <= 8 significant bits: exact */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFF));
}

void orc_round_bf16(const double* d, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(d[i]);
}

void orc_bf16_to_float(const uint16_t* h, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_float(h[i]);
}

/* ------------------------------------------------------------------ */
/* O1  E4M3 codec (why-be.why-be.co.kr 35533 page: E4M3 -- 4 exponent   */
/*     bits, 3 mantissa bits -- for every tensor; bit layout per        */
/*     reading R1)                                                      */
/* ------------------------------------------------------------------ */

/* value = (-1)^s * 2^(e-7) * (1 + m/8) for e > 0, (-1)^s * 2^-6 * m/8 for e = 0 */
double orc_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 0x7;
    if (e == 0xF && m == 0x7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return s ? -mag : mag;
}

/* Round |x| to the E4M3 grid: the grid spacing in the binade [2^E, 2^(E+1))
 * is 2^(E-3); below 2^-6 the spacing stays 2^-9 (subnormals). */
uint8_t orc_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (isinf(a)) return sign | 0x7E;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);
    int E = e - 1;
    if (E < -6) E = -6;
    double quantum = ldexp(1.0, E - 3);
    double v = nearbyint(a / quantum) * quantum;   /* ties to even multiple */
    if (v > 448.0) v = 448.0;                       /* satfinite */
    if (v == 0.0) return sign;
    if (v < 0x1p-6) return sign | (uint8_t)(v * 512.0); /* subnormal: m * 2^-9 */
    frexp(v, &e);
    E = e - 1;
    int m = (int)((v / ldexp(1.0, E) - 1.0) * 8.0);
    return sign | (uint8_t)(((E + 7) << 3) | m);
}

void orc_e4m3_encode_array(const float* x, int64_t n, uint8_t* q) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) q[i] = orc_e4m3_encode(x[i]);
}

/* Encode the fp32 values whose bit patterns are start, start+1, ...  */
void orc_e4m3_encode_bits(uint64_t start, int64_t n, uint8_t* q) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = (uint32_t)(start + (uint64_t)i);
        float f;
        memcpy(&f, &u, sizeof f);
        q[i] = orc_e4m3_encode(f);
    }
}

/* ------------------------------------------------------------------ */
/* O2  Tile scale (jp-study.kr page: max-abs computed online per 1x128  */
/*     activation tile / 128x128 weight block; tmdrlife.com and         */
/*     gnrental.net pages: scales that are integral powers of 2 for     */
/*     some activations).  Readings R2, R3.                             */
/* ------------------------------------------------------------------ */

#define ORC_FLAG_POW2 1u
#define E4M3_MAX 448.0f

float orc_tile_scale(float amax, uint32_t flags, float* inv) {
    float a = amax < 0x1p-64f ? 0x1p-64f : amax;
    if (!(flags & ORC_FLAG_POW2)) {
        *inv = E4M3_MAX / a;
        return a / E4M3_MAX;
    }
    int e;
    float f = frexpf(a, &e);      /* a = f * 2^e, f in [0.5, 1) */
    float m = 2.0f * f;           /* a = m * 2^(e-1), m in [1, 2) */
    int E = e - 1;
    int k = (m <= 1.75f) ? E - 8 : E - 7;   /* smallest k: 448 * 2^k >= a */
    *inv = ldexpf(1.0f, -k);
    return ldexpf(1.0f, k);
}

static uint8_t quant_one(float x, float inv) {
    float p = x * inv;            /* one fp32 multiply, rounded once */
    return orc_e4m3_encode(p);
}

/* ------------------------------------------------------------------ */
/* O3  Quantisers                                                      */
/* ------------------------------------------------------------------ */

/* 1x128 activation tiles: x bf16 [M][ldx], q [M][K], s [K/128][M]. */
void orc_quant_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                         uint8_t* q, float* s, uint32_t flags) {
    int64_t nkb = K / 128;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < nkb; ++kb) {
            const uint16_t* t = x + m * ldx + kb * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float v = fabsf(bf16_to_float(t[i]));
                if (v > amax) amax = v;
            }
            float inv;
            s[kb * M + m] = orc_tile_scale(amax, flags, &inv);
            for (int i = 0; i < 128; ++i)
                q[m * K + kb * 128 + i] = quant_one(bf16_to_float(t[i]), inv);
        }
    }
}

/* 1x128 tiles of an fp32 matrix: x fp32 [M][K], q [M][K], s [K/128][M].
 * The same tile rule as above on fp32 values; it defines the quantisation of
 * a GEMM result in the producer's epilogue (tmdrlife.com page: quantising where the BF16
 * activation is formed instead of re-reading it from HBM). */
void orc_quant_act_1x128_f32(const float* x, int64_t M, int64_t K, uint8_t* q, float* s, uint32_t flags) {
    int64_t nkb = K / 128;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < nkb; ++kb) {
            const float* t = x + m * K + kb * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float v = fabsf(t[i]);
                if (v > amax) amax = v;
            }
            float inv;
            s[kb * M + m] = orc_tile_scale(amax, flags, &inv);
            for (int i = 0; i < 128; ++i) q[m * K + kb * 128 + i] = quant_one(t[i], inv);
        }
    }
}

/* ------------------------------------------------------------------ */
/* SwiGLU fused with 1x128 quantisation of its output (the MoE         */
/* down-projection input; tmdrlife.com page: that activation's scales  */
/* are integral powers of 2)                                            */
/* ------------------------------------------------------------------ */

/* e^x in fp32 by the published Cody-Waite method: x = n*ln2 + r with
 * n = rint(x*log2(e)), ln2 split into a high part exact in 17 bits and a low
 * part (so n*ln2_hi is exact and r keeps its low bits), e^r by its Taylor
 * polynomial of degree 7 on |r| <= ln2/2 (Horner form, fused multiply-adds),
 * then one multiply by 2^n.  x > 88 gives +inf and x < -87 gives 0 (the
 * callers only form 1 + e^x, where both are exact).  Every step is one IEEE
 * fp32 operation, so the result is a fixed function of x. */
float orc_exp_cw(float x) {
    if (x > 88.0f) return INFINITY;
    if (x < -87.0f) return 0.0f;
    const float n = rintf(x * 0x1.715476p+0f);            /* log2(e) */
    float r = fmaf(-n, 0x1.62e4p-1f, x);                    /* ln2, high part */
    r = fmaf(-n, 0x1.7f7d1cp-20f, r);                       /* ln2, low part */
    float p = 0x1.a01a02p-13f;                              /* 1/7! */
    p = fmaf(p, r, 0x1.6c16c2p-10f);                        /* 1/6! */
    p = fmaf(p, r, 0x1.111112p-7f);                         /* 1/5! */
    p = fmaf(p, r, 0x1.555556p-5f);                         /* 1/4! */
    p = fmaf(p, r, 0x1.555556p-3f);                         /* 1/3! */
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return p * ldexpf(1.0f, (int)n);                        /* 2^n is a normal number here */
}

/* h = SiLU(g) * u = (g * sigma(g)) * u with sigma(g) = 1 / (1 + e^-g), each
 * step one fp32 operation. */
static float swiglu_one(float g, float u) {
    const float e = orc_exp_cw(-g);
    const float d = 1.0f + e;
    const float sig = 1.0f / d;
    const float a = g * sig;
    return a * u;
}

/* y bf16 [R][ldy] holds gate = y[:, 0:I] and up = y[:, I:2I]; h fp32 [R][I]. */
void orc_swiglu_f32(const uint16_t* y, int64_t R, int64_t I, int64_t ldy, float* h) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t j = 0; j < I; ++j)
            h[r * I + j] = swiglu_one(bf16_to_float(y[r * ldy + j]), bf16_to_float(y[r * ldy + I + j]));
}

/* SwiGLU, then the 1x128 tile rule on the fp32 h: q [R][I], s [I/128][R]. */
void orc_swiglu_quant_1x128(const uint16_t* y, int64_t R, int64_t I, int64_t ldy, uint8_t* q, float* s,
                            uint32_t flags) {
    int64_t nkb = I / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t kb = 0; kb < nkb; ++kb) {
            float h[128];
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                const int64_t j = kb * 128 + i;
                h[i] = swiglu_one(bf16_to_float(y[r * ldy + j]), bf16_to_float(y[r * ldy + I + j]));
                float v = fabsf(h[i]);
                if (v > amax) amax = v;
            }
            float inv;
            s[kb * R + r] = orc_tile_scale(amax, flags, &inv);
            for (int i = 0; i < 128; ++i) q[r * I + kb * 128 + i] = quant_one(h[i], inv);
        }
    }
}

/* 128x1 activation tiles along tokens, output transposed:
 * x bf16 [T][ldx] (H used columns), qT [H][T], s [T/128][H]. */
void orc_quant_act_128x1(const uint16_t* x, int64_t T, int64_t H, int64_t ldx,
                         uint8_t* qT, float* s, uint32_t flags) {
    int64_t ntb = T / 128;
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < H; ++h) {
        for (int64_t tb = 0; tb < ntb; ++tb) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float v = fabsf(bf16_to_float(x[(tb * 128 + i) * ldx + h]));
                if (v > amax) amax = v;
            }
            float inv;
            s[tb * H + h] = orc_tile_scale(amax, flags, &inv);
            for (int i = 0; i < 128; ++i) {
                int64_t t = tb * 128 + i;
                qT[h * T + t] = quant_one(bf16_to_float(x[t * ldx + h]), inv);
            }
        }
    }
}

/* 128x128 weight blocks: w bf16 [N][ldw], q [N][K], s [N/128][K/128]. */
void orc_quant_weight_128x128(const uint16_t* w, int64_t N, int64_t K, int64_t ldw,
                              uint8_t* q, float* s, uint32_t flags) {
    int64_t nnb = N / 128, nkb = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t nb = 0; nb < nnb; ++nb) {
        for (int64_t kb = 0; kb < nkb; ++kb) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    float v = fabsf(bf16_to_float(w[(nb * 128 + i) * ldw + kb * 128 + j]));
                    if (v > amax) amax = v;
                }
            float inv;
            s[nb * nkb + kb] = orc_tile_scale(amax, flags, &inv);
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    int64_t n = nb * 128 + i, k = kb * 128 + j;
                    q[n * K + k] = quant_one(bf16_to_float(w[n * ldw + k]), inv);
                }
        }
    }
}

/* ------------------------------------------------------------------ */
/* O4  Block-scaled GEMM (tmdrlife.com and gnrental.net pages: each K  */
/*     interval is accumulated, then multiplied by its scaling factors  */
/*     and added into FP32; jp-study.kr page: the interval is 128       */
/*     elements).  D[m][n] = sum_k A^[m][k] * B^[n][k]                 */
/*     with A^ = decode(qA) * sA and B^ = decode(qB) * sB, both exact   */
/*     in fp64.  The sum runs over k ascending in fp64.                 */
/*     b_mode 0: sB [N/128][K/128] (128x128 blocks)                     */
/*     b_mode 1: sB [K/128][N]     (one scale per row and K block)      */
/* ------------------------------------------------------------------ */

static double b_scale(const float* sb, int b_mode, int64_t n, int64_t kb, int64_t N, int64_t nkb) {
    return b_mode == 0 ? (double)sb[(n / 128) * nkb + kb] : (double)sb[kb * N + n];
}

/* Evaluate D at rows[i] x cols[j] (i < nrows, j < ncols) into d[i*ncols+j]. */
void orc_gemm_blockscaled_at(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                             int b_mode, int64_t M, int64_t N, int64_t K,
                             const int64_t* rows, int64_t nrows,
                             const int64_t* cols, int64_t ncols, double* d) {
    int64_t nkb = K / 128;
    double* bh = (double*)malloc(sizeof(double) * (size_t)(ncols * K));
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < ncols; ++j)
        for (int64_t k = 0; k < K; ++k)
            bh[j * K + k] = orc_e4m3_decode(b[cols[j] * K + k]) *
                            b_scale(sb, b_mode, cols[j], k / 128, N, nkb);
#pragma omp parallel
    {
        double* ah = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t m = rows[i];
            for (int64_t k = 0; k < K; ++k)
                ah[k] = orc_e4m3_decode(a[m * K + k]) * (double)sa[(k / 128) * M + m];
            for (int64_t j = 0; j < ncols; ++j) {
                const double* bj = bh + j * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += ah[k] * bj[k];
                d[i * ncols + j] = acc;
            }
        }
        free(ah);
    }
    free(bh);
}

void orc_gemm_blockscaled(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                          int b_mode, int64_t M, int64_t N, int64_t K, double* d) {
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)M);
    int64_t* cols = (int64_t*)malloc(sizeof(int64_t) * (size_t)N);
    for (int64_t i = 0; i < M; ++i) rows[i] = i;
    for (int64_t j = 0; j < N; ++j) cols[j] = j;
    orc_gemm_blockscaled_at(a, sa, b, sb, b_mode, M, N, K, rows, M, cols, N, d);
    free(rows);
    free(cols);
}

/* ------------------------------------------------------------------ */
/* O5  MoE routing and grouped GEMM (jp-study.kr page: 256 routed       */
/*     experts, 8 active per token; activations quantised before        */
/*     dispatch).  Reading R5.                                          */
/* ------------------------------------------------------------------ */

/* logits fp32 [T][E] -> idx int32 [T][k], gate fp32 [T][k],
 * off int32 [E+1], src_row int32 [T*k], pos int32 [T][k]. */
void orc_route_topk(const float* logits, int64_t T, int E, int k,
                    int32_t* idx, float* gate, int32_t* off,
                    int32_t* src_row, int32_t* pos) {
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                int taken = 0;
                for (int p = 0; p < j; ++p) taken |= (idx[t * k + p] == e);
                if (taken) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* strict: ties keep lower e */
            }
            idx[t * k + j] = best;
        }
        double mx = l[idx[t * k]];
        double z = 0.0;
        for (int j = 0; j < k; ++j) z += exp((double)l[idx[t * k + j]] - mx);
        for (int j = 0; j < k; ++j)
            gate[t * k + j] = (float)(exp((double)l[idx[t * k + j]] - mx) / z);
    }
    int32_t* count = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int64_t i = 0; i < T * k; ++i) count[idx[i]]++;
    off[0] = 0;
    for (int e = 0; e < E; ++e) off[e + 1] = off[e] + count[e];
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = idx[t * k + j];
            int32_t p = off[e] + fill[e]++;
            src_row[p] = (int32_t)t;
            pos[t * k + j] = p;
        }
    free(count);
    free(fill);
}

/* Dispatch on one GPU: out row p takes input row src_row[p] (codes and
 * every K-block scale).  q [rows][K], s [K/128][rows] ->
 * q_out [out_rows][K], s_out [K/128][out_rows]. */
void orc_permute_rows(const uint8_t* q, const float* s, int64_t rows, int64_t K,
                      const int32_t* src_row, int64_t out_rows,
                      uint8_t* q_out, float* s_out) {
    int64_t nkb = K / 128;
    for (int64_t p = 0; p < out_rows; ++p) {
        int64_t r = src_row[p];
        memcpy(q_out + p * K, q + r * K, (size_t)K);
        for (int64_t kb = 0; kb < nkb; ++kb) s_out[kb * out_rows + p] = s[kb * rows + r];
    }
}

/* Grouped GEMM: expert e owns rows [off[e], off[e+1]) of A and D and uses
 * B_e = b + e*N*K with scales sb + e*(N/128)*(K/128).  Evaluated only on
 * the listed rows and columns; d[i*ncols+j]. */
void orc_grouped_gemm_at(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                         const int32_t* off, int E, int64_t total_rows, int64_t N, int64_t K,
                         const int64_t* rows, int64_t nrows, const int64_t* cols, int64_t ncols,
                         double* d) {
    int64_t nkb = K / 128, nnb = N / 128;
#pragma omp parallel
    {
        double* ah = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t m = rows[i];
            int e = 0;
            while (e < E && !(off[e] <= m && m < off[e + 1])) ++e;
            const uint8_t* be = b + (int64_t)e * N * K;
            const float* sbe = sb + (int64_t)e * nnb * nkb;
            for (int64_t k = 0; k < K; ++k)
                ah[k] = orc_e4m3_decode(a[m * K + k]) * (double)sa[(k / 128) * total_rows + m];
            for (int64_t j = 0; j < ncols; ++j) {
                int64_t n = cols[j];
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += ah[k] * (orc_e4m3_decode(be[n * K + k]) *
                                    (double)sbe[(n / 128) * nkb + k / 128]);
                d[i * ncols + j] = acc;
            }
        }
        free(ah);
    }
}

/* ------------------------------------------------------------------ */
/* O6  Combine, kept in BF16 (gnrental.net page: forward and backward   */
/*     combine stay in BF16): out[t][n] = sum_j gate[t][j] *           */
/*     y[pos[t][j]][n], summed in slot order in fp64, rounded to bf16   */
/*     once.                                                            */
/* ------------------------------------------------------------------ */

void orc_moe_combine(const uint16_t* y, const int32_t* pos, const float* gate,
                     int64_t T, int k, int64_t N, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += (double)gate[t * k + j] * (double)bf16_to_float(y[(int64_t)pos[t * k + j] * N + n]);
            out[t * N + n] = double_to_bf16(acc);
        }
}

/* ------------------------------------------------------------------ */
/* threads                                                            */
/* ------------------------------------------------------------------ */

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_rounding_is_nearest(void) { return fegetround() == FE_TONEAREST; }
