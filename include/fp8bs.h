/*
 * fp8bs.h -- C ABI of libfp8bs.so: fine-grained FP8 (E4M3) quantisation and
 * block-scaled FP8 GEMMs on one B300 GPU (sm_103a).
 *
 * The method comes from five scraped web pages that restate DeepSeek-V3's FP8
 * training recipe.  They have no titles; each is cited by its host, with the
 * passage it gives:
 *   why-be.why-be.co.kr (wr_id 35533) page   E4M3 for every tensor
 *   tmdrlife.com page (wr_id 13334)          limited-width accumulation,
 *           promotion of partial sums into FP32, power-of-2 scales, the HBM
 *           round trip of quantised activations
 *   gnrental.net page (wr_id 40936)          promotion ("Figure 7 (b)"), BF16
 *           combine, microscaling
 *   jp-study.kr page (document_srl 258368)   online max-abs per 1x128
 *           activation tile / 128x128 weight block, quantise before MoE
 *           dispatch, 256 routed experts with 8 active, 128-element
 *           accumulation interval, FP8 Wgrad ("Figure 6")
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or keeps them.  bf16 data is passed as raw
 *     16-bit words (uint16_t), E4M3 data as bytes (uint8_t).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  No call synchronises the host, except
 *     fp8_get_status.  Stream order always holds: the block-scaled GEMMs
 *     (the fp8_gemm_blockscaled* and fp8_grouped_gemm_blockscaled* calls) are
 *     programmatic dependent launches that set up while the work before them
 *     drains, but touch memory only after it has completed.
 *   - The return value is FP8_OK (0) or a negative FP8_ERR_* code.  On an
 *     argument error (FP8_ERR_ARG, _SHAPE, _ALIGN) nothing is enqueued.
 *     FP8_ERR_CUDA means a launch failed (the CUDA error is left for
 *     cudaGetLastError to report).
 *   - Faults found by a kernel while it runs (a pipeline wait that timed out,
 *     expert offsets out of range) do not trap: the kernel records a code in a
 *     device status word and exits early.  fp8_get_status reads it.
 *   - All row-major matrices are dense with the stated leading dimension (in
 *     elements).  Pointers must be 16-byte aligned and leading dimensions a
 *     multiple of 16 bytes (FP8_ERR_ALIGN otherwise).
 *   - E4M3 here is E4M3FN: bias 7, no infinities, largest finite +-448.
 *     Conversion rounds to nearest-even and saturates to +-448.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fp8_stream_t;   /* same type as cudaStream_t */

#if defined(__GNUC__)
#define FP8_API __attribute__((visibility("default")))
#else
#define FP8_API
#endif

enum fp8_status {
    FP8_OK = 0,
    FP8_ERR_ARG = -1,        /* null pointer, non-positive size, bad enum */
    FP8_ERR_SHAPE = -2,      /* a dimension that must be a multiple of 128 is not */
    FP8_ERR_ALIGN = -3,      /* pointer or leading dimension not 16-byte aligned */
    FP8_ERR_CUDA = -4,       /* a CUDA call or launch failed */
    FP8_ERR_TIMEOUT = -5,    /* a kernel's bounded pipeline wait expired (device status) */
    FP8_ERR_OFFSETS = -6,    /* expert offsets not monotone or out of range (device status) */
    FP8_ERR_DEVICE = -7,     /* no usable sm_100-family device */
    FP8_ERR_SCRATCH = -8,    /* problem larger than the library's static scratch */
    FP8_ERR_SCALE = -9       /* a scale is not a positive normal power of two (device status) */
};

/* flags of the quantisers */
#define FP8_SCALE_POW2 1u     /* scales are exact powers of two (the tmdrlife.com and gnrental.net pages) */

/* b_scale_mode of fp8_gemm_blockscaled */
#define FP8_BSCALE_BLOCK128 0 /* sB [N/128][K/128]: one scale per 128x128 block */
#define FP8_BSCALE_ROW 1      /* sB [K/128][N]: one scale per B row and K block */

/* d_dtype of fp8_gemm_blockscaled */
#define FP8_OUT_BF16 0
#define FP8_OUT_F32 1

/* ------------------------------------------------------------------------
 * Element-wise E4M3 cast (the why-be.why-be.co.kr (wr_id 35533) page: E4M3
 * for every tensor).
 * q[i] = E4M3(x[i]) with round-to-nearest-even and saturation to +-448; the
 * same conversion every quantiser uses.  x: n fp32, q: n bytes.  n >= 0.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_cast_e4m3(const float* x, int64_t n, uint8_t* q, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * 1x128 activation quantiser (the jp-study.kr page: max-abs computed online for each
 * 1x128 activation tile; the tmdrlife.com page: one pass reads the BF16 values and writes
 * the FP8 codes back to HBM).
 * For each row m and K block kb, amax = max |x[m][128kb .. 128kb+127]|,
 * floored at 2^-64.  Default: s = amax/448 and inv = 448/amax (fp32
 * divisions, rounded to nearest).  FP8_SCALE_POW2: s = 2^e with e the
 * smallest integer such that 448*2^e >= amax, inv = 2^-e.  Codes are
 * E4M3(fp32(x * inv)).
 *   x  bf16 [M][ldx] (K columns used), ldx >= K, ldx % 8 == 0
 *   q  E4M3 [M][K] row-major
 *   s  fp32 [K/128][M] (M contiguous: the layout the GEMM reads)
 * M >= 1, K % 128 == 0.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_quant_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                uint8_t* q, float* s, uint32_t flags, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * 128x1 activation quantiser for Wgrad, output transposed (the jp-study.kr page: the
 * Wgrad operation runs in FP8).  Tiles run along tokens: for each column h
 * and token block tb, amax over x[128tb .. 128tb+127][h]; scale rule as
 * above.  The codes are written transposed so that tokens (the K dimension
 * of Wgrad) are contiguous.
 *   x   bf16 [T][ldx] (H columns used), ldx >= H, ldx % 8 == 0
 *   qT  E4M3 [H][T] row-major
 *   s   fp32 [T/128][H]
 * T % 128 == 0, H >= 1, H % 8 == 0.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_quant_act_128x1(const uint16_t* x, int64_t T, int64_t H, int64_t ldx,
                                uint8_t* qT, float* s, uint32_t flags, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * 128x128 weight quantiser (the jp-study.kr page: max-abs computed online for each
 * 128x128 weight block).  One scale per block; scale rule as above.
 *   w  bf16 [N][ldw] (K columns used), ldw >= K, ldw % 8 == 0
 *   q  E4M3 [N][K]
 *   s  fp32 [N/128][K/128]
 * N % 128 == 0, K % 128 == 0.  A stack of E expert matrices [E][N][K] is
 * quantised in one call as N' = E*N rows (blocks never straddle experts);
 * its scales are then [E][N/128][K/128].
 * ---------------------------------------------------------------------- */
FP8_API int fp8_quant_weight_128x128(const uint16_t* w, int64_t N, int64_t K, int64_t ldw,
                                     uint8_t* q, float* s, uint32_t flags, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * Both operands of a linear layer Y = X W^T quantised in one launch:
 * exactly fp8_quant_act_1x128(x, M, K, ldx, qx, sx, ...) and
 * fp8_quant_weight_128x128(w, N, K, ldw, qw, sw, ...) with the same flags
 * (the same codes and scales bit for bit), the two passes sharing the GPU
 * without a second stream.  Layouts and limits as those two calls:
 *   x  bf16 [M][ldx], qx E4M3 [M][K], sx fp32 [K/128][M]
 *   w  bf16 [N][ldw], qw E4M3 [N][K], sw fp32 [N/128][K/128]
 * M >= 1, N % 128 == 0, K % 128 == 0.  The block-scaled GEMMs are
 * programmatic dependent launches, so one queued right after this call sets
 * up while it finishes.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_quant_act_weight(const uint16_t* x, int64_t M, int64_t ldx, uint8_t* qx, float* sx,
                                 const uint16_t* w, int64_t N, int64_t ldw, uint8_t* qw, float* sw, int64_t K,
                                 uint32_t flags, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * SwiGLU fused with 1x128 quantisation of its output: the input of the MoE
 * down-projection (the tmdrlife.com page: that activation's scaling factors are integral
 * powers of 2, so flags = FP8_SCALE_POW2 is its natural setting; the jp-study.kr page:
 * 1x128 tiles).  For each row r and column j < I:
 *   h = (g * sigma(g)) * u,  g = y[r][j], u = y[r][I + j],
 *   sigma(g) = 1 / (1 + e^-g)
 * each step one fp32 operation, with e^x by Cody-Waite reduction and a
 * degree-7 Taylor polynomial (within 1 ulp), so h is a fixed function of the
 * inputs; then the 1x128 tile rule of fp8_quant_act_1x128 on the fp32 h.
 * h is never written to memory.
 *   y  bf16 [R][ldy]: gate in columns 0..I-1, up in I..2I-1; ldy >= 2I,
 *      ldy % 8 == 0
 *   q  E4M3 [R][I]
 *   s  fp32 [I/128][R]
 * I % 128 == 0.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_swiglu_quant_1x128(const uint16_t* y, int64_t R, int64_t I, int64_t ldy,
                                   uint8_t* q, float* s, uint32_t flags, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * Block-scaled FP8 GEMM (the tmdrlife.com and gnrental.net pages: partial sums are accumulated on the
 * tensor cores over a K interval, then multiplied by the scaling factors and
 * added into FP32; the jp-study.kr page: the interval is 128 elements).
 *   D[m][n] = sum_kb  sA[kb][m] * sB(n,kb) * P_kb[m][n],
 *   P_kb[m][n] = sum_{k in block kb} A[m][k] * B[n][k]   (E4M3 values)
 * P_kb is formed by tcgen05 MMAs into tensor memory; the outer sum runs in
 * FP32 registers.
 *   a   E4M3 [M][K] row-major (K contiguous)
 *   sa  fp32 [K/128][M]
 *   b   E4M3 [N][K] row-major (K contiguous)
 *   sb  b_scale_mode FP8_BSCALE_BLOCK128: fp32 [N/128][K/128]
 *       b_scale_mode FP8_BSCALE_ROW:      fp32 [K/128][N]
 *   d   [M][N] row-major, bf16 (FP8_OUT_BF16, rounded to nearest-even) or
 *       fp32 (FP8_OUT_F32)
 * M >= 1, N % 128 == 0, K % 128 == 0.  Wgrad (dW = dY^T X) is this call with
 * a = dY^T and b = X^T from fp8_quant_act_128x1, FP8_BSCALE_ROW, FP8_OUT_F32.
 * The kernel is a programmatic dependent launch: it may start while the work
 * before it on `stream` finishes, and touches global memory only after that
 * work has completed (the stream order is kept).
 * ---------------------------------------------------------------------- */
FP8_API int fp8_gemm_blockscaled(const uint8_t* a, const float* sa,
                                 const uint8_t* b, const float* sb, int b_scale_mode,
                                 void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                                 fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8_gemm_blockscaled with a workspace for splitting the last tiles along
 * K.  Tiles are 256 x 256 and each pair of SMs owns whole tiles; when the
 * tiles leave a last wave of at most half the SM pairs (or are fewer than
 * the pairs), those tiles are computed as K ranges, one per SM pair, each
 * range's promoted fp32 sum written to the workspace, and a second kernel
 * on the same stream adds a tile's ranges in K order and stores D.  D is the
 * same sum of promoted K blocks, grouped into per-range fp32 sums (the
 * order of the fp32 additions differs from fp8_gemm_blockscaled; the result
 * is deterministic).
 *   workspace        device memory, 16-byte aligned, owned by the caller,
 *                    not read before it is written; it must not be used by
 *                    another call until this call's work on `stream` ends.
 *                    NULL (with workspace_bytes 0): no split.
 *   workspace_bytes  its size; fp8_gemm_blockscaled_workspace_bytes gives
 *                    the most a call of that shape uses on the current
 *                    device (0 when it would never split).  A smaller
 *                    workspace disables the split where it does not fit.
 * Other arguments, layouts and errors as fp8_gemm_blockscaled;
 * FP8_ERR_ALIGN for a misaligned workspace, FP8_ERR_ARG for a negative size
 * or a size without a pointer.
 * ---------------------------------------------------------------------- */
FP8_API int64_t fp8_gemm_blockscaled_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* GEMM forms, for the tile and split-plan queries below. */
#define FP8_GEMM_FORM_DENSE   0   /* fp8_gemm_blockscaled(_ws): bf16 or fp32 D */
#define FP8_GEMM_FORM_Q8      1   /* fp8_gemm_blockscaled_q8(_ws): E4M3 D */
#define FP8_GEMM_FORM_GROUPED 2   /* fp8_grouped_gemm_blockscaled */

/* Columns of one output tile of a GEMM form (256 for every form: 256-row
 * tiles on an SM pair for the dense forms, 128-row tiles on one SM for the
 * grouped form).  FP8_ERR_ARG for an unknown form.  Host only. */
FP8_API int fp8_gemm_tile_cols(int form);

/* The tail-split plan of a dense GEMM form (FP8_GEMM_FORM_DENSE or _Q8) for
 * `pairs` SM pairs and a workspace of workspace_bytes (0: none): *split K
 * ranges per split tile (0: no split), *tail0 the first split tile (256-row
 * tiles of fp8_gemm_tile_cols(form) columns, numbered with the 256-row tile
 * index fastest), *launched_pairs the pairs the launch uses.  Host-only
 * arithmetic, no device access; the launch takes `pairs` from the device's
 * occupancy (148 SMs: 74).  FP8_ERR_ARG for another form, otherwise
 * FP8_ERR_ARG / _SHAPE as fp8_gemm_blockscaled. */
FP8_API int fp8_gemm_split_plan(int form, int64_t M, int64_t N, int64_t K, int pairs, int64_t workspace_bytes,
                                int64_t* split, int64_t* tail0, int64_t* launched_pairs);

/* The work units of launched pair `pair` under that plan, in the order the
 * pair runs them: units[4i .. 4i+3] = tile, first K block, end K block,
 * workspace slab (-1: whole tile, stored to D).  Writes at most max_units
 * units and returns how many the pair has (negative: an FP8_ERR_* code). */
FP8_API int64_t fp8_gemm_split_units(int form, int64_t M, int64_t N, int64_t K, int pairs,
                                     int64_t workspace_bytes, int64_t pair, int64_t* units, int64_t max_units);
FP8_API int fp8_gemm_blockscaled_ws(const uint8_t* a, const float* sa,
                                    const uint8_t* b, const float* sb, int b_scale_mode,
                                    void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                                    void* workspace, int64_t workspace_bytes, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * The dense FP8 linear layer called with HOST buffers: Y = X W^T computed as
 * this library's path (the jp-study.kr page: max-abs 1x128 activation tiles
 * and 128x128 weight blocks; the tmdrlife.com page: each 128-element K
 * interval promoted into FP32 with the two scales): fp8_quant_act_1x128 of
 * X, fp8_quant_weight_128x128 of W, fp8_gemm_blockscaled_ws to bf16.  The
 * exception to the device-pointer rule above: x_h, w_h and y_h are HOST
 * pointers.
 *   x_h  bf16 [M][K] row-major, host memory
 *   w_h  bf16 [N][K] row-major, host memory
 *   y_h  bf16 [M][N] row-major, host memory (written)
 *   flags  0 or FP8_SCALE_POW2 (the quantisers' scale rule)
 *   workspace  device memory of fp8_linear_host_workspace_bytes(M, N, K)
 *          bytes, 256-byte aligned, owned by the caller; it holds the device
 *          copies of X, W and Y, their codes and scales, and the GEMM's split
 *          workspace, and must not be used by another call until this call's
 *          work on `stream` ends.
 * The copies are cut into chunks of W's rows (Y's columns) and run on two
 * internal streams (created once per device), overlapped with the
 * quantisation and GEMM of earlier chunks on `stream`; `stream` waits for
 * all of it, so the call is ordered on `stream` like any other.  Host buffers
 * in page-locked memory let the copies run asynchronously; pageable ones work
 * but serialise.  x_h and w_h must not change, and y_h must not be read,
 * until `stream` reaches the end of the call.
 * M >= 1, N % 128 == 0, K % 128 == 0.  Errors as the calls it makes;
 * FP8_ERR_ARG also for a workspace smaller than required, FP8_ERR_ALIGN for
 * a misaligned one.
 * ---------------------------------------------------------------------- */
FP8_API int64_t fp8_linear_host_workspace_bytes(int64_t M, int64_t N, int64_t K);
FP8_API int fp8_linear_host(const uint16_t* x_h, const uint16_t* w_h, int64_t M, int64_t N, int64_t K,
                            uint16_t* y_h, uint32_t flags, void* workspace, int64_t workspace_bytes,
                            fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * The block-scaled GEMM with its result quantised in the epilogue (the tmdrlife.com page:
 * BF16 activations are read from HBM, quantised and written back, only to
 * be read again for the next MMA; quantising the producer's output where it
 * is formed removes that round trip).  D is computed exactly as by
 * fp8_gemm_blockscaled (fp32, promoted per 128-element K block) and, instead
 * of being stored, quantised per 1x128 tile along N (amax in fp32, scale by
 * flags, codes E4M3(fp32(D * inv))), i.e. the output of
 * fp8_quant_act_1x128 applied to the fp32 D, ready to be the A operand of
 * the next GEMM (whose K runs along this N).
 *   a, sa, b, sb, b_scale_mode, M, N, K   as fp8_gemm_blockscaled
 *   q_out  E4M3 [M][N], 16-byte aligned
 *   s_out  fp32 [N/128][M]
 *   flags  0 or FP8_SCALE_POW2
 * ---------------------------------------------------------------------- */
FP8_API int fp8_gemm_blockscaled_q8(const uint8_t* a, const float* sa,
                                    const uint8_t* b, const float* sb, int b_scale_mode,
                                    uint8_t* q_out, float* s_out, uint32_t flags,
                                    int64_t M, int64_t N, int64_t K, fp8_stream_t stream);

/* fp8_gemm_blockscaled_q8 with the tail-split workspace of
 * fp8_gemm_blockscaled_ws (same rules and sizes).  Split tiles are
 * quantised by the fix-up kernel from the fp32 sum of their K ranges, by the
 * same 1x128 rule. */
FP8_API int fp8_gemm_blockscaled_q8_ws(const uint8_t* a, const float* sa,
                                       const uint8_t* b, const float* sb, int b_scale_mode,
                                       uint8_t* q_out, float* s_out, uint32_t flags,
                                       int64_t M, int64_t N, int64_t K,
                                       void* workspace, int64_t workspace_bytes, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * The same GEMM for power-of-two scales (the quantisers' FP8_SCALE_POW2
 * mode; the tmdrlife.com page: integral-power-of-2 scaling factors), with the scales applied
 * by the tensor core (the gnrental.net page: fine-grained tiles match microscaling, which
 * Blackwell tensor cores support; the tmdrlife.com page: tensor cores that take the scaling
 * factors).  Each scale 2^e becomes a UE8M0 scale factor of the block-scaled
 * tcgen05 MMA, repeated over the four 32-element K groups of its 128-element
 * K block, and D accumulates in fp32 in tensor memory over the whole K:
 *   D[m][n] = sum_k (sA[k/128][m] * A[m][k]) * (sB(n, k/128) * B[n][k])
 * which is the block-promoted sum of fp8_gemm_blockscaled up to fp32
 * rounding order.  Arguments, layouts and limits are those of
 * fp8_gemm_blockscaled.  Every scale read (rows < M, columns < N) must be a
 * positive normal power of two; the kernel records FP8_ERR_SCALE in the
 * device status otherwise, and the result is then undefined.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_gemm_blockscaled_pow2(const uint8_t* a, const float* sa,
                                      const uint8_t* b, const float* sb, int b_scale_mode,
                                      void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                                      fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * The grouped (per-expert) GEMM for power-of-two scales, on the microscaled
 * MMA of fp8_gemm_blockscaled_pow2 (the jp-study.kr page: 256 routed experts, each
 * processing the rows dispatched to it; the tmdrlife.com and gnrental.net pages: power-of-two scales,
 * tensor cores that take the scaling factors).  Arguments, layouts, limits
 * and the handling of bad offsets are those of fp8_grouped_gemm_blockscaled;
 * every scale read must be a positive normal power of two (FP8_ERR_SCALE in
 * the device status otherwise).
 * ---------------------------------------------------------------------- */
FP8_API int fp8_grouped_gemm_blockscaled_pow2(const uint8_t* a, const float* sa,
                                              const uint8_t* b, const float* sb,
                                              const int32_t* expert_offsets, int E,
                                              int64_t total_rows, int64_t N, int64_t K,
                                              uint16_t* d, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * Transposed copy of a 128x128-block-quantised E4M3 matrix, for FP8 Dgrad
 * (the why-be.why-be.co.kr (wr_id 35533) page: E4M3 for every tensor,
 * Dgrad included; the jp-study.kr page: weights quantised per 128x128
 * block).  The amax of a 128x128 block is the same after
 * transposition, so (qT, sT) is exactly what fp8_quant_weight_128x128 would
 * give for the transposed bf16 matrix.  Dgrad dX = dY * W is then
 * fp8_gemm_blockscaled(a = 1x128 codes of dY, b = qT, sb = sT,
 * FP8_BSCALE_BLOCK128).
 *   q   E4M3 [N][K], s fp32 [N/128][K/128]   (from fp8_quant_weight_128x128)
 *   qT  E4M3 [K][N], sT fp32 [K/128][N/128]
 * N % 128 == 0, K % 128 == 0; q and qT 16-byte aligned.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_transpose_128x128(const uint8_t* q, const float* s, int64_t N, int64_t K,
                                  uint8_t* qT, float* sT, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * Grouped (per-expert) block-scaled FP8 GEMM for MoE (the jp-study.kr page: 256 routed
 * experts; each expert processes the rows dispatched to it).  Expert e owns
 * rows [off[e], off[e+1]) of a and d and multiplies them by its own B_e:
 *   d[r][n] = sum_kb sa[kb][r] * sb[e][n/128][kb] * P_kb(a[r], b[e][n])
 *   a    E4M3 [total_rows][K] (rows grouped by expert)
 *   sa   fp32 [K/128][total_rows]
 *   b    E4M3 [E][N][K]
 *   sb   fp32 [E][N/128][K/128]
 *   off  int32 [E+1] on the DEVICE: off[0] = 0, non-decreasing,
 *        off[E] = total_rows.  Empty experts are allowed.  The host never
 *        reads it.  Offsets that break these rules make the kernel record
 *        FP8_ERR_OFFSETS in the device status and skip the bad experts.
 *   d    bf16 [total_rows][N]
 * 1 <= E <= 1024, total_rows >= 0, N % 128 == 0, K % 128 == 0.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_grouped_gemm_blockscaled(const uint8_t* a, const float* sa,
                                         const uint8_t* b, const float* sb,
                                         const int32_t* expert_offsets, int E,
                                         int64_t total_rows, int64_t N, int64_t K,
                                         uint16_t* d, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * MoE routing on one GPU (the jp-study.kr page: each token activates 8 of 256 routed
 * experts).  Top-k of each token's logits, ties going to the lower expert
 * index; gates = softmax over the k selected logits (fp32); dispatch order =
 * (token, slot) pairs stably sorted by expert.
 *   logits  fp32 [T][E]
 *   idx     int32 [T][topk]   selected experts, highest logit first
 *   gate    fp32  [T][topk]
 *   off     int32 [E+1]       exclusive prefix sum of rows per expert
 *   src_row int32 [T*topk]    dispatched row p holds token src_row[p]
 *   pos     int32 [T][topk]   row that (token, slot) was dispatched to
 *   work    int32 scratch of fp8_moe_route_workspace_size(T, E) bytes; its
 *           contents on entry do not matter
 * 1 <= E <= 1024, 1 <= topk <= min(E, 32), T >= 1.
 * ---------------------------------------------------------------------- */
FP8_API int64_t fp8_moe_route_workspace_size(int64_t T, int E);
FP8_API int fp8_moe_route_topk(const float* logits, int64_t T, int E, int topk,
                               int32_t* idx, float* gate, int32_t* expert_offsets,
                               int32_t* src_row, int32_t* pos, int32_t* work,
                               fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8_moe_route_topk without the caller's scratch buffer (the pages have no
 * counterpart: this is a convenience of the library).  Some callers cannot
 * allocate device memory where they route: a runtime that gave all of HBM
 * to its own pool at start-up, or a serving loop that forbids cudaMalloc
 * after warm-up because allocating can synchronise the device.  This call
 * takes the same arguments and gives the same results as
 * fp8_moe_route_topk, minus `work`: its scratch is a fixed device array
 * inside the library (FP8_ROUTE_NOALLOC_MAX_WORK int32 words, 1 MiB, held
 * on every GPU that loads the library until the process exits).  It calls no
 * cudaMalloc or cudaFree.
 *   - Limit: ceil(T/64) * E <= FP8_ROUTE_NOALLOC_MAX_WORK (for E = 256,
 *     T <= 65536); larger problems return FP8_ERR_SCRATCH and launch
 *     nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.  The cached address belongs
 *     to the device's primary context: it is not valid after a
 *     cudaDeviceReset of that device, and the library does not clear it, so
 *     do not use this call on a device after resetting it.
 *   - Every call uses the same array and leaves its last contents there
 *     (nothing in it needs clearing: each call writes every word it reads).
 *     Calls whose kernels overlap on the GPU, e.g. on two streams at once,
 *     race on it and give wrong routes: serialise them.
 * ---------------------------------------------------------------------- */
#define FP8_ROUTE_NOALLOC_MAX_WORK (1 << 18)
FP8_API int fp8_moe_route_topk_noalloc(const float* logits, int64_t T, int E, int topk,
                                       int32_t* idx, float* gate, int32_t* expert_offsets,
                                       int32_t* src_row, int32_t* pos, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * Dispatch on one GPU: gather FP8 rows and their scales (the jp-study.kr page: activations
 * are quantised before the MoE up-projection, then dispatched in FP8).
 *   q_out[p][:] = q[src_row[p]][:],  s_out[kb][p] = s[kb][src_row[p]]
 *   q [rows][K], s [K/128][rows], src_row int32 [out_rows] (values in
 *   [0, rows)), q_out [out_rows][K], s_out [K/128][out_rows].  K % 128 == 0.
 * An index out of range records FP8_ERR_OFFSETS and that row is zero-filled.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_permute_rows(const uint8_t* q, const float* s, int64_t rows, int64_t K,
                             const int32_t* src_row, int64_t out_rows,
                             uint8_t* q_out, float* s_out, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * Combine kept in BF16 (the gnrental.net page: forward and backward combine stay in BF16):
 *   out[t][n] = bf16( sum_{j < topk} gate[t][j] * y[pos[t][j]][n] )
 * summed in fp32 in slot order, rounded to nearest-even once.
 *   y bf16 [rows][N], pos int32 [T][topk] (values in [0, rows)),
 *   gate fp32 [T][topk], out bf16 [T][N].  N % 8 == 0.
 * An index out of range records FP8_ERR_OFFSETS and contributes zero.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_moe_combine_bf16(const uint16_t* y, int64_t rows, const int32_t* pos,
                                 const float* gate, int64_t T, int topk, int64_t N,
                                 uint16_t* out, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * Device status: synchronises `stream`, then returns and clears the first
 * error code that a kernel recorded on the current device (FP8_OK if none).
 * ---------------------------------------------------------------------- */
FP8_API int fp8_get_status(fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * Failure-detection self-test (no counterpart on the pages): launches one
 * thread that waits on a pipeline barrier nobody arrives on, with the same
 * bounded wait the GEMMs use, shortened to timeout_ns (1 ns .. 2 s).  The
 * wait gives up, FP8_ERR_TIMEOUT is recorded in the device status, and the
 * kernel exits normally; fp8_get_status then returns FP8_ERR_TIMEOUT.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_selftest_wait_timeout(uint64_t timeout_ns, fp8_stream_t stream);

/* ------------------------------------------------------------------------
 * Reciprocal self-test (no counterpart on the pages): the SwiGLU kernel's
 * sigma = 1/d (d = 1 + e^-g >= 1) comes from the hardware approximation
 * corrected by Markstein's method; this counts, for every float d whose bit
 * pattern lies in [first_bits, last_bits], the d where that reciprocal
 * differs in any bit from __frcp_rn(d), adding the count to *mismatches
 * (a device counter the caller zeroes).  first_bits >= 0x3F800000 (d >= 1);
 * [0x3F800000, 0x7FFFFFFF] covers every d >= 1, +inf and the NaNs.
 * ---------------------------------------------------------------------- */
FP8_API int fp8_selftest_reciprocal(uint32_t first_bits, uint32_t last_bits, unsigned long long* mismatches,
                                    fp8_stream_t stream);

/* Human-readable name of a status code (static string). */
FP8_API const char* fp8_strerror(int code);

/* Library ABI version (major*100 + minor). */
FP8_API int fp8_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FP8BS_H */
