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
// One CTA (256 threads) per 128x128 byte tile.  Thread (warp w, lane l)
// loads the 16-byte pieces at byte column 16s of the input rows 4q .. 4q+3
// (s = l % 8, q = 4w + l / 8): every load instruction of a warp reads four
// whole 128-byte rows.  Each of its four 4x4 byte blocks is transposed in
// registers (byte permutes) and lands in a shared tile whose words are
// rotated per output row c by rot(c) = 4 * ((c + c/16) mod 8) words.  The
// stores are conflict-free (for a store instruction c/16 = s and c mod 8 is
// fixed, so slot q + 4 * ((k + s) mod 8) takes 32 distinct banks), and since
// the rotation is a multiple of four words the loads are aligned 16-byte
// pieces, also conflict-free (the eight threads of a load phase read four
// consecutive rows, two halves each, whose rotations differ by one piece and
// whose halves by four): four loads per thread instead of sixteen, which
// relieves the shared-memory instruction queue that throttled the copy.  The
// output leaves as 16-byte pieces of whole 128-byte rows.
#include "common.cuh"

namespace fp8bs {

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

__global__ void __launch_bounds__(256) transpose_128x128_kernel(const uint8_t* __restrict__ q,
                                                                const float* __restrict__ s, int64_t N,
                                                                int64_t K, uint8_t* __restrict__ qT,
                                                                float* __restrict__ sT) {
    // T[c][slot]: output row c (= input column), 32 words = input rows 4*word ..
    // 4*word+3; word `wd` of row c sits at slot (wd + rot(c)) % 32.
    __shared__ __align__(16) uint32_t T[128 * 32];
    auto rot = [](int c) { return 4 * ((c + (c >> 4)) & 7); };
    const int64_t nkb = K >> 7, nnb = N >> 7;
    const int64_t nb = blockIdx.x / nkb, kb = blockIdx.x - nb * nkb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint8_t* src = q + (nb * 128) * K + kb * 128;

    {
        const int sg = lane & 7, qd = 4 * warp + (lane >> 3);    // 16-byte column piece, input row quad
        uint4 in4[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
            in4[r] = __ldg(reinterpret_cast<const uint4*>(src + (4 * qd + r) * K) + sg);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t in[4] = {(&in4[0].x)[w], (&in4[1].x)[w], (&in4[2].x)[w], (&in4[3].x)[w]};
            uint32_t out[4];
            transpose4x4(in, out);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = 16 * sg + 4 * w + i;         // input column = output row
                T[c * 32 + ((qd + rot(c)) & 31)] = out[i];
            }
        }
    }
    __syncthreads();
    // output row c = t / 2, words 16h .. 16h+15 (h = t % 2), four 16-byte stores
    const int c = threadIdx.x >> 1, h = threadIdx.x & 1;
    uint8_t* dst = qT + (kb * 128 + c) * N + nb * 128 + 64 * h;
#pragma unroll
    for (int v = 0; v < 4; ++v)
        reinterpret_cast<uint4*>(dst)[v] =
            *reinterpret_cast<const uint4*>(&T[c * 32 + ((16 * h + 4 * v + rot(c)) & 31)]);
    if (threadIdx.x == 0) sT[kb * nnb + nb] = s[nb * nkb + kb];
}

}  // namespace fp8bs

using namespace fp8bs;

extern "C" int fp8_transpose_128x128(const uint8_t* q, const float* s, int64_t N, int64_t K, uint8_t* qT, float* sT,
                                     fp8_stream_t stream) {
    if (!q || !s || !qT || !sT || N <= 0 || K <= 0) return FP8_ERR_ARG;
    if (N % 128 || K % 128) return FP8_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(qT) || ((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(sT)) & 3u))
        return FP8_ERR_ALIGN;
    const int64_t blocks = (N / 128) * (K / 128);
    if (blocks > 0x7FFFFFFFll) return FP8_ERR_SHAPE;
    transpose_128x128_kernel<<<unsigned(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(q, s, N, K, qT, sT);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}
