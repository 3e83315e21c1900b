// moe.cu -- the MoE pieces around the grouped GEMM on one GPU (the jp-study.kr page: 256
// routed experts, 8 active per token, activations quantised to FP8 before
// dispatch; the gnrental.net page: the combine stays in BF16).
//
//   routing   top-k of each token's logits (ties to the lower expert),
//             softmax gates over the selected logits, and a stable
//             counting sort of (token, slot) pairs by expert:
//               kernel 1: one warp per token -> idx, gate, per-chunk counts
//                         (global atomics into a zeroed workspace)
//               kernel 2: one warp per expert turns the counts into
//                         running totals over the chunks, in place
//               kernel 3: per chunk of 64 tokens -> expert offsets and the
//                         rank of each pair among the chunk's pairs of the
//                         same expert (64-bit token masks + popcount)
//             kernels 2 and 3 are programmatic dependent launches.
//   permute   gathers FP8 rows and their K-block scales (dispatch)
//   combine   out[t] = sum_j gate[t][j] * y[pos[t][j]] in fp32 -> bf16
#include <mutex>

#include "common.cuh"

namespace fp8bs {

__device__ int g_moe_status;

FP8_DEV void moe_record(int code) { atomicCAS(&g_moe_status, 0, code); }

constexpr int kChunk = 64;            // tokens per routing chunk (one 64-bit mask per expert)
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;

// ------------------------------------------------------------------ routing, kernel 1
// One warp per token, 8 tokens per CTA (so every SM takes part: the ranking
// is ALU-bound).  Lane l holds logits e = l + 32j (j < EPL).  Each of the k
// rounds takes the warp-wide maximum among unselected experts, the lower
// index winning ties.  Each selected (token, expert) pair is counted into
// work[chunk][expert] (chunk = token / 64) with a global atomic; the caller
// zeroes work first.
template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k,
                                                        int32_t* __restrict__ idx, float* __restrict__ gate,
                                                        int32_t* __restrict__ work) {
    const int lane = threadIdx.x & 31;
    const int64_t t = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    pdl_launch_dependents();
    if (t >= T) return;                                   // warp-uniform
    float v[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < E ? __ldg(logits + t * E + e) : 0.0f;
    }
    uint32_t taken = 0;                          // bit j: expert lane+32j already selected
    int my_e = -1;                               // lane j < k keeps slot j
    float my_v = 0.0f;
    for (int r = 0; r < k; ++r) {
        float bv = 0.0f;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((taken >> j) & 1u) && (be == 0x7FFFFFFF || v[j] > bv)) {
                bv = v[j];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
            if (oe != 0x7FFFFFFF && (be == 0x7FFFFFFF || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == r) {
            my_e = be;
            my_v = bv;
        }
    }
    const float vmax = __shfl_sync(0xFFFFFFFFu, my_v, 0);
    const float ex = lane < k ? expf(my_v - vmax) : 0.0f;
    float z = ex;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
    pdl_wait();                                           // work has been zeroed
    if (lane < k) {
        idx[t * k + lane] = my_e;
        gate[t * k + lane] = __fdiv_rn(ex, z);
        atomicAdd(&work[(t / kChunk) * E + my_e], 1);
    }
}

// ------------------------------------------------------------------ routing, kernel 2
// work[c][e] (pairs of chunk c that chose expert e) -> the running total over
// chunks 0..c, in place.  One warp per expert: lane l takes chunk c0 + l of
// each group of 32 chunks, a shuffle scan forms the group's running totals,
// and the group's sum carries into the next group.  Four groups' loads are
// issued before any of them is scanned.
constexpr int kScanGroups = 4;

__global__ void __launch_bounds__(256) route_chunk_scan_kernel(int32_t* __restrict__ work, int64_t nchunks, int E) {
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
    pdl_launch_dependents();
    pdl_wait();                                               // the counts are complete
    if (e >= E) return;                                       // warp-uniform
    int carry = 0;
    for (int64_t c0 = 0; c0 < nchunks; c0 += 32 * kScanGroups) {
        int v[kScanGroups];
#pragma unroll
        for (int g = 0; g < kScanGroups; ++g) {
            const int64_t c = c0 + 32 * g + lane;
            v[g] = c < nchunks ? work[c * E + e] : 0;
        }
#pragma unroll
        for (int g = 0; g < kScanGroups; ++g) {
            int x = v[g];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            const int64_t c = c0 + 32 * g + lane;
            if (c < nchunks) work[c * E + e] = carry + x;
            carry += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
    }
}

// ------------------------------------------------------------------ routing, kernel 3
// One CTA (512 threads) per chunk.  Expert e's rows start at
//   off[e] + (pairs of expert e in earlier chunks) + (rank inside this chunk),
// the rank being the number of earlier tokens of the chunk that chose e; the
// running totals of kernel 2 give the earlier chunks' pairs (row chunk - 1)
// and each expert's total (row nchunks - 1).
__global__ void __launch_bounds__(512) route_positions_kernel(const int32_t* __restrict__ idx, int64_t T, int E,
                                                              int k, const int32_t* __restrict__ work,
                                                              int64_t nchunks, int32_t* __restrict__ off,
                                                              int32_t* __restrict__ src_row,
                                                              int32_t* __restrict__ pos) {
    __shared__ int base[kMaxE];
    __shared__ int scan[kMaxE + 1];
    __shared__ unsigned long long mask[kMaxE];
    __shared__ int warp_sum[16];
    const int tid = threadIdx.x;
    const int64_t chunk = blockIdx.x;
    pdl_wait();                                               // idx and the running totals are complete

    for (int e = tid; e < E; e += blockDim.x) {
        scan[e] = __ldg(work + (nchunks - 1) * E + e);
        base[e] = chunk > 0 ? __ldg(work + (chunk - 1) * E + e) : 0;
        mask[e] = 0ull;
    }
    __syncthreads();
    // exclusive scan of scan[0..E) (E <= 1024): each thread owns two slots
    {
        const int lane = tid & 31, wid = tid >> 5;
        const int i0 = 2 * tid, i1 = 2 * tid + 1;
        const int a = i0 < E ? scan[i0] : 0, b = i1 < E ? scan[i1] : 0;
        int incl = a + b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += x;
        }
        if (lane == 31) warp_sum[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            int w = lane < 16 ? warp_sum[lane] : 0;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                const int x = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o) w += x;
            }
            if (lane < 16) warp_sum[lane] = w;     // inclusive over warps
        }
        __syncthreads();
        const int warp_excl = wid > 0 ? warp_sum[wid - 1] : 0;
        const int excl = warp_excl + incl - (a + b);
        __syncthreads();
        if (i0 < E) scan[i0] = excl;
        if (i1 < E) scan[i1] = excl + a;
        if (tid == 0) scan[E] = warp_sum[15];
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) base[e] += scan[e];
    if (chunk == 0)
        for (int e = tid; e <= E; e += blockDim.x) off[e] = scan[e];

    const int64_t t0 = chunk * kChunk;
    const int npairs = kChunk * k;
    for (int i = tid; i < npairs; i += blockDim.x) {
        const int tt = i / k;
        if (t0 + tt < T) atomicOr(&mask[idx[(t0 + tt) * k + (i - tt * k)]], 1ull << tt);
    }
    __syncthreads();
    for (int i = tid; i < npairs; i += blockDim.x) {
        const int tt = i / k, j = i - tt * k;
        const int64_t t = t0 + tt;
        if (t >= T) continue;
        const int e = idx[t * k + j];
        const int rank = __popcll(mask[e] & ((1ull << tt) - 1ull));
        const int p = base[e] + rank;
        pos[t * k + j] = p;
        src_row[p] = int32_t(t);
    }
}

// ------------------------------------------------------------------ permute
// 256 threads per 32 output rows.  Codes: each warp copies 4 rows in 16-byte
// pieces.  Scales: thread i handles (kb = i / 32, row = i % 32) so the 32
// scales of one K block are written as one 128-byte segment.
__global__ void __launch_bounds__(256) permute_rows_kernel(const uint8_t* __restrict__ q, const float* __restrict__ s,
                                                          int64_t rows, int64_t K, const int32_t* __restrict__ src_row,
                                                          int64_t out_rows, uint8_t* __restrict__ q_out,
                                                          float* __restrict__ s_out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t p0 = int64_t(blockIdx.x) * 32;
    const int64_t n16 = K / 16;
#pragma unroll 1
    for (int rr = 0; rr < 4; ++rr) {
        const int64_t p = p0 + warp * 4 + rr;
        if (p >= out_rows) break;
        const int32_t r = __ldg(src_row + p);
        const bool ok = r >= 0 && r < rows;
        if (!ok && lane == 0) moe_record(FP8_ERR_OFFSETS);
        const uint4* src = reinterpret_cast<const uint4*>(q + (ok ? int64_t(r) : 0) * K);
        uint4* dst = reinterpret_cast<uint4*>(q_out + p * K);
        for (int64_t i = lane; i < n16; i += 32) dst[i] = ok ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
    }
    const int64_t nkb = K / 128;
    for (int64_t i = threadIdx.x; i < 32 * nkb; i += blockDim.x) {
        const int64_t kb = i / 32, p = p0 + (i & 31);
        if (p >= out_rows) continue;
        const int32_t r = __ldg(src_row + p);
        const bool ok = r >= 0 && r < rows;
        s_out[kb * out_rows + p] = ok ? __ldg(s + kb * rows + r) : 0.0f;
    }
}

// ------------------------------------------------------------------ combine
// Thread = (token t, 8 consecutive columns).  Consecutive threads take
// consecutive column groups of one token, so every y row is read in full
// 16-byte pieces and the output row is written coalesced.  With KC > 0 the
// token's k = KC positions and gates are loaded first and then all KC rows
// at once, so the row loads are in flight together; the sum runs in slot
// order either way.
template <int KC>
__global__ void __launch_bounds__(256) moe_combine_kernel(const uint16_t* __restrict__ y, int64_t rows,
                                                         const int32_t* __restrict__ pos,
                                                         const float* __restrict__ gate, int64_t T, int k, int64_t N,
                                                         uint16_t* __restrict__ out) {
    const int64_t groups = N / 8;
    const int64_t total = T * groups;
    for (int64_t it = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; it < total;
         it += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = it / groups, g = it - t * groups;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        if constexpr (KC > 0) {
            int32_t p[KC];
            float w[KC];
            uint4 v[KC];
#pragma unroll
            for (int j = 0; j < KC; ++j) {
                p[j] = __ldg(pos + t * KC + j);
                w[j] = __ldg(gate + t * KC + j);
            }
#pragma unroll
            for (int j = 0; j < KC; ++j) {
                const bool ok = p[j] >= 0 && p[j] < rows;
                v[j] = ok ? __ldg(reinterpret_cast<const uint4*>(y + int64_t(p[j]) * N) + g) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < KC; ++j) {
                if (p[j] < 0 || p[j] >= rows) {
                    moe_record(FP8_ERR_OFFSETS);
                    continue;
                }
                const uint32_t ww[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = fmaf(w[j], bf16_lo(ww[i]), acc[2 * i]);
                    acc[2 * i + 1] = fmaf(w[j], bf16_hi(ww[i]), acc[2 * i + 1]);
                }
            }
        } else {
            for (int j = 0; j < k; ++j) {
                const int32_t p = __ldg(pos + t * k + j);
                const float w = __ldg(gate + t * k + j);
                if (p < 0 || p >= rows) {
                    moe_record(FP8_ERR_OFFSETS);
                    continue;
                }
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(y + int64_t(p) * N) + g);
                const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = fmaf(w, bf16_lo(ww[i]), acc[2 * i]);
                    acc[2 * i + 1] = fmaf(w, bf16_hi(ww[i]), acc[2 * i + 1]);
                }
            }
        }
        reinterpret_cast<uint4*>(out + t * N)[g] =
            make_uint4(cvt_bf16x2(acc[0], acc[1]), cvt_bf16x2(acc[2], acc[3]), cvt_bf16x2(acc[4], acc[5]),
                       cvt_bf16x2(acc[6], acc[7]));
    }
}

static int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0)
        return 148;
    return n;
}

}  // namespace fp8bs

using namespace fp8bs;

extern "C" int64_t fp8_moe_route_workspace_size(int64_t T, int E) {
    if (T <= 0 || E <= 0) return 0;
    return ((T + kChunk - 1) / kChunk) * int64_t(E) * int64_t(sizeof(int32_t));
}

extern "C" int fp8_moe_route_topk(const float* logits, int64_t T, int E, int topk, int32_t* idx, float* gate,
                                  int32_t* expert_offsets, int32_t* src_row, int32_t* pos, int32_t* work,
                                  fp8_stream_t stream) {
    if (!logits || !idx || !gate || !expert_offsets || !src_row || !pos || !work) return FP8_ERR_ARG;
    if (T <= 0 || E <= 0 || E > kMaxE || topk <= 0 || topk > kMaxK || topk > E) return FP8_ERR_ARG;
    if (T * topk > 0x7FFFFFFFll) return FP8_ERR_SHAPE;
    const uintptr_t any = reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(idx) |
                          reinterpret_cast<uintptr_t>(gate) | reinterpret_cast<uintptr_t>(expert_offsets) |
                          reinterpret_cast<uintptr_t>(src_row) | reinterpret_cast<uintptr_t>(pos) |
                          reinterpret_cast<uintptr_t>(work);
    if (any & 3u) return FP8_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t nchunks = (T + kChunk - 1) / kChunk;
    if (nchunks > 0x7FFFFFFFll) return FP8_ERR_SHAPE;
    const int epl = (E + 31) / 32;
    const unsigned g = unsigned(nchunks);
    if (cudaMemsetAsync(work, 0, size_t(nchunks) * size_t(E) * sizeof(int32_t), s) != cudaSuccess) return FP8_ERR_CUDA;
    const unsigned gt = unsigned((T + 7) / 8);
    if (epl <= 1) route_topk_kernel<1><<<gt, 256, 0, s>>>(logits, T, E, topk, idx, gate, work);
    else if (epl <= 2) route_topk_kernel<2><<<gt, 256, 0, s>>>(logits, T, E, topk, idx, gate, work);
    else if (epl <= 4) route_topk_kernel<4><<<gt, 256, 0, s>>>(logits, T, E, topk, idx, gate, work);
    else if (epl <= 8) route_topk_kernel<8><<<gt, 256, 0, s>>>(logits, T, E, topk, idx, gate, work);
    else if (epl <= 16) route_topk_kernel<16><<<gt, 256, 0, s>>>(logits, T, E, topk, idx, gate, work);
    else route_topk_kernel<32><<<gt, 256, 0, s>>>(logits, T, E, topk, idx, gate, work);
    if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
    // the scan and the positions start early (programmatic dependent
    // launches) and wait inside for the kernel before them
    if (launch_pdl(route_chunk_scan_kernel, dim3(unsigned((E + 7) / 8)), dim3(256), 0, s, work, nchunks, E) !=
        cudaSuccess)
        return FP8_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
    if (launch_pdl(route_positions_kernel, dim3(g), dim3(512), 0, s, static_cast<const int32_t*>(idx), T, E, topk,
                   static_cast<const int32_t*>(work), nchunks, expert_offsets, src_row, pos) != cudaSuccess)
        return FP8_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" int fp8_permute_rows(const uint8_t* q, const float* s, int64_t rows, int64_t K, const int32_t* src_row,
                                int64_t out_rows, uint8_t* q_out, float* s_out, fp8_stream_t stream) {
    if (rows <= 0 || K <= 0 || out_rows < 0) return FP8_ERR_ARG;
    if (K % 128) return FP8_ERR_SHAPE;
    if (out_rows == 0) return FP8_OK;
    if (!q || !s || !src_row || !q_out || !s_out) return FP8_ERR_ARG;
    if (!aligned16(q) || !aligned16(q_out) ||
        ((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(s_out) | reinterpret_cast<uintptr_t>(src_row)) &
         3u))
        return FP8_ERR_ALIGN;
    const int64_t blocks = (out_rows + 31) / 32;
    if (blocks > 0x7FFFFFFFll) return FP8_ERR_SHAPE;
    permute_rows_kernel<<<unsigned(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(q, s, rows, K, src_row,
                                                                                            out_rows, q_out, s_out);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" int fp8_moe_combine_bf16(const uint16_t* y, int64_t rows, const int32_t* pos, const float* gate, int64_t T,
                                    int topk, int64_t N, uint16_t* out, fp8_stream_t stream) {
    if (!y || !pos || !gate || !out || rows <= 0 || T <= 0 || topk <= 0 || N <= 0) return FP8_ERR_ARG;
    if (N % 8) return FP8_ERR_SHAPE;
    if (!aligned16(y) || !aligned16(out) ||
        ((reinterpret_cast<uintptr_t>(pos) | reinterpret_cast<uintptr_t>(gate)) & 3u))
        return FP8_ERR_ALIGN;
    const int64_t total = T * (N / 8);
    const int64_t blocks = (total + 255) / 256;
    const int64_t cap = int64_t(sm_count()) * 8;
    const unsigned grid = unsigned(blocks < cap ? blocks : cap);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (topk == 8)
        moe_combine_kernel<8><<<grid, 256, 0, st>>>(y, rows, pos, gate, T, topk, N, out);
    else
        moe_combine_kernel<0><<<grid, 256, 0, st>>>(y, rows, pos, gate, T, topk, N, out);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// ------------------------------------------------------------------ routing without caller scratch
// Variant of fp8_moe_route_topk for callers that cannot allocate device
// memory where they call it.  The per-chunk expert counts live in this
// file-scope device array instead of a caller buffer; every GPU that loads
// the library keeps it (1 MiB) until the process exits.  No element needs to
// start at zero: the first kernel writes all nchunks x E counts before the
// later kernels of the same call read any of them.  Calls share the array,
// so two calls whose kernels overlap on the GPU race on it.
namespace fp8bs {
static __device__ __align__(256) int32_t g_route_scratch[FP8_ROUTE_NOALLOC_MAX_WORK];

constexpr int kMaxDevices = 64;

// Device address of g_route_scratch for the current device.  In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.  The
// cached address belongs to the device's primary context: after a
// cudaDeviceReset of that device it is stale, and the cache is not cleared.
static int32_t* route_scratch_address() {
    static std::mutex mu;
    static int32_t* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev] = static_cast<int32_t*>(p);
    }
    return addr[dev];
}
}  // namespace fp8bs

extern "C" int fp8_moe_route_topk_noalloc(const float* logits, int64_t T, int E, int topk, int32_t* idx, float* gate,
                                          int32_t* expert_offsets, int32_t* src_row, int32_t* pos,
                                          fp8_stream_t stream) {
    if (T <= 0 || E <= 0 || E > kMaxE || topk <= 0 || topk > kMaxK || topk > E) return FP8_ERR_ARG;
    if (fp8_moe_route_workspace_size(T, E) > int64_t(sizeof(int32_t)) * FP8_ROUTE_NOALLOC_MAX_WORK)
        return FP8_ERR_SCRATCH;
    int32_t* work = route_scratch_address();
    if (!work) return FP8_ERR_CUDA;
    return fp8_moe_route_topk(logits, T, E, topk, idx, gate, expert_offsets, src_row, pos, work, stream);
}

extern "C" int fp8bs_moe_take_status(cudaStream_t stream) {
    int v = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP8_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_moe_status, sizeof v) != cudaSuccess) return FP8_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_moe_status, &zero, sizeof zero) != cudaSuccess) return FP8_ERR_CUDA;
    return v;
}
