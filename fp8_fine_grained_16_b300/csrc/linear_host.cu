// linear_host.cu -- the dense FP8 linear layer called with HOST buffers:
// Y = X W^T with X bf16 [M][K] and W bf16 [N][K] in host memory, Y bf16
// [M][N] returned to host memory.  On the GPU it is the library's own path
// (the jp-study.kr page: 1x128 activation tiles, 128x128 weight blocks; the
// tmdrlife.com page: partial sums promoted into FP32 with the two scales):
// quantise X 1x128, quantise W 128x128, block-scaled GEMM to bf16.
//
// The host<->device copies dominate such a call (PCIe moves ~55 GB/s against
// HBM's 6.5 TB/s), so the call is cut into chunks of W's rows (= Y's columns)
// on three streams:
//   copy-in stream   X, then W chunk 0, 1, ...        (one cudaMemcpyAsync each)
//   caller's stream  quantise X; per chunk: quantise W_j, GEMM_j -> Y_j
//   copy-out stream  per chunk: Y_j -> the host's Y columns (cudaMemcpy2DAsync)
// so that the weight chunks still in flight, the GPU work and the results on
// their way back overlap; what is left after the last input byte lands is one
// chunk's quantisation, GEMM and copy back.  Chunk GEMMs of fewer tiles than
// SM pairs are split along K through the GEMM workspace, so a narrow chunk
// still fills the GPU.
//
// The internal streams and events are created once per device and reused;
// the enqueue is serialised per device by a mutex (an event's later record
// does not affect waits already enqueued, so reuse across calls is safe).
#include <mutex>

#include "common.cuh"

namespace fp8bs {

constexpr int64_t kLinChunkMin = 1024;       // W rows (Y columns) per chunk
constexpr int kLinMaxChunks = 64;
constexpr int kLinMaxDevices = 64;

struct LinStreams {
    std::mutex mu;
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, x_in = nullptr, done = nullptr;
    cudaEvent_t w_in[kLinMaxChunks] = {}, y_out[kLinMaxChunks] = {};
};

LinStreams g_lin[kLinMaxDevices];
std::mutex g_lin_init;

// This device's streams and events, created on first use (nullptr on failure).
LinStreams* lin_streams() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kLinMaxDevices) return nullptr;
    LinStreams& L = g_lin[dev];
    std::lock_guard<std::mutex> lk(g_lin_init);
    if (L.ready) return &L;
    // handles made before a failed attempt are kept, so a retry creates only the rest
    const unsigned ef = cudaEventDisableTiming;
    auto stream_ = [](cudaStream_t& s) { return s || cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) == cudaSuccess; };
    auto event_ = [ef](cudaEvent_t& e) { return e || cudaEventCreateWithFlags(&e, ef) == cudaSuccess; };
    bool ok = stream_(L.h2d) && stream_(L.d2h) && event_(L.start) && event_(L.x_in) && event_(L.done);
    for (int j = 0; ok && j < kLinMaxChunks; ++j) ok = event_(L.w_in[j]) && event_(L.y_out[j]);
    if (!ok) return nullptr;
    L.ready = true;
    return &L;
}

// Chunk width: a multiple of 512 rows, so that every chunk's first row of
// 128x128 block scales starts 16-byte aligned (the GEMM reads them with TMA);
// at most kLinMaxChunks chunks.
inline int64_t lin_chunk(int64_t N) {
    int64_t c = kLinChunkMin;
    const int64_t need = (N + kLinMaxChunks - 1) / kLinMaxChunks;
    if (need > c) c = (need + 511) / 512 * 512;
    return c < N ? c : N;
}

inline int64_t align256(int64_t v) { return (v + 255) / 256 * 256; }

// Byte offsets of the workspace's parts.
struct LinLayout {
    int64_t x, qx, sx, w, qw, sw, y, g, g_bytes, total;
};

inline bool lin_layout(int64_t M, int64_t N, int64_t K, LinLayout& L) {
    const int64_t nc = lin_chunk(N);
    int64_t g = 0;
    for (int64_t n0 = 0; n0 < N; n0 += nc) {
        const int64_t b = fp8_gemm_blockscaled_workspace_bytes(M, (N - n0) < nc ? N - n0 : nc, K);
        if (b < 0) return false;
        if (b > g) g = b;
    }
    int64_t o = 0;
    L.x = o;  o = align256(o + M * K * 2);
    L.qx = o; o = align256(o + M * K);
    L.sx = o; o = align256(o + (K / 128) * M * 4);
    L.w = o;  o = align256(o + N * K * 2);
    L.qw = o; o = align256(o + N * K);
    L.sw = o; o = align256(o + (N / 128) * (K / 128) * 4);
    L.y = o;  o = align256(o + M * N * 2);
    L.g = o;  o = align256(o + g);
    L.g_bytes = g;
    L.total = o;
    return true;
}

}  // namespace fp8bs

using namespace fp8bs;

extern "C" int64_t fp8_linear_host_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return FP8_ERR_ARG;
    if (N % 128 || K % 128) return FP8_ERR_SHAPE;
    LinLayout L;
    if (!lin_layout(M, N, K, L)) return FP8_ERR_DEVICE;
    return L.total;
}

extern "C" int fp8_linear_host(const uint16_t* x_h, const uint16_t* w_h, int64_t M, int64_t N, int64_t K,
                               uint16_t* y_h, uint32_t flags, void* workspace, int64_t workspace_bytes,
                               fp8_stream_t stream) {
    if (!x_h || !w_h || !y_h || !workspace || M <= 0 || N <= 0 || K <= 0 || (flags & ~FP8_SCALE_POW2))
        return FP8_ERR_ARG;
    if (N % 128 || K % 128) return FP8_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FP8_ERR_ALIGN;
    LinLayout lay;
    if (!lin_layout(M, N, K, lay)) return FP8_ERR_DEVICE;
    if (workspace_bytes < lay.total) return FP8_ERR_ARG;
    LinStreams* Ls = lin_streams();
    if (!Ls) return FP8_ERR_CUDA;
    LinStreams& L = *Ls;
    std::lock_guard<std::mutex> lk(L.mu);

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint16_t* x_d = reinterpret_cast<uint16_t*>(ws + lay.x);
    uint8_t* qx = ws + lay.qx;
    float* sx = reinterpret_cast<float*>(ws + lay.sx);
    uint16_t* w_d = reinterpret_cast<uint16_t*>(ws + lay.w);
    uint8_t* qw = ws + lay.qw;
    float* sw = reinterpret_cast<float*>(ws + lay.sw);
    uint16_t* y_d = reinterpret_cast<uint16_t*>(ws + lay.y);
    void* g = lay.g_bytes ? static_cast<void*>(ws + lay.g) : nullptr;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t nc = lin_chunk(N);
    const int nchunks = int((N + nc - 1) / nc);
    const int64_t kb = K / 128;
    auto cu = [](cudaError_t e) { return e == cudaSuccess; };

    // the copies start after the caller's earlier work on `stream`
    bool ok = cu(cudaEventRecord(L.start, st)) && cu(cudaStreamWaitEvent(L.h2d, L.start, 0)) &&
              cu(cudaStreamWaitEvent(L.d2h, L.start, 0));
    ok = ok && cu(cudaMemcpyAsync(x_d, x_h, size_t(M * K * 2), cudaMemcpyHostToDevice, L.h2d)) &&
         cu(cudaEventRecord(L.x_in, L.h2d));
    for (int j = 0; ok && j < nchunks; ++j) {
        const int64_t n0 = j * nc, ncj = (N - n0) < nc ? N - n0 : nc;
        ok = cu(cudaMemcpyAsync(w_d + n0 * K, w_h + n0 * K, size_t(ncj * K * 2), cudaMemcpyHostToDevice, L.h2d)) &&
             cu(cudaEventRecord(L.w_in[j], L.h2d));
    }
    int rc = ok ? FP8_OK : FP8_ERR_CUDA;
    if (rc == FP8_OK) {
        rc = cu(cudaStreamWaitEvent(st, L.x_in, 0)) ? fp8_quant_act_1x128(x_d, M, K, K, qx, sx, flags, stream)
                                                     : FP8_ERR_CUDA;
    }
    for (int j = 0; rc == FP8_OK && j < nchunks; ++j) {
        const int64_t n0 = j * nc, ncj = (N - n0) < nc ? N - n0 : nc;
        uint16_t* y_j = y_d + M * n0;          // chunk j of Y, [M][ncj] contiguous
        if (!cu(cudaStreamWaitEvent(st, L.w_in[j], 0))) { rc = FP8_ERR_CUDA; break; }
        rc = fp8_quant_weight_128x128(w_d + n0 * K, ncj, K, K, qw + n0 * K, sw + (n0 / 128) * kb, flags, stream);
        if (rc != FP8_OK) break;
        rc = fp8_gemm_blockscaled_ws(qx, sx, qw + n0 * K, sw + (n0 / 128) * kb, FP8_BSCALE_BLOCK128, y_j,
                                     FP8_OUT_BF16, M, ncj, K, g, lay.g_bytes, stream);
        if (rc != FP8_OK) break;
        if (!cu(cudaEventRecord(L.y_out[j], st)) || !cu(cudaStreamWaitEvent(L.d2h, L.y_out[j], 0)) ||
            !cu(cudaMemcpy2DAsync(y_h + n0, size_t(N * 2), y_j, size_t(ncj * 2), size_t(ncj * 2), size_t(M),
                                  cudaMemcpyDeviceToHost, L.d2h)))
            rc = FP8_ERR_CUDA;
    }
    // whatever was enqueued, the caller's stream continues after all of it
    // (so the workspace and the host buffers are free once it gets there)
    const bool tail = cu(cudaEventRecord(L.x_in, L.h2d)) && cu(cudaStreamWaitEvent(L.d2h, L.x_in, 0)) &&
                      cu(cudaEventRecord(L.done, L.d2h)) && cu(cudaStreamWaitEvent(st, L.done, 0));
    if (!tail && rc == FP8_OK) rc = FP8_ERR_CUDA;
    return rc;
}
