// status.cu -- device status, error strings and version of libfp8bs.
#include "common.cuh"

extern "C" int fp8bs_gemm_take_status(cudaStream_t stream);
extern "C" int fp8bs_moe_take_status(cudaStream_t stream);
extern "C" int fp8bs_gemm_mx_take_status(cudaStream_t stream);
extern "C" int fp8bs_transpose_take_status(cudaStream_t stream);

extern "C" int fp8_get_status(fp8_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int a = fp8bs_gemm_take_status(s);
    const int b = fp8bs_moe_take_status(s);
    const int c = fp8bs_gemm_mx_take_status(s);
    const int d = fp8bs_transpose_take_status(s);
    return a != FP8_OK ? a : (b != FP8_OK ? b : (c != FP8_OK ? c : d));
}

extern "C" const char* fp8_strerror(int code) {
    switch (code) {
        case FP8_OK: return "ok";
        case FP8_ERR_ARG: return "invalid argument";
        case FP8_ERR_SHAPE: return "unsupported shape (a dimension must be a multiple of 128)";
        case FP8_ERR_ALIGN: return "pointer or leading dimension not 16-byte aligned";
        case FP8_ERR_CUDA: return "CUDA launch or runtime call failed";
        case FP8_ERR_TIMEOUT: return "device pipeline wait timed out";
        case FP8_ERR_OFFSETS: return "expert offsets or row indices out of range";
        case FP8_ERR_DEVICE: return "no usable sm_100-family device";
        case FP8_ERR_SCRATCH: return "problem larger than the library's static scratch";
        case FP8_ERR_SCALE: return "a scale given to the power-of-two GEMM is not a positive normal power of two";
        default: return "unknown status";
    }
}

extern "C" int fp8_version(void) { return 100; }
