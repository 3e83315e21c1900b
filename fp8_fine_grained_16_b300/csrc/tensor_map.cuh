// tensor_map.cuh -- host helpers shared by the GEMM translation units: TMA
// tensor maps for E4M3 operands and fp32 scale vectors, and the device check.
#pragma once
#include <cudaTypedefs.h>

#include "common.cuh"

namespace fp8bs {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// K-major E4M3 operand [rows][K] (rank 2), or a stack [batch][rows][K]
// (rank 3, even when batch == 1), box = 128 (K) x box_rows (x 1), 128-byte
// swizzle, zero fill out of bounds.
inline bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows,
                             int64_t batch, bool stacked) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cuuint64_t(K), cuuint64_t(rows), cuuint64_t(batch)};
    cuuint64_t strides[2] = {cuuint64_t(K), cuuint64_t(K) * cuuint64_t(rows)};
    cuuint32_t box[3] = {128u, cuuint32_t(box_rows), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    const cuuint32_t rank = stacked ? 3u : 2u;
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Rank-1 fp32 view of a scale tensor of n elements, box of `box` floats, no
// swizzle, zero fill past the end.
inline bool make_scale_map(CUtensorMap* map, const float* base, int64_t n, int box) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[1] = {cuuint64_t(n)};
    cuuint64_t strides[1] = {0};
    cuuint32_t boxd[1] = {cuuint32_t(box)};
    cuuint32_t estr[1] = {1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1u, const_cast<float*>(base), dims, strides, boxd, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Opt `kern` into `bytes` of dynamic shared memory (above the 48 KB default)
// on the current device, once per device: the attribute belongs to the
// device's context, so a process that drives several GPUs sets it on each.
constexpr int kMaxDevices = 64;
template <typename Kern>
inline bool opt_in_dynamic_smem(Kern kern, int bytes, unsigned char (&done)[kMaxDevices]) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    done[dev] = 1;
    return true;
}

inline int device_sms() {
    int dev = 0, n = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess || major != 10) return -1;
    return n;
}

}  // namespace fp8bs
