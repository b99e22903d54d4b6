// Host-side encoding of TMA tensor maps for K-major f16 matrices.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace qwen2 {

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime
// (no link-time dependency on libcuda).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        cudaGetLastError();
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// Map of a row-major f16 matrix [rows][k] read in boxes of 64 (k) x
// box_rows (rows) with the 128-byte swizzle; reads past `rows` return zeros.
// Requirements checked here: base 16-byte aligned, k a multiple of 64,
// box_rows in [1, 256].
inline bool encode_kmajor_f16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t k, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || !base || (reinterpret_cast<uintptr_t>(base) & 15) || k % 64 || rows == 0 || box_rows == 0 ||
        box_rows > 256)
        return false;
    const cuuint64_t dims[2] = {k, rows};
    const cuuint64_t strides[1] = {k * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map of a row-major f32 matrix [rows][64] read in boxes of 32 floats (128
// bytes) x box_rows rows with the 128-byte swizzle; reads past `rows` return
// zeros.  Requirements checked here: base 16-byte aligned, rows < 2^31,
// box_rows in [1, 256].
inline bool encode_rows64_f32(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || !base || (reinterpret_cast<uintptr_t>(base) & 15) || rows == 0 || rows >= (1ull << 31) ||
        box_rows == 0 || box_rows > 256)
        return false;
    const cuuint64_t dims[2] = {64, rows};
    const cuuint64_t strides[1] = {64 * 4};
    const cuuint32_t box[2] = {32, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace qwen2
