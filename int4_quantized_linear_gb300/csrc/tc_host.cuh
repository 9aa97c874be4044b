// tc_host.cuh -- host helpers shared by the tensor-core kernels: TMA tensor-map encoding
// (through the driver entry point, so the library needs no link-time libcuda), SM count.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace w4a8 {
namespace tch {

// The per-process and per-device caches below are filled on first use; threads that race on a
// first use compute and store the same value, and the atomics make that race well defined.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
    if (!f) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
            fn.store(f, std::memory_order_release);
        }
    }
    return f;
}

// 2-D tensor map over a row-major [rows, cols] array of 1-byte (or 4-bit) elements.
inline bool tmap_2d(CUtensorMap *m, CUtensorMapDataType type, const void *base, uint64_t rows,
                    uint64_t cols_elems, uint64_t row_stride_bytes, uint32_t box_rows,
                    uint32_t box_cols_elems, CUtensorMapSwizzle swz)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols_elems, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_stride_bytes};
    cuuint32_t box[2] = {box_cols_elems, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, type, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D tensor map over a row-major [rows, row_bytes] array viewed as [k-tile][row][128 elements]:
// dim 0 = the 128 elements of a k-tile (4- or 8-bit), dim 1 = rows (stride row_bytes), dim 2 =
// k-tiles (stride ktile_bytes).  Box = 128 elements x box_rows x box_ktiles, 128-byte swizzle.
inline bool tmap_3d_ktiles(CUtensorMap *m, CUtensorMapDataType type, const void *base, uint64_t rows,
                           uint64_t row_bytes, uint64_t ktile_bytes, uint64_t ktiles, uint32_t box_rows,
                           uint32_t box_ktiles)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)ktiles};
    cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)ktile_bytes};
    cuuint32_t box[3] = {128, box_rows, box_ktiles};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, type, 3, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int num_sms()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (!v) {
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        v = v > 0 ? v : 148;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Set the dynamic shared-memory limit of a kernel once per device (setting it twice is harmless).
template <typename K>
inline bool set_smem_once(K kern, int bytes, std::atomic<int> (&done)[64])
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!done[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
            return false;
        done[dev].store(1, std::memory_order_release);
    }
    return true;
}

}  // namespace tch
}  // namespace w4a8
