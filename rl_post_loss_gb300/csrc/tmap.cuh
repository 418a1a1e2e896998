// Host-side encoding of 2-D tensor maps (TMA descriptors) with the 128-byte
// swizzle, through the driver's cuTensorMapEncodeTiled (looked up once).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace rlk {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
        cudaGetLastError();
    });
    return fn;
}

// 2-D tensor map over a row-major [rows x cols] array with row stride `ld`
// elements of `esize` bytes: boxes of box_rows x box_cols with the 128-byte
// swizzle (box_cols x esize = 128 bytes; a box lands in shared memory with
// 16-byte unit j of row r at j ^ (r % 8)). Out-of-range parts of a box read as
// zero and are not written. False if the driver refuses the map (alignment).
inline bool make_tmap_sw128(CUtensorMap *m, CUtensorMapDataType type, uint32_t esize, const void *base, int64_t rows,
                            int64_t cols, int64_t ld, uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc || !base) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * esize};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, type, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace rlk
