// tmap.cuh -- host-side encoding of TMA tensor maps for bf16 tiles with the
// 128-byte swizzle.  cuTensorMapEncodeTiled is reached through the runtime's
// driver entry point, so the library does not link libcuda directly.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace gdn {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A rank-3 bf16 tensor: dims[0] contiguous (elements), strides of dims 1 and 2
// in bytes (multiples of 16), box {box0, box1, box2}.  swizzle128: the
// 128-byte swizzle (box0 = 64), else rows land unswizzled.  Out-of-range box
// elements read as zero.  Returns false if encoding fails.
inline bool make_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                              uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                              uint32_t box2, bool swizzle128 = true) {
    if (reinterpret_cast<uintptr_t>(base) & 15u) return false;
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {box0, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token-indexed bf16 tensor [B, T, heads, 128] as a 4-D map (128, heads, T, B): a box
// that runs past a sequence's last token reads zeros and a store there is clipped,
// so a partial last chunk never touches the next sequence.
inline bool make_tmap_tokens(CUtensorMap *map, const void *base, uint64_t heads, uint64_t T, uint64_t B,
                             uint32_t box_x, uint32_t box_rows, bool swizzle128 = true) {
    if (reinterpret_cast<uintptr_t>(base) & 15u) return false;
    auto enc = tmap_encoder();
    if (!enc) return false;
    const uint64_t row = 128 * 2;
    cuuint64_t dims[4] = {128, heads, T, B};
    cuuint64_t strides[3] = {row, heads * row, T * heads * row};
    cuuint32_t box[4] = {box_x, 1, box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Head-major bf16 tensor [B, heads, T, 128] (the workspace's U for bf16 storage) as a 4-D
// map (128, T, heads, B): a head's token rows are contiguous, so a chunk's tile is one
// contiguous block.  Coordinates (x, token, head, sequence); a box past a sequence's last
// token reads zeros and a store there is clipped.
inline bool make_tmap_headmajor(CUtensorMap *map, const void *base, uint64_t heads, uint64_t T, uint64_t B,
                                uint32_t box_x, uint32_t box_rows, bool swizzle128 = true) {
    if (reinterpret_cast<uintptr_t>(base) & 15u) return false;
    auto enc = tmap_encoder();
    if (!enc) return false;
    const uint64_t row = 128 * 2;
    cuuint64_t dims[4] = {128, T, heads, B};
    cuuint64_t strides[3] = {row, T * row, heads * T * row};
    cuuint32_t box[4] = {box_x, box_rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A rank-2 fp32 tensor: dims[0] contiguous (elements), rows stride1_bytes apart (a multiple
// of 16), box {box0, box1}, no swizzle.  Returns false if encoding fails.
inline bool make_tmap_f32_2d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t stride1_bytes,
                             uint32_t box0, uint32_t box1) {
    if (reinterpret_cast<uintptr_t>(base) & 15u) return false;
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {d0, d1};
    cuuint64_t strides[1] = {stride1_bytes};
    cuuint32_t box[2] = {box0, box1};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gdn
