// pd_tmap.h -- host helpers that encode TMA tensor maps (128-byte swizzle)
// for the paged pools and the packed query tensor.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "pd_attn.h"

namespace pd {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

inline CUtensorMapDataType tmap_dtype(pd_dtype dt) {
    return dt == PD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// A pool [NB][Hk][S][D] seen as [NB*Hk*S rows][D]; box = box_rows rows x 64
// values (one 128-byte swizzle atom wide).  False if encoding fails.
inline bool encode_pool_map(CUtensorMap* m, const void* pool, int D, unsigned long long rows,
                            int box_rows, pd_dtype dt) {
    auto encode = tensor_map_encoder();
    if (!encode) return false;
    cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(D) * 2};
    cuuint32_t box[2] = {64u, cuuint32_t(box_rows)};
    cuuint32_t es[2] = {1u, 1u};
    return encode(m, tmap_dtype(dt), 2, const_cast<void*>(pool), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP8 pool viewed as rows of D bytes; box = one [box_rows][D] slab, packed
// rows, no swizzle, or 128-byte swizzle when swizzled (D must be 128).
inline bool encode_pool_map_u8(CUtensorMap* m, const void* pool, int D, unsigned long long rows,
                               int box_rows, bool swizzled = false) {
    auto encode = tensor_map_encoder();
    if (!encode) return false;
    cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(D)};
    cuuint32_t box[2] = {cuuint32_t(D), cuuint32_t(box_rows)};
    cuuint32_t es[2] = {1u, 1u};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzled ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed queries [total_q][H][D]; box = 64 values x heads x tokens.
inline bool encode_q_map(CUtensorMap* m, const void* q, int D, int H, int total_q,
                         int box_heads, int box_tokens, pd_dtype dt) {
    auto encode = tensor_map_encoder();
    if (!encode) return false;
    cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(total_q)};
    cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(H) * D * 2};
    cuuint32_t box[3] = {64u, cuuint32_t(box_heads), cuuint32_t(box_tokens)};
    cuuint32_t es[3] = {1u, 1u, 1u};
    return encode(m, tmap_dtype(dt), 3, const_cast<void*>(q), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pd
