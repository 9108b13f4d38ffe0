// tmap.h -- host-side TMA descriptor (CUtensorMap) construction.  The driver
// entry point is looked up through the runtime, so the library does not link
// libcuda and still loads on a machine without a GPU driver.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ctxattn {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// A TMA map over a logical [B,S,H,D] bf16 tensor.  The three outer
// dimensions are handed to the driver in increasing-stride order; ord[i]
// says which logical coordinate (0 = s, 1 = h, 2 = b) feeds map dimension
// i + 1, so a kernel builds its coordinates with tma_coord().
struct TmaMap {
    CUtensorMap map;
    int32_t ord[3];
};

// Box = box_d x box_s rows of one (b, h), 128-byte swizzle (box_d * 2 == 128).
// Rows outside [0, S) read as zero.
inline bool make_tmap_bshd(TmaMap* out, const void* base, int64_t B, int64_t S, int64_t H,
                           int64_t D, int64_t sb, int64_t ss, int64_t sh, uint32_t box_d,
                           uint32_t box_s) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    int64_t size[3] = {S, H, B}, stride[3] = {ss, sh, sb};
    int64_t extent = 0;  // elements spanned by the tensor
    for (int i = 0; i < 3; ++i)
        if (size[i] > 1 && stride[i] * size[i] > extent) extent = stride[i] * size[i];
    if (extent < D) extent = D;
    for (int i = 0; i < 3; ++i)  // a size-1 dimension's stride is never used: make it outermost
        if (size[i] == 1) stride[i] = extent;
    int idx[3] = {0, 1, 2};
    for (int i = 0; i < 3; ++i)  // stable sort of the outer dims by stride
        for (int j = 0; j + 1 < 3 - i; ++j)
            if (stride[idx[j]] > stride[idx[j + 1]]) {
                int t = idx[j];
                idx[j] = idx[j + 1];
                idx[j + 1] = t;
            }
    cuuint64_t dims[4] = {(cuuint64_t)D, 0, 0, 0};
    cuuint64_t strides[3];
    cuuint32_t box[4] = {box_d, 1, 1, 1};
    for (int i = 0; i < 3; ++i) {
        dims[i + 1] = (cuuint64_t)size[idx[i]];
        strides[i] = (cuuint64_t)(stride[idx[i]] * 2);
        if (idx[i] == 0) box[i + 1] = box_s;
        out->ord[i] = idx[i];
    }
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(&out->map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace ctxattn
